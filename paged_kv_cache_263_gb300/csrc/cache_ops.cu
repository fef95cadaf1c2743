// cache_ops.cu -- cache write (reshape_and_cache), the copy-on-write block
// copy, and the device status word reader.
//
// Cache write: new K/V rows of each token land in the slot the scheduler gave
// them, block slot/16 at offset slot%16 -- blocks are handed out on demand as a
// sequence grows ("PagedAttention, chunked prefill, and the launch that
// cascades", section "PagedAttention: an OS idea, not an ML one"; "M.65
// Inference serving", block management (c)).  For the fp8 cache each element
// is stored as one e4m3 byte ("Waste, and three ways to reclaim it", section
// "Quantising the cache"; "M.65 Inference serving", quantisation (b), (d)):
// e4m3(x / scale[h]) with IEEE fp32 division, round-to-nearest-even and
// saturation at +-448 -- the hardware conversion cvt.rn.satfinite.
//
// Copy-on-write block copy: "Waste, and three ways to reclaim it", section
// "Sharing, and what makes a prefix reusable" (a writer into a shared block
// first gets its own copy); "M.65 Inference serving", block management (g).
#include "common.cuh"
#include "trace.h"

#include <algorithm>

namespace {

__device__ uint32_t g_status;

using namespace pkv;

// One thread per 16-byte chunk (8 bf16) of one (token, head) row of K and V.
template <bool FP8>
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                             uint8_t *__restrict__ kc, uint8_t *__restrict__ vc,
                             const int64_t *__restrict__ slots, int64_t total_chunks, int hkv,
                             int64_t num_slots, const float *__restrict__ ks,
                             const float *__restrict__ vs)
{
    // the attention kernel that follows may begin scheduling at once; it waits
    // for this grid to finish before it reads the cache
    griddep_launch_dependents();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total_chunks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int chunk = static_cast<int>(i & 15);
        const int64_t th = i >> 4;
        const int h = static_cast<int>(th % hkv);
        const int64_t t = th / hkv;
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (chunk == 0) atomicOr(&g_status, ST_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot >> 4, off = slot & 15;
        const int64_t dst = ((blk * hkv + h) * BS + off) * D + chunk * 8;  // element index
        const uint4 kx = __ldg(k + i);
        const uint4 vx = __ldg(v + i);
        if constexpr (!FP8) {
            *reinterpret_cast<uint4 *>(kc + dst * 2) = kx;
            *reinterpret_cast<uint4 *>(vc + dst * 2) = vx;
        } else {
            const float sk = __ldg(ks + h), sv = __ldg(vs + h);
            auto q2 = [](uint32_t w, float sc) -> uint32_t {
                // two bf16 -> two e4m3 (low element in the low byte)
                const float lo = __fdiv_rn(bf16_lo(w), sc);
                const float hi = __fdiv_rn(bf16_hi(w), sc);
                uint16_t r;
                asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
                return r;
            };
            uint2 ko, vo;
            ko.x = q2(kx.x, sk) | (q2(kx.y, sk) << 16);
            ko.y = q2(kx.z, sk) | (q2(kx.w, sk) << 16);
            vo.x = q2(vx.x, sv) | (q2(vx.y, sv) << 16);
            vo.y = q2(vx.z, sv) | (q2(vx.w, sv) << 16);
            *reinterpret_cast<uint2 *>(kc + dst) = ko;
            *reinterpret_cast<uint2 *>(vc + dst) = vo;
        }
    }
}

// Copies every (head) tile of block src to block dst, K and V.
__global__ void __launch_bounds__(256)
    block_copy_kernel(uint4 *__restrict__ kc, uint4 *__restrict__ vc, int64_t src, int64_t dst,
                      int64_t chunks_per_block)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < chunks_per_block;
         i += (int64_t)gridDim.x * blockDim.x) {
        kc[dst * chunks_per_block + i] = kc[src * chunks_per_block + i];
        vc[dst * chunks_per_block + i] = vc[src * chunks_per_block + i];
    }
}

// Failure-path self-test: one thread waits, with the given limit, on an
// mbarrier phase that nothing completes -- the bounded wait every pipeline wait
// uses -- gives up, and records ST_TIMEOUT in the status word.  Nothing faults
// or traps, and the context stays usable.  The loop ends on the clock or, as a
// second bound, after 2^20 tries.
__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(unsigned long long limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 0; it < (1u << 20); ++it) {
        if (mbar_try_wait(b, 0)) return;           // nothing ever arrives on this barrier
        if (globaltimer() - t0 > limit_ns) break;
    }
    atomicOr(&g_status, ST_TIMEOUT);
}

}  // namespace

namespace pkv_decode { uint32_t take_status(); }
namespace pkv_prefill { uint32_t take_status(); }
namespace pkv_swap { uint32_t take_status(); }

static uint32_t take_status_cache()
{
    uint32_t v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_status, &z, sizeof z);
    return v;
}

static std::atomic<uint32_t> g_last_flags{0};   // read from any host thread

kv_status pkv_launch_block_copy(void *k_cache, void *v_cache, int32_t src, int32_t dst,
                                int32_t num_kv_heads, kv_dtype dtype, cudaStream_t stream)
{
    if (!pkv_host::aligned(k_cache, 16) || !pkv_host::aligned(v_cache, 16)) return KV_ERR_INVALID;
    const int64_t bytes = (int64_t)num_kv_heads * BS * D * (dtype == KV_BF16 ? 2 : 1);
    const int64_t chunks = bytes / 16;
    const int threads = 256;
    const int blocks = static_cast<int>(std::min<int64_t>((chunks + threads - 1) / threads, 1024));
    block_copy_kernel<<<blocks, threads, 0, stream>>>(static_cast<uint4 *>(k_cache),
                                                       static_cast<uint4 *>(v_cache), src, dst,
                                                       chunks);
    return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

extern "C" {

kv_status reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                            const int64_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                            int32_t num_blocks, kv_dtype dtype, const float *k_scale,
                            const float *v_scale, void *stream)
{
    PKV_NVTX_RANGE("reshape_and_cache");
    if (num_tokens == 0) return KV_OK;
    if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 1) return KV_ERR_INVALID;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return KV_ERR_INVALID;
    if (dtype != KV_BF16 && dtype != KV_FP8_E4M3) return KV_ERR_UNSUPPORTED;
    if (dtype == KV_FP8_E4M3 && (!k_scale || !v_scale)) return KV_ERR_INVALID;
    if (!pkv_host::aligned(k, 16) || !pkv_host::aligned(v, 16) || !pkv_host::aligned(k_cache, 16) ||
        !pkv_host::aligned(v_cache, 16) || !pkv_host::aligned(slot_mapping, 8))
        return KV_ERR_INVALID;
    const int64_t total = (int64_t)num_tokens * num_kv_heads * 16;
    const int threads = 256;
    const int64_t want = (total + threads - 1) / threads;
    const int blocks = static_cast<int>(std::min<int64_t>(want, 152 * 16));
    const int64_t num_slots = (int64_t)num_blocks * BS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == KV_BF16)
        reshape_and_cache_kernel<false><<<blocks, threads, 0, st>>>(
            static_cast<const uint4 *>(k), static_cast<const uint4 *>(v),
            static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), slot_mapping, total,
            num_kv_heads, num_slots, nullptr, nullptr);
    else
        reshape_and_cache_kernel<true><<<blocks, threads, 0, st>>>(
            static_cast<const uint4 *>(k), static_cast<const uint4 *>(v),
            static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), slot_mapping, total,
            num_kv_heads, num_slots, k_scale, v_scale);
    return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

kv_status kv_last_device_status(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KV_ERR_CUDA;
    uint32_t f = take_status_cache() | pkv_decode::take_status() | pkv_prefill::take_status() |
                 pkv_swap::take_status();
    g_last_flags.store(f, std::memory_order_relaxed);
    return f ? KV_ERR_DEVICE_BOUNDS : KV_OK;
}

uint32_t kv_last_device_status_flags(void) { return g_last_flags.load(std::memory_order_relaxed); }

kv_status kv_selftest_bounded_wait(uint32_t limit_us, void *stream)
{
    if (limit_us == 0 || limit_us > 2000000u) return KV_ERR_INVALID;
    bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        (unsigned long long)limit_us * 1000ull);
    return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

}  // extern "C"
