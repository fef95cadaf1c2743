// swap.cu -- swap-out of KV blocks to host memory and swap-in back into the
// paged caches (sm_103a).
//
// When the cache is full mid-generation a request can be preempted and its
// blocks shipped to host memory, to be brought back later wherever the pool
// has room ("Waste, and three ways to reclaim it", section "When it runs out
// anyway": swap to host memory instead of recomputing the prefill; "M.65
// Inference serving", block management (f) preemption).
//
// Design (GB300): the GPU reaches its Grace host's memory over NVLink-C2C, so
// the SMs move the data themselves -- one kernel gathers the scattered (block,
// KV head) tiles of both caches straight into page-locked host memory (or
// scatters them back), with no device staging buffer and no per-block copy
// launches.  Each thread moves 16-byte units; consecutive lanes take
// consecutive units of one block, so every warp writes 512 contiguous bytes,
// and each thread keeps UNROLL units in flight to cover the link's latency.
// The grid is a whole number of waves over the 152 SMs.
#include "common.cuh"
#include "trace.h"

#include <algorithm>

namespace {

__device__ uint32_t g_status;

using namespace pkv;

constexpr int THREADS = 256;
constexpr int UNROLL = 4;

// to_host: cache tiles of ids[i] -> host slot i; else host slot i -> cache
// tiles of ids[i].  Units are 16 bytes; a block of one cache is upb units.
template <bool TO_HOST>
__global__ void __launch_bounds__(THREADS)
    swap_kernel(uint4 *__restrict__ kc, uint4 *__restrict__ vc, uint4 *__restrict__ hk, uint4 *__restrict__ hv,
                const int32_t *__restrict__ ids, int64_t n, int64_t upb, int32_t num_blocks)
{
    const int64_t per_cache = n * upb;
    const int64_t total = 2 * per_cache;
    const int64_t stride = (int64_t)gridDim.x * THREADS;
    for (int64_t base = blockIdx.x * (int64_t)THREADS + threadIdx.x; base < total; base += stride * UNROLL) {
        uint4 val[UNROLL];
        uint4 *dst[UNROLL];
#pragma unroll
        for (int r = 0; r < UNROLL; ++r) {
            dst[r] = nullptr;
            const int64_t u = base + r * stride;
            if (u >= total) continue;
            const bool is_v = u >= per_cache;
            const int64_t w = is_v ? u - per_cache : u;
            const int64_t i = w / upb, off = w - i * upb;
            const int32_t b = __ldg(ids + i);
            if (b < 0 || b >= num_blocks) {
                if (off == 0) atomicOr(&g_status, ST_BAD_BLOCK);
                continue;
            }
            uint4 *cache = (is_v ? vc : kc) + (int64_t)b * upb + off;
            uint4 *host = (is_v ? hv : hk) + i * upb + off;
            if constexpr (TO_HOST) {
                val[r] = __ldg(cache);
                dst[r] = host;
            } else {
                val[r] = *host;
                dst[r] = cache;
            }
        }
#pragma unroll
        for (int r = 0; r < UNROLL; ++r)
            if (dst[r]) *dst[r] = val[r];
    }
}

// device-visible address of a page-locked host range, or nullptr
void *device_view(const void *host, size_t bytes)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess || a.type != cudaMemoryTypeHost || !a.devicePointer) {
        cudaGetLastError();
        return nullptr;
    }
    cudaPointerAttributes e{};
    const void *last = static_cast<const uint8_t *>(host) + bytes - 1;
    if (cudaPointerGetAttributes(&e, last) != cudaSuccess || e.type != cudaMemoryTypeHost) {
        cudaGetLastError();
        return nullptr;
    }
    return a.devicePointer;
}

kv_status launch(bool to_host, void *k_cache, void *v_cache, int32_t num_blocks, int32_t num_kv_heads,
                 kv_dtype dtype, const int32_t *block_ids, int32_t n, const void *host_k, const void *host_v,
                 cudaStream_t st)
{
    if (n == 0) return KV_OK;
    if (n < 0 || num_blocks < 1 || num_kv_heads < 1 || !k_cache || !v_cache || !block_ids || !host_k ||
        !host_v)
        return KV_ERR_INVALID;
    if (dtype != KV_BF16 && dtype != KV_FP8_E4M3) return KV_ERR_UNSUPPORTED;
    if (!pkv_host::aligned(k_cache, 16) || !pkv_host::aligned(v_cache, 16) || !pkv_host::aligned(host_k, 16) ||
        !pkv_host::aligned(host_v, 16))
        return KV_ERR_INVALID;
    const int64_t block_bytes = (int64_t)num_kv_heads * BS * D * (dtype == KV_BF16 ? 2 : 1);
    const size_t host_bytes = (size_t)n * block_bytes;
    void *dk = device_view(host_k, host_bytes);
    void *dv = device_view(host_v, host_bytes);
    if (!dk || !dv) return KV_ERR_INVALID;
    const int64_t upb = block_bytes / 16;
    const int64_t units = 2 * (int64_t)n * upb;
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (units + (int64_t)THREADS * UNROLL - 1) / ((int64_t)THREADS * UNROLL);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * 8));
    auto *kc = static_cast<uint4 *>(k_cache);
    auto *vc = static_cast<uint4 *>(v_cache);
    if (to_host)
        swap_kernel<true><<<grid, THREADS, 0, st>>>(kc, vc, static_cast<uint4 *>(dk), static_cast<uint4 *>(dv),
                                                    block_ids, n, upb, num_blocks);
    else
        swap_kernel<false><<<grid, THREADS, 0, st>>>(kc, vc, static_cast<uint4 *>(dk), static_cast<uint4 *>(dv),
                                                     block_ids, n, upb, num_blocks);
    return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

}  // namespace

namespace pkv_swap {
uint32_t take_status()
{
    uint32_t v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_status, &z, sizeof z);
    return v;
}
}  // namespace pkv_swap

extern "C" {

kv_status kv_swap_out(const void *k_cache, const void *v_cache, int32_t num_blocks, int32_t num_kv_heads,
                      kv_dtype dtype, const int32_t *block_ids, int32_t n, void *host_k, void *host_v,
                      void *stream)
{
    PKV_NVTX_RANGE("kv_swap_out");
    return launch(true, const_cast<void *>(k_cache), const_cast<void *>(v_cache), num_blocks, num_kv_heads, dtype,
                  block_ids, n, host_k, host_v, static_cast<cudaStream_t>(stream));
}

kv_status kv_swap_in(void *k_cache, void *v_cache, int32_t num_blocks, int32_t num_kv_heads, kv_dtype dtype,
                     const int32_t *block_ids, int32_t n, const void *host_k, const void *host_v, void *stream)
{
    PKV_NVTX_RANGE("kv_swap_in");
    return launch(false, k_cache, v_cache, num_blocks, num_kv_heads, dtype, block_ids, n, host_k, host_v,
                  static_cast<cudaStream_t>(stream));
}

}  // extern "C"
