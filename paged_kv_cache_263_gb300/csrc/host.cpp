// host.cpp -- host side of the paged KV-cache library: the block manager
// (free-list pool, refcounts, copy-on-write bookkeeping), status strings and
// TMA tensor-map encoding.
//
// Block management follows "M.65 Inference serving", PagedAttention block
// management: (b) a per-request block table of block ids, (c) O(1) allocation
// from a free list, every block returned when the request completes, (e)
// reference-counted sharing of prefix blocks (refcount 2 -> 1 -> 0, free at 0),
// (g) copy-on-write when shared generations diverge; and "Waste, and three ways
// to reclaim it", section "Sharing, and what makes a prefix reusable" (one
// physical copy, many block tables; a writer first gets its own copy).
#include <cuda.h>
#include "trace.h"
#include <cuda_runtime.h>

#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"
#include "common.cuh"

struct kv_pool {
    int32_t num_blocks = 0;
    std::vector<int32_t> stack;  // top (back) = next block handed out
    std::vector<int32_t> ref;
    int64_t cow_copies = 0;
    int64_t alloc_failures = 0;
    int32_t fail_after = 0;      // fault injection: fail the k-th alloc from now
    mutable std::mutex mu;
};

// launches the block copy of copy-on-write (cache_ops.cu)
extern "C++" kv_status pkv_launch_block_copy(void *k_cache, void *v_cache, int32_t src,
                                             int32_t dst, int32_t num_kv_heads, kv_dtype dtype,
                                             cudaStream_t stream);

namespace {

// consumes one "allocation attempt" of the fault-injection counter; true = fail
bool injected_failure(kv_pool *p)
{
    if (p->fail_after <= 0) return false;
    if (--p->fail_after == 0) return true;
    return false;
}

kv_status alloc_locked(kv_pool *p, int32_t n, int32_t *out)
{
    if (n < 0 || (n > 0 && !out)) return KV_ERR_INVALID;
    if (injected_failure(p) || static_cast<size_t>(n) > p->stack.size()) {
        p->alloc_failures++;
        return KV_ERR_OUT_OF_BLOCKS;
    }
    for (int32_t i = 0; i < n; ++i) {
        int32_t b = p->stack.back();
        p->stack.pop_back();
        p->ref[b] = 1;
        out[i] = b;
    }
    return KV_OK;
}

// every id in ids[0..n) must hold at least `need_each` references, counting
// repeats (need_each = 0 means: as many references as occurrences)
bool check_live(const kv_pool *p, const int32_t *ids, int32_t n, bool count_repeats)
{
    if (n < 0 || (n > 0 && !ids)) return false;
    std::unordered_map<int32_t, int32_t> cnt;
    for (int32_t i = 0; i < n; ++i) {
        int32_t b = ids[i];
        if (b < 0 || b >= p->num_blocks) return false;
        cnt[b]++;
    }
    for (auto &kv : cnt) {
        int32_t need = count_repeats ? kv.second : 1;
        if (p->ref[kv.first] < need) return false;
    }
    return true;
}

}  // namespace

extern "C" {

const char *kv_status_string(kv_status s)
{
    switch (s) {
    case KV_OK: return "ok";
    case KV_ERR_INVALID: return "invalid argument";
    case KV_ERR_OUT_OF_BLOCKS: return "out of blocks";
    case KV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case KV_ERR_CUDA: return "CUDA error";
    case KV_ERR_DEVICE_BOUNDS: return "device data out of range";
    }
    return "unknown status";
}

kv_status kv_pool_create(int32_t num_blocks, const int32_t *initial_free_order, kv_pool **out)
{
    if (!out || num_blocks < 1) return KV_ERR_INVALID;
    kv_pool *p = new (std::nothrow) kv_pool;
    if (!p) return KV_ERR_INVALID;
    p->num_blocks = num_blocks;
    p->ref.assign(num_blocks, 0);
    p->stack.resize(num_blocks);
    if (initial_free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            int32_t b = initial_free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete p;
                return KV_ERR_INVALID;
            }
            seen[b] = 1;
            p->stack[num_blocks - 1 - i] = b;
        }
    } else {
        for (int32_t i = 0; i < num_blocks; ++i) p->stack[num_blocks - 1 - i] = i;
    }
    *out = p;
    return KV_OK;
}

void kv_pool_destroy(kv_pool *pool) { delete pool; }

kv_status kv_block_alloc(kv_pool *pool, int32_t n, int32_t *out_ids)
{
    if (!pool) return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(pool->mu);
    return alloc_locked(pool, n, out_ids);
}

kv_status kv_block_free(kv_pool *pool, const int32_t *ids, int32_t n)
{
    if (!pool) return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(pool->mu);
    if (!check_live(pool, ids, n, true)) return KV_ERR_INVALID;
    for (int32_t i = 0; i < n; ++i) {
        int32_t b = ids[i];
        if (--pool->ref[b] == 0) pool->stack.push_back(b);
    }
    return KV_OK;
}

kv_status kv_block_share(kv_pool *pool, const int32_t *ids, int32_t n)
{
    if (!pool) return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(pool->mu);
    if (!check_live(pool, ids, n, false)) return KV_ERR_INVALID;
    for (int32_t i = 0; i < n; ++i) pool->ref[ids[i]]++;
    return KV_OK;
}

kv_status kv_copy_on_write(kv_pool *pool, int32_t id, int32_t *out_id, void *k_cache,
                           void *v_cache, int32_t num_kv_heads, kv_dtype dtype, void *stream)
{
    PKV_NVTX_RANGE("kv_copy_on_write");
    if (!pool || !out_id) return KV_ERR_INVALID;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return KV_ERR_INVALID;
    if (k_cache && (num_kv_heads < 1 || (dtype != KV_BF16 && dtype != KV_FP8_E4M3)))
        return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(pool->mu);
    if (id < 0 || id >= pool->num_blocks || pool->ref[id] < 1) return KV_ERR_INVALID;
    if (pool->ref[id] == 1) {
        *out_id = id;
        return KV_OK;
    }
    int32_t nb;
    kv_status st = alloc_locked(pool, 1, &nb);
    if (st != KV_OK) return st;
    if (k_cache) {
        st = pkv_launch_block_copy(k_cache, v_cache, id, nb, num_kv_heads, dtype,
                                   static_cast<cudaStream_t>(stream));
        if (st != KV_OK) {  // roll back: the pool is left as it was
            pool->ref[nb] = 0;
            pool->stack.push_back(nb);
            return st;
        }
    }
    pool->ref[id]--;
    pool->cow_copies++;
    *out_id = nb;
    return KV_OK;
}

kv_status kv_block_refcount(const kv_pool *pool, int32_t id, int32_t *out)
{
    if (!pool || !out) return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(pool->mu);
    if (id < 0 || id >= pool->num_blocks) return KV_ERR_INVALID;
    *out = pool->ref[id];
    return KV_OK;
}

kv_status kv_pool_stats(const kv_pool *pool, kv_pool_stats_t *out)
{
    if (!pool || !out) return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(pool->mu);
    int32_t live = 0, shared = 0;
    for (int32_t r : pool->ref) {
        live += r > 0;
        shared += r > 1;
    }
    out->num_blocks = pool->num_blocks;
    out->free_blocks = static_cast<int32_t>(pool->stack.size());
    out->live_blocks = live;
    out->shared_blocks = shared;
    out->cow_copies = pool->cow_copies;
    out->alloc_failures = pool->alloc_failures;
    return KV_OK;
}

kv_status kv_waste_stats(const int32_t *lens, int32_t n, int32_t reservation_tokens, kv_waste_stats_t *out)
{
    if (!out || n < 0 || reservation_tokens < 0 || (n > 0 && !lens)) return KV_ERR_INVALID;
    int64_t used = 0, blocks = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (lens[i] < 0 || lens[i] > reservation_tokens) return KV_ERR_INVALID;
        used += lens[i];
        blocks += (lens[i] + 15) / 16;
    }
    out->used_tokens = used;
    out->contiguous_reserved_slots = (int64_t)reservation_tokens * n;
    out->contiguous_untouched_slots = out->contiguous_reserved_slots - used;
    out->paged_blocks = blocks;
    out->paged_slots = blocks * 16;
    out->paged_waste_slots = out->paged_slots - used;
    out->contiguous_untouched_percent =
        out->contiguous_reserved_slots ? 100.0 * (double)out->contiguous_untouched_slots /
                                             (double)out->contiguous_reserved_slots
                                       : 0.0;
    out->paged_waste_percent =
        out->paged_slots ? 100.0 * (double)out->paged_waste_slots / (double)out->paged_slots : 0.0;
    return KV_OK;
}

kv_status kv_pool_fail_alloc_after(kv_pool *pool, int32_t k)
{
    if (!pool) return KV_ERR_INVALID;
    std::lock_guard<std::mutex> g(pool->mu);
    pool->fail_after = k > 0 ? k : 0;
    return KV_OK;
}

}  // extern "C"

// ------------------------------------------------------------ tensor maps
namespace pkv_host {

namespace {
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode()
{
    static EncodeFn fn = []() -> EncodeFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeFn>(p);
    }();
    return fn;
}
}  // namespace

bool encode_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, uint64_t dim0,
                    uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                    CUtensorMapSwizzle swizzle)
{
    EncodeFn fn = get_encode();
    if (!fn) return false;
    cuuint64_t dims[2] = {dim0, dim1};
    cuuint64_t strides[1] = {stride1_bytes};
    cuuint32_t box[2] = {box0, box1};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, uint64_t dim0,
                    uint64_t dim1, uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                    uint32_t box0, uint32_t box1, uint32_t box2, CUtensorMapSwizzle swizzle)
{
    EncodeFn fn = get_encode();
    if (!fn) return false;
    cuuint64_t dims[3] = {dim0, dim1, dim2};
    cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    cuuint32_t box[3] = {box0, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pkv_host
