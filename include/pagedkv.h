/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache attention library.
 *
 * The library implements the data-parallel hot path of PagedAttention: a KV
 * cache held in fixed 16-token physical blocks, reached through a
 * per-sequence block table, with GQA head groups, ref-counted shared-prefix
 * blocks with copy-on-write, chunked-prefill query chunks mixed with decode
 * queries, split-KV partitions merged by a log-sum-exp reduction, and an
 * fp8-e4m3 cache.
 *
 * Sources (web pages; cited by title and section):
 *  [P1] "PagedAttention, chunked prefill, and the launch that cascades"
 *       (deepnotes.pages.dev), sections "PagedAttention: an OS idea, not an ML
 *       one", "Serving systems: the layer that survives real traffic",
 *       "FlashAttention: why the mechanism this whole layer runs on isn't
 *       compute-bound", "Kernel engineering: the layer underneath everything
 *       else here".
 *  [P2] "Waste, and three ways to reclaim it" (runbooks.in, Document 10 - Quick
 *       learn), sections "PagedAttention - operating-system virtual memory,
 *       applied to attention", "Sharing, and what makes a prefix reusable",
 *       "Quantising the cache".
 *  [P3] "M.65 Inference serving" (systemdesigntutorial.com), paragraphs on the
 *       KV-cache memory math, PagedAttention block management (a)-(h),
 *       prefill vs decode (a)-(f), and quantisation (a)-(f).
 *
 * Conventions for every call:
 *  - Fixed geometry: head_dim D = 128 and block size BS = 16 tokens ([P3] block
 *    management (a): fixed at compile time, 16 tokens).  Other values are not
 *    representable in the ABI.
 *  - Cache layout (chosen here; the pages give none): k_cache and v_cache are
 *    each [num_blocks][num_kv_heads][16][128] elements of the cache dtype, so one
 *    (block, kv head) tile is contiguous: 4 KiB in bf16, 2 KiB in fp8.
 *  - Query/output layout: q is [rows][num_q_heads][128] bf16; out is
 *    [rows][num_q_heads][128] fp32.  Query head h reads KV head h / G, with
 *    G = num_q_heads / num_kv_heads (the repeat_interleave grouping of [P1]
 *    "Kernel engineering"); G must be 1, 2, 4, 8 or 16.
 *  - Block ids are int32.  Unused block-table entries may hold any value; only
 *    the first ceil(context_len / 16) entries of a row are read.
 *  - Ownership: every device buffer (caches, q, out, tables, lengths, slot
 *    mapping, scales, workspace) belongs to the caller; the attention and
 *    cache-write calls allocate no device memory.  A kv_pool is a host object
 *    owned by the library between kv_pool_create and kv_pool_destroy.
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  Device
 *    work is enqueued asynchronously; the calls return once it is launched.
 *  - Errors: every call returns a kv_status; nothing is thrown across the ABI.
 *    Host-visible argument errors are reported before anything is launched
 *    (KV_ERR_INVALID / KV_ERR_UNSUPPORTED); launch failures as KV_ERR_CUDA.
 *    Errors that only device data can show (a block id outside the pool, a slot
 *    outside the pool, a context length outside [1, max_blocks_per_seq*16], a
 *    query chunk longer than its context, a pipeline wait that timed out) never
 *    fault: the kernel skips the offending access, sets a sticky device status
 *    word and continues; kv_last_device_status() reports and clears it.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PAGEDKV_API __attribute__((visibility("default")))
#else
#define PAGEDKV_API
#endif

#define PAGEDKV_HEAD_DIM 128
#define PAGEDKV_BLOCK_SIZE 16

typedef enum {
    KV_OK = 0,
    KV_ERR_INVALID = 1,        /* bad argument, double free, sharing a free block */
    KV_ERR_OUT_OF_BLOCKS = 2,  /* pool exhausted; the pool is left unchanged */
    KV_ERR_UNSUPPORTED = 3,    /* shape or dtype this library does not handle */
    KV_ERR_CUDA = 4,           /* a CUDA runtime/driver call or launch failed */
    KV_ERR_DEVICE_BOUNDS = 5   /* device data was out of range (see above) */
} kv_status;

typedef enum { KV_BF16 = 0, KV_FP8_E4M3 = 1 } kv_dtype;

typedef struct kv_pool kv_pool; /* opaque, host-only */

typedef struct {
    int32_t num_blocks;      /* pool size */
    int32_t free_blocks;     /* blocks on the free list */
    int32_t live_blocks;     /* blocks with refcount >= 1 */
    int32_t shared_blocks;   /* blocks with refcount >= 2 */
    int64_t cow_copies;      /* copy-on-write forks that copied a block */
    int64_t alloc_failures;  /* allocations refused for lack of blocks */
} kv_pool_stats_t;

/* Human-readable name of a status code (static storage). */
PAGEDKV_API const char *kv_status_string(kv_status s);

/* ------------------------------------------------------------------------
 * Host block manager: free-list pool, block ids, refcounts, copy-on-write.
 * [P3] block management (b) per-request block table, (c) O(1) allocation from
 * a free list and return of all blocks on completion, (e) reference-counted
 * prefix sharing, (g) copy-on-write; [P2] "Sharing, and what makes a prefix
 * reusable" (one physical copy, many block tables; copy on write).
 * Free-list order is deterministic: a LIFO stack whose first hand-out is
 * initial_free_order[0] (ascending ids when NULL); a freed block is the next
 * one handed out.  All calls on one pool are serialised by a mutex.
 * ---------------------------------------------------------------------- */

/* Creates a pool of num_blocks (>= 1) blocks.  initial_free_order, if not NULL,
 * must be a permutation of 0..num_blocks-1 (KV_ERR_INVALID otherwise). */
PAGEDKV_API kv_status kv_pool_create(int32_t num_blocks, const int32_t *initial_free_order, kv_pool **out);
PAGEDKV_API void kv_pool_destroy(kv_pool *pool);

/* Allocates n (>= 0) blocks into out_ids[0..n) with refcount 1.  All-or-nothing:
 * on KV_ERR_OUT_OF_BLOCKS nothing changes except stats.alloc_failures. */
PAGEDKV_API kv_status kv_block_alloc(kv_pool *pool, int32_t n, int32_t *out_ids);

/* Drops one reference per listed id (an id may repeat, once per reference it
 * drops); a block reaching refcount 0 returns to the free list, in list order.
 * Validated first: any id not holding enough references -> KV_ERR_INVALID and
 * nothing changes. */
PAGEDKV_API kv_status kv_block_free(kv_pool *pool, const int32_t *ids, int32_t n);

/* Adds one reference per listed id; every id must be live (refcount >= 1),
 * else KV_ERR_INVALID and nothing changes. */
PAGEDKV_API kv_status kv_block_share(kv_pool *pool, const int32_t *ids, int32_t n);

/* Copy-on-write of block `id` before a write into it.
 *  refcount == 1: *out_id = id; nothing is copied.
 *  refcount >= 2: one new block is allocated (KV_ERR_OUT_OF_BLOCKS if none, pool
 *    unchanged), the caller's reference moves to it (old refcount - 1), and --
 *    if k_cache and v_cache are not NULL -- all num_kv_heads tiles of K and V of
 *    `id` are copied to the new block by a kernel on `stream`.  With both cache
 *    pointers NULL only the bookkeeping is done and the caller copies.
 *  The caches must hold the pool's num_blocks blocks in the layout above. */
PAGEDKV_API kv_status kv_copy_on_write(kv_pool *pool, int32_t id, int32_t *out_id, void *k_cache,
                           void *v_cache, int32_t num_kv_heads, kv_dtype dtype, void *stream);

/* Current refcount of block id (0 = free). */
PAGEDKV_API kv_status kv_block_refcount(const kv_pool *pool, int32_t id, int32_t *out);

PAGEDKV_API kv_status kv_pool_stats(const kv_pool *pool, kv_pool_stats_t *out);

/* Memory waste of a set of requests, contiguous against paged ([P2]
 * "PagedAttention": each request reserving a maximum-length buffer leaves most
 * of it untouched; "Small block size": paged waste is at most 15 tokens per
 * sequence; [P3] block management (a), (f) efficiency tracking).
 *  lens                host int32 [n], tokens of each request, 0..reservation_tokens
 *  reservation_tokens  slots a contiguous allocator reserves per request
 *  Contiguous: n x reservation_tokens slots reserved, those no token uses are
 *  untouched.  Paged: ceil(len/16) blocks per request; the unused slots of each
 *  last block are the waste.  KV_ERR_INVALID for a length outside the range. */
typedef struct {
    int64_t used_tokens;
    int64_t contiguous_reserved_slots;
    int64_t contiguous_untouched_slots;
    int64_t paged_blocks;
    int64_t paged_slots;
    int64_t paged_waste_slots;
    double contiguous_untouched_percent;
    double paged_waste_percent;
} kv_waste_stats_t;

PAGEDKV_API kv_status kv_waste_stats(const int32_t *lens, int32_t n, int32_t reservation_tokens,
                                     kv_waste_stats_t *out);

/* Host fault injection: the k-th kv_block_alloc call from now (k >= 1),
 * including the allocation inside kv_copy_on_write, fails with
 * KV_ERR_OUT_OF_BLOCKS exactly as if the pool were empty; k <= 0 disarms. */
PAGEDKV_API kv_status kv_pool_fail_alloc_after(kv_pool *pool, int32_t k);

/* ------------------------------------------------------------------------
 * Prefix cache: keeps the full blocks of finished requests so that a later
 * request starting with the same tokens reuses their K/V instead of
 * prefilling them again ([P1] opening section: hash the prefix, reuse the
 * computed blocks across requests; [P2] "Block sharing versus prefix
 * caching?", "SGLang -- RadixAttention": finished requests' cache filed in a
 * tree of shared beginnings, LRU eviction; [P3] block management (h)(ii)).
 *
 *  - Matching is on exact token ids, block-aligned, from the very start
 *    ([P2] "Why does my prefix cache hit rate not match what I expect?"): the
 *    cached block j of a sequence stands for tokens[0 .. 16(j+1)) under a
 *    tenant key `salt` ([P2] "The isolation question": key the cache per
 *    tenant).  Only full 16-token blocks are cached.  Lookup hashes the chain
 *    block by block; every candidate is then compared token by token with its
 *    parent identity, so a hash collision never returns a wrong block.
 *  - The cache holds one pool reference per cached block.  Blocks form a tree
 *    (block j's parent is block j-1 of the same prefix).  Eviction frees, one
 *    at a time, the least recently used leaf that only the cache holds
 *    (refcount 1); recency is a clock advanced once per match or insert and
 *    stamped on every block the call touches (ties: the block cached first).
 *  - Host only; all calls on one cache are serialised by its mutex.  The pool
 *    must outlive the cache.
 * ---------------------------------------------------------------------- */
typedef struct kv_prefix_cache kv_prefix_cache; /* opaque, host-only */

typedef struct {
    int64_t lookups;          /* kv_prefix_match calls */
    int64_t query_blocks;     /* full blocks asked for by those calls */
    int64_t hit_blocks;       /* full blocks they returned */
    int64_t inserted_blocks;  /* blocks newly cached */
    int64_t evicted_blocks;   /* blocks freed by eviction */
    int32_t cached_blocks;    /* blocks the cache holds now */
    int32_t evictable_blocks; /* of those, how many repeated eviction could free now */
} kv_prefix_stats_t;

/* Creates an empty cache over `pool` (not NULL). */
PAGEDKV_API kv_status kv_prefix_cache_create(kv_pool *pool, kv_prefix_cache **out);

/* Drops the cache's reference on every cached block, then frees the cache. */
PAGEDKV_API void kv_prefix_cache_destroy(kv_prefix_cache *cache);

/* Longest run of cached blocks matching tokens[0 .. n_tokens) from the start
 * under `salt`, at most max_blocks of them: their ids go to out_block_ids
 * (capacity max_blocks), their count to *out_n_blocks.  The caller receives one
 * pool reference per returned block (drop it with kv_block_free).  The blocks
 * returned are marked used now. */
PAGEDKV_API kv_status kv_prefix_match(kv_prefix_cache *cache, const int32_t *tokens, int32_t n_tokens,
                                      uint64_t salt, int32_t max_blocks, int32_t *out_block_ids,
                                      int32_t *out_n_blocks);

/* Caches the full blocks of a sequence: block j (j < min(n_tokens / 16,
 * n_blocks)) holds tokens[16j .. 16j+15] in physical block block_ids[j], whose
 * K/V the caller has written.  Every listed block must be live (KV_ERR_INVALID,
 * nothing changes, otherwise).  A block whose prefix is already cached keeps the
 * cached copy (marked used now); a new one gets one pool reference held by the
 * cache.  *out_n_new (nullable) = blocks newly cached. */
PAGEDKV_API kv_status kv_prefix_insert(kv_prefix_cache *cache, const int32_t *tokens, int32_t n_tokens,
                                       uint64_t salt, const int32_t *block_ids, int32_t n_blocks,
                                       int32_t *out_n_new);

/* Evicts up to n blocks (least recently used evictable leaf first), returning
 * them to the pool; their ids go to out_ids (nullable, capacity n) in eviction
 * order, their count to *out_n (nullable). */
PAGEDKV_API kv_status kv_prefix_evict(kv_prefix_cache *cache, int32_t n, int32_t *out_ids, int32_t *out_n);

/* kv_block_alloc on the cache's pool after evicting as many cached blocks as
 * the free list is short of n.  If the pool is still short the call fails with
 * KV_ERR_OUT_OF_BLOCKS; evictions it made stand. */
PAGEDKV_API kv_status kv_prefix_alloc(kv_prefix_cache *cache, int32_t n, int32_t *out_ids);

PAGEDKV_API kv_status kv_prefix_stats(const kv_prefix_cache *cache, kv_prefix_stats_t *out);

/* ------------------------------------------------------------------------
 * Cache write ("blocks allocated on demand as a sequence grows" [P1]
 * "PagedAttention: an OS idea"; [P3] block management (c)).
 *  k, v          device, bf16 [num_tokens][num_kv_heads][128]
 *  slot_mapping  device, int64 [num_tokens]; token t goes to block slot/16,
 *                offset slot%16; a negative slot skips the token (padding)
 *  k_cache/v_cache  device, layout above, num_blocks blocks
 *  dtype KV_BF16: the bytes are copied.  KV_FP8_E4M3: each element is stored as
 *    e4m3(round-to-nearest-even, saturating at +-448)(fp32(x) / scale[h]) with
 *    the IEEE fp32 division and per-KV-head k_scale/v_scale (device fp32
 *    [num_kv_heads]); [P2] "Quantising the cache", [P3] quantisation (b),(d).
 *  A slot >= num_blocks*16 is skipped and flagged (KV_ERR_DEVICE_BOUNDS).
 * ---------------------------------------------------------------------- */
PAGEDKV_API kv_status reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                            const int64_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                            int32_t num_blocks, kv_dtype dtype, const float *k_scale,
                            const float *v_scale, void *stream);

/* ------------------------------------------------------------------------
 * Paged attention, decode: one query token per sequence at position
 * context_len-1, attending keys 0..context_len-1 read through the block table
 * ([P2] "PagedAttention", "a matching attention kernel that knows how to read
 * from scattered blocks"; [P3] block management (d)).  Softmax is computed
 * online, block by block ([P1] "FlashAttention": running max and normaliser).
 * Long contexts are cut into split-KV partitions of whole logical blocks;
 * partitions are merged with a log-sum-exp reduction (the running max and
 * normaliser of two partitions combine exactly).  Split points depend only on
 * logical positions, and no atomics touch the arithmetic, so the output is
 * bitwise identical under any physical placement of the blocks.
 *
 *  out            device fp32 [num_seqs][num_q_heads][128]
 *  q              device bf16 [num_seqs][num_q_heads][128]
 *  block_tables   device int32 [num_seqs][max_blocks_per_seq]
 *  context_lens   device int32 [num_seqs], 1 <= len <= max_blocks_per_seq*16
 *  scale          softmax scale (1/sqrt(128) for the standard head)
 *  dtype          cache element type; for KV_FP8_E4M3 k_scale/v_scale are the
 *                 device fp32 [num_kv_heads] dequantisation scales, one per KV
 *                 head and separate for K and V: query head h reads KV head
 *                 g = h / (num_q_heads / num_kv_heads), its keys are e4m3 x
 *                 k_scale[g] and its values e4m3 x v_scale[g].
 *                 Query range with KV_FP8_E4M3: the kernels multiply in f16, so
 *                 each bf16 query component is rounded to f16 once -- exact for
 *                 2^-14 <= |q| < 65,520; smaller magnitudes keep fewer bits
 *                 (f16 subnormals; zero at or below 2^-25), and |q| >= 65,520 becomes
 *                 infinite (the output is then NaN).  The bf16 cache has no such
 *                 limit: Q stays bf16.
 *  num_splits     maximum partitions per sequence; partition length is
 *                 ceil(max_blocks_per_seq / num_splits) blocks.  0 = choose.
 *  workspace      device scratch of at least paged_attention_workspace_size()
 *                 bytes (256-byte aligned), or NULL when that size is 0.
 * ---------------------------------------------------------------------- */
PAGEDKV_API size_t paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                      int32_t max_blocks_per_seq, int32_t num_splits);

PAGEDKV_API kv_status paged_attention_decode(float *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 int32_t max_blocks_per_seq, const int32_t *context_lens,
                                 int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t num_blocks, float scale, kv_dtype dtype,
                                 const float *k_scale, const float *v_scale, int32_t num_splits,
                                 void *workspace, size_t workspace_bytes, void *stream);

/* Decode for callers that cannot allocate device memory.  The paper has no
 * counterpart of this call; it is an addition of this library.  Some callers cannot call cudaMalloc
 * where they run attention -- code inside an allocator or memory-pool hook of
 * its own, a serving runtime that forbids allocation once it is up, or a host
 * that links this library without any allocator -- so they cannot provide the
 * workspace paged_attention_decode needs for split-KV partials.  This call is
 * paged_attention_decode with that scratch held in one fixed-size device array
 * inside the library (paged_attention_decode_static_scratch_bytes(): 32 MiB),
 * which every GPU that loads the library keeps until the process exits.  The
 * caller still passes every input and output.
 *  - A call whose partials need more than that size returns KV_ERR_UNSUPPORTED
 *    and launches nothing.  The call allocates no memory of any kind.
 *  - All calls share the array: calls that overlap on the GPU (other streams,
 *    other host threads on the same device) race on it and must be serialised.
 *    It keeps the last call's contents; nothing in it has to start at zero.
 *  - The first call on a device looks up the array's device address with that
 *    device current; make that first call before any stream capture.  The
 *    address is kept with the context that was current; after a device reset
 *    (a new context) the next call looks it up again, so that call also
 *    belongs outside any capture. */
PAGEDKV_API size_t paged_attention_decode_static_scratch_bytes(void);
PAGEDKV_API kv_status paged_attention_decode_static_scratch(
    float *out, const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t num_blocks, float scale, kv_dtype dtype, const float *k_scale,
    const float *v_scale, int32_t num_splits, void *stream);

/* ------------------------------------------------------------------------
 * Paged attention over a mixed batch of chunked-prefill and decode queries
 * ([P1] "Serving systems": long prompts split into ~1K-token chunks interleaved
 * with decode; [P3] prefill vs decode (e)).  Sequence s owns query rows
 * cu_q_lens[s] .. cu_q_lens[s+1]-1; its n_s rows sit at positions
 * context_len-n_s .. context_len-1, row i attends keys 0 .. context_len-n_s+i
 * (causal inside the chunk, everything before it visible).  Rows with n_s = 1
 * are decode rows and take the decode kernel; with a bf16 cache, chunks
 * (n_s >= 2) take the tensor-core (tcgen05) kernel.  Every kernel of the call
 * runs on `stream`: the decode kernel is launched programmatically right behind
 * the chunk kernel and runs beside it, on a few SMs that the chunk kernel
 * leaves free while it computes, then on all of them; work enqueued on `stream`
 * afterwards sees the whole output.  When total_q_tokens = num_seqs x max_q_len
 * every query is max_q_len rows long, so there are no decode rows (a query of 1
 * row is then flagged as out of range).  Short
 * chunks -- max_q_len x (num_q_heads / num_kv_heads) <= 8, e.g. a speculative
 * draft of 2 tokens under a GQA group of 4 ([P3] speculative decoding) -- run
 * instead with the whole batch in the decode kernel, whose CTA then covers all
 * rows of a sequence so each K/V tile is read once; longer drafts (N = 4-8)
 * take the tensor-core kernel.  With an fp8 cache the chunks run
 * on the tensor cores as well: each e4m3 K/V tile is widened exactly to f16
 * operands, Q is rounded to f16 once (the query range of the decode call above
 * applies), and the products accumulate in fp32.
 * The tensor-core kernel runs one CTA per SM over a work list the library
 * builds on the device (query tile, KV head and key partition, longest first).
 * A chunk's keys are cut into equal partitions of at most 16,384 keys, or left
 * whole, merged with the same log-sum-exp reduction; the library picks the
 * partition length from the batch shape and the context lengths (num_splits
 * applies to the decode rows), so a row's last bits may differ between batches
 * of different shapes or lengths, never with the physical placement of the
 * blocks.
 *
 *  out, q          device [total_q_tokens][num_q_heads][128] (fp32 / bf16)
 *  cu_q_lens       device int32 [num_seqs+1], cu_q_lens[0] = 0, non-decreasing,
 *                  cu_q_lens[num_seqs] = total_q_tokens
 *  context_lens    device int32 [num_seqs]; includes the chunk; n_s <= len
 *  max_q_len       host int: an upper bound on every n_s (sizes the grid and the
 *                  plan; a longer query is flagged as out of range and left out)
 *  other arguments as for paged_attention_decode; workspace must be at least
 *  paged_attention_chunked_prefill_workspace_size() bytes (one size serves
 *  both cache dtypes).
 * ---------------------------------------------------------------------- */
PAGEDKV_API size_t paged_attention_chunked_prefill_workspace_size(int32_t num_seqs, int32_t total_q_tokens,
                                                      int32_t max_q_len, int32_t num_q_heads,
                                                      int32_t num_kv_heads,
                                                      int32_t max_blocks_per_seq,
                                                      int32_t num_splits);

/* Number of kernels one successful paged_attention_chunked_prefill call with
 * these sizes enqueues on the caller's stream (host-only; reads no device
 * memory).  With max_q_len = 1 it is also
 * the count of a paged_attention_decode call with the same num_seqs,
 * num_q_heads, max_blocks_per_seq and num_splits.  Returns 0 for sizes a call
 * would accept without launching anything (no sequences or no query rows) and
 * for sizes it would reject. */
PAGEDKV_API int32_t paged_attention_launch_count(int32_t num_seqs, int32_t total_q_tokens, int32_t max_q_len,
                                                 int32_t num_q_heads, int32_t num_kv_heads,
                                                 int32_t max_blocks_per_seq, int32_t num_splits);

PAGEDKV_API kv_status paged_attention_chunked_prefill(float *out, const void *q, const int32_t *cu_q_lens,
                                          const int32_t *context_lens, int32_t num_seqs,
                                          int32_t total_q_tokens, int32_t max_q_len,
                                          const void *k_cache, const void *v_cache,
                                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                                          int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t num_blocks, float scale, kv_dtype dtype,
                                          const float *k_scale, const float *v_scale,
                                          int32_t num_splits, void *workspace,
                                          size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Swap of KV blocks to host memory and back ([P2] "When it runs out anyway":
 * ship a preempted request's blocks over the host link and bring them back;
 * [P3] block management (f) preemption, swap out to CPU).
 *
 *  kv_swap_out copies, for i < n, every (block, KV head) tile of K and V of
 *  block block_ids[i] to host_k[i] / host_v[i]; kv_swap_in copies host_k[i] /
 *  host_v[i] into block block_ids[i] (the ids of a swap-in must be distinct; the
 *  blocks may differ from the ones swapped out -- rewrite the block table).
 *
 *  k_cache/v_cache  device, the pool layout above, num_blocks blocks
 *  block_ids        device int32 [n]; an id outside 0..num_blocks-1 is skipped
 *                   and flagged (KV_ERR_DEVICE_BOUNDS, flag 1)
 *  host_k/host_v    page-locked host memory the device can address
 *                   (cudaHostAlloc / cudaHostRegister), each
 *                   n x num_kv_heads x 16 x 128 elements of the cache dtype in
 *                   list order, 16-byte aligned; other memory -> KV_ERR_INVALID
 *  One kernel on `stream` moves the data over the host link; the host buffers
 *  must stay valid until the stream has passed it.
 * ---------------------------------------------------------------------- */
PAGEDKV_API kv_status kv_swap_out(const void *k_cache, const void *v_cache, int32_t num_blocks,
                                  int32_t num_kv_heads, kv_dtype dtype, const int32_t *block_ids, int32_t n,
                                  void *host_k, void *host_v, void *stream);

PAGEDKV_API kv_status kv_swap_in(void *k_cache, void *v_cache, int32_t num_blocks, int32_t num_kv_heads,
                                 kv_dtype dtype, const int32_t *block_ids, int32_t n, const void *host_k,
                                 const void *host_v, void *stream);

/* Tracing aid.  While enabled, each paged_attention_chunked_prefill call records
 * CUDA events around its tensor-core chunk kernel on `stream` (only outside
 * stream capture); kv_trace_prefill_kernel_ms waits for the last such kernel of
 * the current device and returns its duration in ms, or a negative value if no
 * kernel was recorded since the previous query. */
PAGEDKV_API kv_status kv_trace_prefill(int32_t enable);
PAGEDKV_API double kv_trace_prefill_kernel_ms(void);

/* Waits for `stream`, then returns and clears the sticky device status word
 * set by earlier calls (KV_OK or KV_ERR_DEVICE_BOUNDS); KV_ERR_CUDA if the
 * stream itself reports an error. */
PAGEDKV_API kv_status kv_last_device_status(void *stream);

/* Bit flags of the last non-OK device status (0 if none), for diagnostics:
 * 1 block id outside the pool, 2 slot outside the pool, 4 bad context length
 * or chunk, 8 a pipeline wait timed out.  Read together with
 * kv_last_device_status (which clears them). */
PAGEDKV_API uint32_t kv_last_device_status_flags(void);

/* Self-test of the failure path ([P3] failure handling is the serving
 * system's; here: every device-side wait is bounded).  Launches one CTA on
 * `stream` whose thread waits, at most limit_us microseconds (1 .. 2,000,000),
 * on an mbarrier phase that nothing completes -- the same kind of bounded wait
 * the attention pipelines use -- then gives up and sets the timeout flag (8) in
 * the device status word.  Nothing faults, traps or hangs; the next
 * kv_last_device_status(stream) returns KV_ERR_DEVICE_BOUNDS with flag 8, and
 * the context stays usable.  KV_ERR_INVALID for a limit outside the range
 * (nothing launched). */
PAGEDKV_API kv_status kv_selftest_bounded_wait(uint32_t limit_us, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
