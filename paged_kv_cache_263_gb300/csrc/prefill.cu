// prefill.cu -- paged attention over a mixed batch of chunked-prefill query
// chunks and decode queries (sm_103a, 5th-generation tensor cores).
//
// A sequence with n >= 2 query rows is a prefill chunk: its rows sit at
// positions L-n .. L-1 and row i attends keys 0 .. L-n+i (causal inside the
// chunk, all earlier context visible) -- "PagedAttention, chunked prefill,
// and the launch that cascades", section "Serving systems" (long prompts split
// into ~1K-token chunks interleaved with decode); "M.65 Inference serving",
// prefill vs decode (a) prefill is a dense O(N^2) contraction, (e) chunked
// prefill.  Rows with n = 1 are decode rows and go to the decode kernel.
//
// Tensor-core kernel (bf16 cache), one CTA per (pair of 128-row query tiles,
// KV head, KV partition):
//  * A query tile packs 128/G chunk tokens x the G query heads of one KV head
//    (row = token * G + head), so every K/V tile is shared by the whole GQA
//    group; the two tiles of a pair share every K/V tile as well.  Both Q tiles
//    land in shared memory with one 3-D TMA load each.
//  * K/V tiles of 64 keys = 4 physical blocks, gathered through the block
//    table by TMA loads (128-byte swizzle) into a 5-stage ring (warp 8): K as
//    two 2-D boxes per block (each 64-dim half of the tile's keys contiguous, as
//    the QK^T operand needs), V as one 3-D box per block holding both halves.
//  * Chunks whose rows x heads fit one 128-row tile (speculative drafts) take a
//    second layout: one query tile per CTA, tiles of 128 keys (N = 128 QK^T
//    products, half the instructions per key for the single issuer), three
//    stages, and two producer warps (K and V).
//  * S[128x64] = Q K^T and O[128x128] += P V run as tcgen05.mma (K=16 steps),
//    one issuing warp per query tile (warps 9 and 10).  S is double-buffered
//    per tile in tensor memory, so QK^T of tile j+2 runs while the softmax
//    works on tile j; the softmax waits for the previous PV product only when
//    it must rescale O.  P (bf16) is written over its S buffer and read by the
//    second product as the A operand straight from tensor memory; K is the
//    K-major B operand of the first product, V the MN-major B operand of the
//    second, both from the same shared-memory stage.  Tensor memory: S 2 x 64
//    columns and O 128 columns per query tile, 512 in all.
//  * Two softmax warpgroups (warps 0-7), one per query tile, own one TMEM lane
//    (= one query row) per thread.  They read S with tcgen05.ld, apply the
//    causal mask on diagonal tiles, keep the online max / normaliser
//    ("FlashAttention" section: running max and normaliser per block) on
//    packed fp32 pairs, write P, and rescale O in tensor memory only when the
//    running max grew by more than 2^8 (otherwise the stale max is kept; exact
//    in the end).
//  * Keys at or past the context end inside the last tile are masked in S; the
//    producer zeroes their V rows after the load lands (0 x garbage could be
//    NaN), signalled on its own barrier.
//  * Long contexts are cut into equal partitions of whole tiles (at most
//    16,384 keys, less when the grid would be too small to fill the GPU),
//    merged by a fixed-order log-sum-exp kernel (no atomics).
//  * Decode rows (n = 1) of the batch run in the decode kernel, launched
//    programmatically right behind the chunk kernel on the caller's stream.  A
//    chunk CTA's shared memory leaves no room for a decode CTA beside it, so the
//    work-list kernel leaves a few SMs without a chunk CTA (a model of both
//    kernels' rates), and the decode CTAs stream their K/V there while the
//    chunk tiles compute on the others; once the chunk kernel is done they take
//    every SM.
//
// fp8 cache: the same kernel with four more warps that widen each e4m3 K/V tile
// (landed by TMA in a staging ring) to f16 operand tiles -- exact, as every
// e4m3 value is an f16 value -- zeroing keys past the context on the way; Q is
// rounded to f16 once in shared memory, so both products run as kind::f16 with
// f16 operands (one type per product); k_scale folds into the softmax scale and
// v_scale into O.  Quantising Q to e4m3 for a kind::f8f6f4 product would cost
// precision the bf16 queries carry.
#include "common.cuh"
#include "trace.h"

#include <algorithm>
#include <mutex>

namespace {

__device__ uint32_t g_status;

using namespace pkv;

constexpr int BM = 128, BN = 64;               // 128 query rows x 64 keys (4 blocks) per tile
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 8.0f;
// shared memory: Q 2 x 32 KiB | K/V operand stages of (K 16 KiB, V 16 KiB) | (fp8
// cache: e4m3 staging stages of (K 8 KiB, V 8 KiB)) | barriers.  P lives in
// tensor memory.
constexpr uint32_t SQ = 0, Q_TILE = 32768;
constexpr uint32_t F8_STAGE_BYTES = 16384, F8_V_OFF = 8192;
// bf16 cache: warps 0-3 softmax of query tile 0, 4-7 softmax of query tile 1, 8 TMA
// producer, 9 and 10 MMA issuers of query tile 0 and 1.  fp8 cache: in addition
// warps 11-14 widen each e4m3 K/V tile to f16 operand tiles (the products then
// run in kind::f16 with f16 operands: e4m3 -> f16 is exact, and Q is converted
// to f16 once in shared memory).
//
// BIG (bf16 cache, chunks whose rows x heads fit one 128-row tile, such as the
// drafts of speculative decoding): one query tile per CTA -- warps 0-3 softmax,
// 4 producer of K, 5 issuer, 6 producer of V -- and tiles of 128 keys.  With one query tile the
// tensor memory holds two S buffers of 128 columns next to O, so each QK^T
// product is N = 128: half the product instructions per key, which is what a
// CTA with a single issuer waits on.  Three stages of 64 KiB (192 KiB) are as
// many as fit beside the query tile.
constexpr int MAX_KV_STAGES = 5;   // room in the barrier table
template <bool FP8, bool BIG = false>
struct Lay {
    static constexpr int BNK = BIG ? 128 : 64;               // keys per KV tile
    static constexpr int NG = BIG ? 1 : 2;                   // query tiles per CTA
    static constexpr int W_PROD = 4 * NG;                    // the TMA producer warp
    static constexpr int W_MMA = W_PROD + 1;                 // the first MMA issuer warp
    static constexpr int W_WIDEN = W_MMA + NG;               // fp8 cache: the first widening warp
    // BIG: a second producer warp issues the V boxes; a CTA with one issuer is
    // bound by how fast its loads leave, and two warps issue them faster than one
    static constexpr int W_PROD2 = BIG ? W_WIDEN : -1;
    // BIG: a warp zeroes the V rows past the context in an item's last tile once
    // it has landed, so that the producer never waits for a load to land (short
    // items come one after another); the 64-key bf16 layout's producer does it
    // itself, between items that are long
    static constexpr int W_TAIL = BIG ? W_PROD2 + 1 : -1;
    static constexpr int THREADS = 32 * (W_WIDEN + (FP8 ? 4 : 0) + (BIG ? 2 : 0));
    // (bf16 two-tile layout: five stages, 224 KiB with Q; measured on GB300 the
    // fifth stage took 1.6-1.9 % off the long chunk's kernel time)
    static constexpr int KV_STAGES = BIG ? 3 : (FP8 ? 3 : 5);
    static constexpr uint32_t KV_HALF = BNK * 128;           // one 64-dim half of a K or V tile
    static constexpr uint32_t V_OFF = 2 * KV_HALF;
    static constexpr uint32_t KV_STAGE_BYTES = 4 * KV_HALF;  // K and V
    static constexpr int F8_STAGES = FP8 ? 3 : 0;
    static constexpr uint32_t SKV = NG * 32768;               // K/V stages follow the Q tiles
    static constexpr uint32_t SF8 = SKV + KV_STAGES * KV_STAGE_BYTES;
    static constexpr uint32_t SBAR = SF8 + F8_STAGES * F8_STAGE_BYTES;
    // barriers, the TMEM address, the abort flag and the work-item slots; + 1 KiB:
    // the dynamic shared memory is aligned to 1 KiB at run time
    static constexpr int SMEM_BYTES = SBAR + 1024 + 1024;
    static constexpr uint32_t S_COLS = 2 * BNK;               // two S buffers per query tile
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(NG * (S_COLS + 128) <= 512, "tensor memory");
    static_assert(!(FP8 && BIG), "the 128-key layout is for the bf16 cache");
    static_assert(KV_STAGES <= MAX_KV_STAGES && F8_STAGES <= 3, "barrier table");
};
// work items a CTA's producer may have fetched ahead of its slowest warp
constexpr int NSLOT = 4;
// barriers (room for the larger of the two layouts)
enum {
    B_KVF = 0,                      // + stage: K and V operand tiles ready
    B_KVE = B_KVF + MAX_KV_STAGES,              // + stage: every MMA reading the stage is done
    B_Q = B_KVE + MAX_KV_STAGES,                // the item's Q tiles landed
    B_QFREE = B_Q + 1,              // every QK^T product of the item finished (one per issuer)
    B_QC = B_QFREE + 1,             // + group: fp8 cache: the group's Q tile is in f16
    B_S = B_QC + 2,                 // + 2*group + buffer: an S tile of the group is in TMEM
    B_P = B_S + 4,                  // + 2*group + buffer: the group's P is in TMEM (128 arrivals)
    B_PVD = B_P + 4,                // + group: the group's latest PV product finished
    B_DRAIN = B_PVD + 2,            // + group: every MMA of the group's item finished
    B_TAIL = B_DRAIN + 2,           // + stage: bf16 cache: the V rows past the context are zeroed
    B_F8F = B_TAIL + MAX_KV_STAGES,             // + staging stage: fp8 cache: e4m3 K and V landed
    B_F8E = B_F8F + 3,              // + staging stage: fp8 cache: the stage was widened
    B_IFULL = B_F8E + 3,            // + slot: the producer wrote a work item into the slot
    B_IEMPTY = B_IFULL + NSLOT,     // + slot: every other warp has read it
    B_TGO = B_IEMPTY + NSLOT,       // + stage: bf16 cache: an item's last tile, past the context, landed
    NBAR = B_TGO + MAX_KV_STAGES
};
// a work item as the producer hands it to the other warps (valid = 0: no more)
struct ItemSlot {
    int s, row0, n, L, t0q, has1, j0, T, nsplit, g, split, valid, pad[4];
};
constexpr uint32_t SLOT_OFF = 512;   // within the barrier area
static_assert(NBAR * 8 + 8 <= SLOT_OFF && SLOT_OFF + NSLOT * sizeof(ItemSlot) <= 1024, "barrier area");

// instruction descriptors, kind::f16: fp32 accumulate, bf16 A and B, M=128
constexpr uint32_t idesc(int n, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(BM >> 4) << 24);
}
constexpr uint32_t IDESC_S = idesc(BN, false);    // S[128 x 64] = Q K^T, K K-major
constexpr uint32_t IDESC_S128 = idesc(128, false); // S[128 x 128] = Q K^T (128-key tiles)
constexpr uint32_t IDESC_PV = idesc(D, true);     // O[128 x 128] += P V, V MN-major
// the same with f16 A and B (fp8 cache widened to f16)
constexpr uint32_t F16_OPS = (1u << 7) | (1u << 10);
constexpr uint32_t IDESC_S16 = IDESC_S & ~F16_OPS;
constexpr uint32_t IDESC_PV16 = IDESC_PV & ~F16_OPS;

struct PrefillParams {
    float *out;
    const uint16_t *q;   // [rows][Hq][128] bf16
    const int32_t *cu_q_lens;
    const int32_t *context_lens;
    const int32_t *block_tables;
    int32_t *tile_off;   // [num_seqs + 1] pairs of query tiles per sequence, prefix sums
    int4 *order;         // work items, longest first: two int4 each (see tile_prefix_kernel)
    int32_t *row_info;   // [rows] key partitions of the row's query item (0: not a chunk row)
    int32_t *order_count;  // [0] items listed, [1] items taken so far (the CTAs' counter), [2] any cut,
                           // [3] CTAs that take items (the others leave their SMs to the decode rows)
    int items_cap;       // query items the order array has room for (x 1 KV head x 1 partition)
    float *part_o;       // [rows][Hq][max_splits][128]
    float *part_ml;      // [rows][Hq][max_splits][2]
    int max_blocks, num_seqs, hq, hkv, group, num_blocks, total_rows;
    int tiles_per_split, max_splits;   // the shortest partition length allowed; room for partitions
    int num_sms;
    float bytes_per_tile;              // HBM bytes the GPU moves in one KV tile's time
    int rows1;                         // the call runs decode rows (queries of 1); else a 1 is flagged
    int max_q_len;                     // the caller's bound on every query's rows (a longer one is flagged)
    int grid_ctas;                     // the chunk kernel's CTAs
    int q_box_bytes;                   // one 64-dim half of a query tile as loaded (rows x G x 128 B)
    int corun;           // the decode rows run beside the chunk kernel, on SMs it leaves free
    float decode_key_bytes;   // K and V bytes of one key of a decode row (all KV heads)
    float decode_sm_bytes;    // bytes the decode CTAs of one SM read in one KV tile's time
    int item_tiles;      // query tiles per CTA: 2 (a pair), or 1 (the 128-key layout)
    int tile_keys;       // keys per KV tile: 64, or 128 (the 128-key layout)
    float scale_log2;
    const float *k_scale;  // fp8 cache: [Hkv] (folded into the softmax scale)
    const float *v_scale;  // fp8 cache: [Hkv] (applied to O)
};

__device__ __forceinline__ void flag(uint32_t bits) { atomicOr(&g_status, bits); }

// One CTA's work: query item x (a pair of query tiles, or one tile in the
// 128-key layout) of some chunk sequence, and key partition `split` of the keys
// its rows see.  The keys are cut into nsplit partitions of (nearly) equal
// length, at most tiles_per_split KV tiles each.  False when the partition is
// empty.
struct Work {
    int s, item, row0, n, L, t0q, KT, nsplit, j0, T;
    bool has1;
};
// (toff, cu, cl: the query items' prefix sums, cu_q_lens and context_lens, in
// global or shared memory; s_hint: the item's sequence if known, else -1;
// tpt_log2, tk_log2: log2 of the query rows per tile and of the keys per tile)
__device__ __forceinline__ bool locate(const PrefillParams &p, const int32_t *toff, const int32_t *cu,
                                       const int32_t *cl, int x, int split, int item_tiles, int tpt_log2,
                                       int tk_log2, int tiles_per_split, Work &w, int s_hint = -1)
{
    int lo = s_hint;
    if (lo < 0) {
        lo = 0;
        int hi = p.num_seqs;                     // toff[lo] <= x < toff[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (toff[mid] <= x) lo = mid;
            else hi = mid;
        }
    }
    w.s = lo;
    w.item = x - toff[lo];
    w.row0 = cu[lo];
    w.n = cu[lo + 1] - w.row0;
    w.L = cl[lo];
    const int tpt = 1 << tpt_log2;
    const int tiles = (w.n + tpt - 1) >> tpt_log2;
    w.t0q = item_tiles * w.item;                  // the CTA's first query tile
    w.has1 = item_tiles == 2 && w.t0q + 1 < tiles;   // the pair's second query tile exists
    const int last = w.has1 ? w.t0q + 1 : w.t0q;
    const int kmax = w.L - w.n + min(w.n, (last + 1) * tpt);   // keys visible to the last row
    w.KT = (kmax + (1 << tk_log2) - 1) >> tk_log2;
    w.nsplit = (w.KT + tiles_per_split - 1) / tiles_per_split;
    const int tps = (w.KT + w.nsplit - 1) / w.nsplit;   // ceil(KT / tps) == nsplit
    w.j0 = split * tps;
    w.T = min(w.KT, w.j0 + tps) - w.j0;
    return w.j0 < w.KT;
}

// bounded wait for a warp that waits long and has nothing else to do: it
// sleeps between polls, leaving its scheduler's issue slots to the other warps
__device__ __forceinline__ bool wait_bar_lazy(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        __nanosleep(256);
        if (*abort_flag) return false;
        if (globaltimer() - t0 > WAIT_LIMIT_NS) {
            *abort_flag = 1;
            flag(ST_TIMEOUT);
            return false;
        }
    }
    return true;
}

// bounded wait that also gives up as soon as another role has aborted
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > WAIT_LIMIT_NS) {
                *abort_flag = 1;
                flag(ST_TIMEOUT);
                return false;
            }
        }
    }
}

// The chunk kernel's work list, one CTA of 128 to 1024 threads (sized by the
// host to the batch; every phase is written for any whole number of warps):
//  1. per sequence (a thread each): the chunk metadata validated, its query
//     items counted (then a block-wide scan), and its share of the partition
//     length estimates below;
//  2. the partition length; with decode rows in the batch, 2b. the number of
//     chunk CTAs that take items;
//  3. per query row, the number of key partitions its item is cut into (for
//     the merge kernel); the work items' bucket counts;
//  4. the work items in launch order.
// Sequence data is staged in shared memory when there are at most PREFIX_SMAX
// sequences, so that the searches cost no global-memory round trips.
//
// The partition length.  The host's plan (tiles_per_split) is the shortest
// allowed: the workspace holds that many partitions.  Here the real key ranges
// are known, and a longer length (fewer partitions) is taken where a makespan
// estimate favours it.  The CTAs take the items longest first, so the grid ends
// about max(longest item, S / m + shortest item / 2) after it starts (S: all
// items' tiles, m: SMs); each item adds a fixed cost, and a cut key range adds
// its partial results' write and merge (and the merge kernel's start).  The
// candidates are the host's length and uncut; every item of a sequence is taken
// to see as many keys as its last one.
constexpr int PREFIX_SMAX = 2048;
constexpr int PREFIX_XMAX = 8192;   // query items whose sequence is tabled in shared memory
constexpr float ITEM_TILES = 0.5f;   // a work item's Q load and epilogue, in tile-times
__global__ void __launch_bounds__(1024) tile_prefix_kernel(PrefillParams p)
{
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    __shared__ int32_t sh_toff[PREFIX_SMAX + 1], sh_cu[PREFIX_SMAX + 1], sh_cl[PREFIX_SMAX];
    __shared__ uint16_t sh_xs[PREFIX_XMAX];     // query item -> its sequence (num_seqs <= 65,535)
    // per candidate (0: the host's length, 1: uncut): items, longest and shortest
    // partition; the cut ranges' rows x partitions; all items' tiles (summed a
    // warp at a time: shared-memory atomics on one word serialise a warp)
    __shared__ unsigned int c_items[2];
    __shared__ int c_tmax[2], c_tmin[2];
    __shared__ float c_mrows, s_tiles, s_dkeys, s_merge;
    __shared__ int s_tps, s_nsmax, s_cut, s_ctas, s_tbest;
    constexpr int NBKT = 32;
    static_assert(NBKT == 32, "one warp scans the buckets");
    __shared__ int32_t cnt[32][NBKT];
    __shared__ int32_t bstart[NBKT];
    // the chunk kernel (launched with programmatic serialisation) may set up its
    // CTAs meanwhile; it waits for this grid before it reads the work list
    griddep_launch_dependents();
    // (launched with programmatic serialisation itself when the caller's stream
    // ran a kernel just before: nothing is read or written before this)
    griddep_wait();
    const bool staged = p.num_seqs <= PREFIX_SMAX;
    const int tpt = BM / p.group, tk = p.tile_keys, tps0 = max(1, p.tiles_per_split);
    const int tpt_log2 = __ffs(tpt) - 1, tk_log2 = __ffs(tk) - 1;   // both powers of two
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (threadIdx.x < 2) {
        c_items[threadIdx.x] = 0u;
        c_tmax[threadIdx.x] = 0;
        c_tmin[threadIdx.x] = INT_MAX;
    }
    for (int i = threadIdx.x; i < 32 * NBKT; i += blockDim.x) cnt[i / NBKT][i % NBKT] = 0;
    if (threadIdx.x == 0) {
        carry = 0;
        s_tiles = 0.f;
        s_dkeys = 0.f;
        c_mrows = 0.f;
        sh_toff[0] = 0;
    }
    __syncthreads();

    // ---- 1. per sequence
    for (int base = 0; base < p.num_seqs; base += blockDim.x) {
        const int s = base + threadIdx.x;
        int tiles = 0, n = 0, L = 0;
        if (s < p.num_seqs) {
            const int a = p.cu_q_lens[s], b = p.cu_q_lens[s + 1];
            n = b - a;
            L = p.context_lens[s];
            if (n >= 2) {
                if (a < 0 || b > p.total_rows || L < n || L > p.max_blocks * BS || n > p.max_q_len) flag(ST_BAD_LEN);
                else tiles = ((n + tpt - 1) / tpt + p.item_tiles - 1) / p.item_tiles;   // query items
            } else if (n < 0 || (n == 1 && !p.rows1)) {
                flag(ST_BAD_LEN);
            }
            if (staged) {
                sh_cu[s] = a;
                sh_cl[s] = L;
                if (s == p.num_seqs - 1) sh_cu[s + 1] = b;
            }
        }
        {
            // this sequence's share of the estimates (zeros for no chunk), summed
            // over the warp, then one shared-memory update per warp
            unsigned it0 = 0u, it1 = 0u;
            int mx0 = 0, mn0 = INT_MAX, mx1 = 0, mn1 = INT_MAX;
            float tl = 0.f, mr = 0.f;
            // a decode row's keys (read by the decode kernel beside this one)
            float dk = (n == 1 && L > 0) ? (float)min(L, p.max_blocks * BS) : 0.f;
            if (tiles > 0) {
                const int KT = (L + tk - 1) / tk;
                // the items' tiles: item x sees L - n + min(n, (x + 1) r) keys, r rows per item
                const float r = (float)(tpt * p.item_tiles);
                tl = (tiles * (float)(L - n) + r * 0.5f * (tiles - 1) * tiles + n) / tk;
                const int ns = (KT + tps0 - 1) / tps0, len = (KT + ns - 1) / ns;
                it0 = (unsigned)(tiles * ns);
                mx0 = len;
                mn0 = KT - (ns - 1) * len;
                if (ns > 1) mr = (float)n * ns;
                it1 = (unsigned)tiles;
                mx1 = mn1 = KT;
            }
            if (p.corun && __any_sync(0xffffffffu, dk > 0.f)) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dk += __shfl_xor_sync(0xffffffffu, dk, o);
                if (lane == 0) atomicAdd(&s_dkeys, dk);
            }
            if (__any_sync(0xffffffffu, tiles > 0)) {
                it0 = __reduce_add_sync(0xffffffffu, it0);
                it1 = __reduce_add_sync(0xffffffffu, it1);
                mx0 = __reduce_max_sync(0xffffffffu, mx0);
                mx1 = __reduce_max_sync(0xffffffffu, mx1);
                mn0 = __reduce_min_sync(0xffffffffu, mn0);
                mn1 = __reduce_min_sync(0xffffffffu, mn1);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    tl += __shfl_xor_sync(0xffffffffu, tl, o);
                    mr += __shfl_xor_sync(0xffffffffu, mr, o);
                }
                if (lane == 0) {
                    atomicAdd(&c_items[0], it0);
                    atomicAdd(&c_items[1], it1);
                    atomicMax(&c_tmax[0], mx0);
                    atomicMax(&c_tmax[1], mx1);
                    atomicMin(&c_tmin[0], mn0);
                    atomicMin(&c_tmin[1], mn1);
                    atomicAdd(&s_tiles, tl);
                    atomicAdd(&c_mrows, mr);
                }
            }
        }
        // block-wide inclusive scan of the item counts
        int v = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        if (lane == 31) warp_sums[w] = v;
        __syncthreads();
        if (w == 0) {
            int x = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int t = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += t;
            }
            warp_sums[lane] = x;
        }
        __syncthreads();
        const int incl = v + (w > 0 ? warp_sums[w - 1] : 0) + carry;
        if (s < p.num_seqs) {
            p.tile_off[s + 1] = incl;
            if (staged) sh_toff[s + 1] = incl;
            for (int x = incl - tiles; x < min(incl, PREFIX_XMAX); ++x) sh_xs[x] = (uint16_t)s;
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = incl;
        __syncthreads();
    }

    // ---- 2. the partition length
    if (threadIdx.x == 0) {
        p.tile_off[0] = 0;
        const float m = (float)p.num_sms, S = s_tiles * p.hkv;
        // a partial result (130 floats per head) is written and read once
        const float per_row_split = (float)p.hq * 130.f * 4.f * 2.f / p.bytes_per_tile;
        const float merge_start = 3.f * 64.f / tk;   // the merge kernel's start, in tile-times
        auto est = [&](int k, float merge) {
            return fmaxf((float)c_tmax[k], S / m + 0.5f * (float)c_tmin[k]) +
                   (float)c_items[k] * p.hkv * ITEM_TILES / m + merge;
        };
        const bool cut0 = c_mrows > 0.f;
        int pick = tps0, cut = cut0 ? 1 : 0;
        // (uncut only while an item's tiles fit the entry's 16-bit field)
        if (cut0 && c_tmax[1] < 65536 && est(1, 0.f) <= est(0, c_mrows * per_row_split + merge_start)) {
            pick = max(tps0, c_tmax[1]);             // uncut: every range in one partition
            cut = 0;
        }
        s_tps = pick;
        s_nsmax = (max(c_tmax[1], 1) + pick - 1) / pick;   // the most partitions of any item
        s_cut = cut;
        p.order_count[2] = cut;                      // the merge kernel has work
        s_merge = cut ? c_mrows * per_row_split + merge_start : 0.f;
        s_tbest = __float_as_int(INFINITY);
        s_ctas = p.corun && s_dkeys > 0.f ? 0 : p.grid_ctas;
    }
    __syncthreads();
    // ---- 2b. The decode rows run beside this kernel on the SMs that its CTAs
    // leave free (the decode kernel is launched right behind it, and a chunk CTA's
    // shared memory leaves no room for a decode CTA): c CTAs take items, the other
    // SMs read decode K/V at decode_sm_bytes per tile-time each, and what is left
    // when the chunk work ends is read by every SM at the HBM rate.  c is the
    // largest count whose modelled end of both is within 0.1 % of the least (one
    // candidate per thread).
    if (s_ctas == 0) {
        const int c_lo = max(1, p.grid_ctas / 2);
        const int ncand = min(p.grid_ctas - c_lo + 1, (int)blockDim.x);
        int c = 0;
        float t = INFINITY;
        if ((int)threadIdx.x < ncand) {
            c = p.grid_ctas - (int)threadIdx.x;
            const int k = s_cut ? 0 : 1;
            const float fc = (float)c, S = s_tiles * p.hkv;
            const float chunk = fmaxf((float)c_tmax[k], S / fc + 0.5f * (float)c_tmin[k]) +
                                (float)c_items[k] * p.hkv * ITEM_TILES / fc + s_merge;
            const float beside = fminf((float)(p.num_sms - c) * p.decode_sm_bytes, p.bytes_per_tile);
            t = chunk + fmaxf(0.f, s_dkeys * p.decode_key_bytes - chunk * beside) / p.bytes_per_tile;
        }
        float tm = t;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tm = fminf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
        if (lane == 0 && tm < INFINITY) atomicMin(&s_tbest, __float_as_int(tm));   // (t >= 0)
        __syncthreads();
        const int cm = __reduce_max_sync(0xffffffffu, t <= __int_as_float(s_tbest) * 1.001f ? c : 0);
        if (lane == 0 && cm > 0) atomicMax(&s_ctas, cm);
        __syncthreads();
    }
    if (threadIdx.x == 0) p.order_count[3] = s_ctas;
    const int tps = s_tps;
    const int32_t *toff = staged ? sh_toff : p.tile_off;
    const int32_t *cu = staged ? sh_cu : p.cu_q_lens;
    const int32_t *cl = staged ? sh_cl : p.context_lens;
    // query items over all chunks; more than the host's bound only with chunk
    // metadata that overlaps (flagged), and then the excess is left out
    const int X = min(carry, p.items_cap);
    if (threadIdx.x == 0 && carry > p.items_cap) flag(ST_BAD_LEN);

    // ---- 3. per query row: its item's partition count (0 for rows outside any
    // chunk; not needed when no key range is cut: the merge kernel then has no
    // work); and the work items' bucket counts
    for (int row = threadIdx.x; s_cut && row < p.total_rows; row += blockDim.x) {
        int lo = 0, hi = p.num_seqs;                 // cu[lo] <= row < cu[hi]
        int ns = 0;
        if (row < cu[p.num_seqs]) {
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (cu[mid] <= row) lo = mid;
                else hi = mid;
            }
            const int a = cu[lo], n = cu[lo + 1] - a, L = cl[lo];
            if (n >= 2 && n <= p.max_q_len && a >= 0 && row >= a && L >= n && L <= p.max_blocks * BS) {
                const int i = row - a, mt = i >> tpt_log2, tiles = (n + tpt - 1) >> tpt_log2;
                const int last = min(tiles - 1, (mt / p.item_tiles) * p.item_tiles + p.item_tiles - 1);
                const int KT = (L - n + min(n, (last + 1) * tpt) + tk - 1) >> tk_log2;
                ns = (KT + tps - 1) / tps;
            }
        }
        p.row_info[row] = ns;
    }
    // The work items in launch order, longest first: the CTAs take them one
    // after another, so a long item taken last would set the makespan (ragged
    // speculative drafts).  Longest-processing-time-first list order instead:
    // (query item, partition) pairs are bucketed by length relative to the
    // partition length (NBKT buckets) and sorted stably, so that within a bucket
    // they keep the order item fastest, then partition, under which concurrent
    // CTAs share their keys in L2; each pair then takes hkv consecutive places,
    // one per KV head.  Each warp takes a contiguous segment of the pairs; a
    // pair's rank is its bucket's start + the earlier warps' counts in that
    // bucket + its rank in its own warp's segment, so the order is
    // deterministic.  An entry (two int4) holds everything a CTA needs:
    //   s, row0, n, L | j0, T | nsplit << 16, KV head | partition << 16, t0q | has1 << 30
    // (the pair count x hkv is below 2^31: the host bounds the grid by it)
    const long long nslot = (long long)X * min(p.max_splits, s_nsmax);
    const long long seg = (nslot + nw - 1) / nw;
    const long long s0 = (long long)w * seg, s1 = min(nslot, s0 + seg);
    auto bucket_of = [&](long long e, int4 &e0, int4 &e1) -> int {
        const unsigned eu = (unsigned)e, split = eu / (unsigned)X;
        const int x = (int)(eu - split * (unsigned)X);
        Work wk;
        if (!locate(p, toff, cu, cl, x, (int)split, p.item_tiles, tpt_log2, tk_log2, tps, wk,
                    x < PREFIX_XMAX ? (int)sh_xs[x] : -1))
            return -1;
        e0 = make_int4(wk.s, wk.row0, wk.n, wk.L);
        e1 = make_int4(wk.j0, wk.T | (wk.nsplit << 16), (int)(split << 16), wk.t0q | (wk.has1 ? 1 << 30 : 0));
        return min(NBKT - 1, (max(0, tps - wk.T) * NBKT) / tps);   // (tps x 32 < 2^31)
    };
    // (a warp's first 32 slots -- all of them in small batches -- are kept in
    // registers for the second pass)
    int4 f_e0 = make_int4(0, 0, 0, 0), f_e1 = f_e0;
    int f_bk = -1;
    for (long long b0 = s0; b0 < s1; b0 += 32) {
        int4 e0, e1;
        const int bk = b0 + lane < s1 ? bucket_of(b0 + lane, e0, e1) : -1;
        if (b0 == s0) {
            f_e0 = e0;
            f_e1 = e1;
            f_bk = bk;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, bk);
        if (bk >= 0 && lane == __ffs(peers) - 1) cnt[w][bk] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    if (w == 0) {
        // per bucket (a lane each): the earlier warps' counts, then the buckets' starts
        int run = 0;
        for (int i = 0; i < nw; ++i) {
            const int t = cnt[i][lane];
            cnt[i][lane] = run;
            run += t;
        }
        int v = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        bstart[lane] = v - run;
        if (lane == 31) {
            p.order_count[0] = v * p.hkv;
            // the persistent CTAs' fetch counter: CTA c takes item c first, the
            // rest through the counter
            p.order_count[1] = s_ctas;
        }
    }
    __syncthreads();
    // ---- 4. the entries
    for (long long b0 = s0; b0 < s1; b0 += 32) {
        int4 e0 = f_e0, e1 = f_e1;
        const int bk = b0 == s0 ? f_bk : (b0 + lane < s1 ? bucket_of(b0 + lane, e0, e1) : -1);
        const unsigned peers = __match_any_sync(0xffffffffu, bk);
        if (bk >= 0) {
            const int pos = (bstart[bk] + cnt[w][bk] + __popc(peers & ((1u << lane) - 1u))) * p.hkv;
            for (int g = 0; g < p.hkv; ++g) {
                p.order[2 * (size_t)(pos + g)] = e0;
                p.order[2 * (size_t)(pos + g) + 1] = make_int4(e1.x, e1.y, e1.z | g, e1.w);
            }
        }
        __syncwarp();
        if (bk >= 0 && lane == __ffs(peers) - 1) cnt[w][bk] += __popc(peers);
        __syncwarp();
    }
}

// (the fp8 variant declares 512 threads so that registers stay <= 128, which 15
// warps need on an SM partition holding four of them)
//
// Persistent: the grid holds one CTA per SM, and each CTA takes work items
// (query item, KV head, partition) from the longest-first list that
// tile_prefix_kernel wrote, one after another (CTA c takes item c first, then
// the next free one through an atomic counter), until the list is used up.  The producer warp fetches an item and hands it to the
// other warps through a ring of NSLOT shared-memory slots; the K/V stage ring,
// the S buffers and every barrier phase run on across items, so the next item's
// Q and first K/V tiles load, and its first QK^T products run, while the
// softmax warps still finish the item before.
template <bool FP8, bool BIG>
__global__ void __launch_bounds__(FP8 ? 512 : Lay<FP8, BIG>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p)
{
    using LY = Lay<FP8, BIG>;
    constexpr int KV_STAGES = LY::KV_STAGES, F8_STAGES = LY::F8_STAGES;
    constexpr int BN = LY::BNK;                                   // keys per KV tile
    constexpr uint32_t SKV = LY::SKV, KV_STAGE_BYTES = LY::KV_STAGE_BYTES, V_OFF = LY::V_OFF,
                       KV_HALF = LY::KV_HALF;
    constexpr int NWARPS = LY::THREADS / 32;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + LY::SBAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile ItemSlot *slots = reinterpret_cast<volatile ItemSlot *>(smem + LY::SBAR + SLOT_OFF);
    auto bar = [&](int i) -> uint32_t { return smem_u32(bars + i); };
    // warp-uniform wait: every role below runs warp-collective instructions
    // (ballots, tcgen05.ld/st), so a warp leaves a loop only as a whole
    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait_bar(b, parity, abort_flag));
    };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group, tpt = BM / G;
    griddep_launch_dependents();   // the merge kernel may be scheduled; it waits for this grid
    if (sbase & 1023u) {
        // the 128-byte swizzle needs 1024-byte aligned tiles; never observed, but
        // refuse rather than compute with a wrong layout
        if (threadIdx.x == 0) flag(ST_TIMEOUT);
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < KV_STAGES; ++i) {
            mbar_init(bar(B_KVF + i), FP8 ? 128 : 1);   // fp8: the widening warps arrive
            mbar_init(bar(B_KVE + i), LY::NG);          // one release per MMA issuer
            mbar_init(bar(B_TAIL + i), 1);
            mbar_init(bar(B_TGO + i), 1);
        }
        for (int i = 0; i < F8_STAGES; ++i) {
            mbar_init(bar(B_F8F + i), 1);
            mbar_init(bar(B_F8E + i), 128);
        }
        mbar_init(bar(B_Q), 1);
        mbar_init(bar(B_QFREE), LY::NG);
        for (int i = 0; i < 2; ++i) mbar_init(bar(B_QC + i), 128);
        for (int i = 0; i < 4; ++i) {
            mbar_init(bar(B_S + i), 1);
            mbar_init(bar(B_P + i), 128);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_PVD + i), 1);
            mbar_init(bar(B_DRAIN + i), 1);
        }
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(bar(B_IFULL + i), 1);
            mbar_init(bar(B_IEMPTY + i), NWARPS - 1);   // every warp but the producer
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM columns per query tile gi: two S buffers of BN fp32 columns at
    // S_COLS gi + BN b (P overwrites the first BN/2 of a buffer with 16-bit pairs
    // once its S has been read), O after all S buffers, 128 columns per tile
    auto tS = [&](int gi, int b) -> uint32_t { return tmem + gi * LY::S_COLS + b * BN; };
    auto tO = [&](int gi) -> uint32_t { return tmem + LY::NG * LY::S_COLS + gi * D; };
    // the k-th work item of this CTA, as every warp but the producer reads it
    // (false: the list is used up, or the CTA gave up)
    auto read_item = [&](int k, ItemSlot &it) -> bool {
        const int sl = k % NSLOT;
        if (!wait_w(bar(B_IFULL + sl), (k / NSLOT) & 1)) return false;
        it.s = slots[sl].s;
        it.row0 = slots[sl].row0;
        it.n = slots[sl].n;
        it.L = slots[sl].L;
        it.t0q = slots[sl].t0q;
        it.has1 = slots[sl].has1;
        it.j0 = slots[sl].j0;
        it.T = slots[sl].T;
        it.nsplit = slots[sl].nsplit;
        it.g = slots[sl].g;
        it.split = slots[sl].split;
        it.valid = slots[sl].valid;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_IEMPTY + sl));
        return it.valid != 0;
    };
    // a tile whose keys run past the context (only ever an item's last tile):
    // its V rows there are zeroed before PV reads them (bf16 cache)
    auto has_tail = [&](const ItemSlot &it) -> bool { return (it.j0 + it.T) * BN > it.L; };
    // zeroes V rows first .. BN-1 of the landed tile in stage st (one warp), then
    // releases its PV products (B_TAIL)
    auto zero_tail = [&](int st, int first) {
        const uint32_t vb = sbase + SKV + st * KV_STAGE_BYTES + V_OFF;
        for (int c = lane; c < (BN - first) * 16; c += 32) {
            const int r = first + (c >> 4), h = (c >> 3) & 1, ch = c & 7;
            st_shared_v4(vb + (r >> 4) * 4096 + h * 2048 + (r & 15) * 128 + ch * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_TAIL + st));
    };

    if (warp == LY::W_PROD || warp == LY::W_PROD2) {
        // ======================= TMA producer.  Role 0 fetches the work items,
        // loads Q and the K boxes and arms each stage's barrier; role 1 (the
        // 128-key layout) issues the V boxes.
        const int role = warp == LY::W_PROD ? 0 : 1;
        // bf16 cache: one lane per box, so a tile's loads leave in one instruction.
        // K: two 2 KiB boxes per block (dims 0-63 and 64-127; the QK^T operand needs
        // each half of all the tile's keys contiguous), lanes 0 .. 2 NB - 1, lane =
        // 2 x block + half.  V: one 4 KiB box per block holding both halves (a 3-D
        // tensor map), lanes 2 NB .. 3 NB - 1.  NB = blocks per tile (4 or 8).  Each
        // lane's block id for the next tile is read while the producer waits for
        // the stage to free up.
        constexpr int NB = BN / BS, K_LANES = 2 * NB;
        const int BOX_LANES = BIG ? (role == 0 ? K_LANES : NB) : 3 * NB;
        const bool is_v = BIG ? role == 1 : lane >= K_LANES;
        const int blk = BIG ? (role == 1 ? lane & (NB - 1) : (lane >> 1) & (NB - 1))
                            : (is_v ? (lane - K_LANES) & (NB - 1) : (lane >> 1) & (NB - 1));
        const int opnd = lane & 1;
        // fp8 cache: lanes 0-7 each load one 2 KiB box per tile: lane = 2 x block + (K | V)
        const int blk8 = (lane >> 1) & 3, kv = lane & 1;
        int u = 0;          // K/V tiles issued so far: the position in the stage rings
        int kq = 0;         // items whose Q tiles were loaded
        bool failed = false;
        // the work list (and everything before it on the stream) is complete;
        // the other warps learn of each item through the slots, after this wait
        griddep_wait();
        for (int k = 0; !failed; ++k) {
            ItemSlot it;
            if (role == 0) {
                const int sl = k % NSLOT;
                if (k >= NSLOT && !wait_w(bar(B_IEMPTY + sl), (k / NSLOT - 1) & 1)) break;
                // the next listed item (tile_prefix_kernel wrote all its fields);
                // every listed partition is non-empty, but a CTA never trusts that
                // to keep its pipelines in step
                it.valid = 0;
                // CTAs past the work list's count leave their SMs to the decode rows
                const bool idle = k == 0 && (int)blockIdx.x >= p.order_count[3];
                for (int tries = 0; !idle; ++tries) {
                    int idx = (int)blockIdx.x;           // the first item: no round trip
                    if (k > 0 || tries > 0) {
                        if (lane == 0) idx = atomicAdd(p.order_count + 1, 1);
                        idx = __shfl_sync(0xffffffffu, idx, 0);
                    }
                    if (idx >= p.order_count[0]) break;
                    const int4 e0 = p.order[2 * (size_t)idx], e1 = p.order[2 * (size_t)idx + 1];
                    it.s = e0.x;
                    it.row0 = e0.y;
                    it.n = e0.z;
                    it.L = e0.w;
                    it.j0 = e1.x;
                    it.T = e1.y & 0xffff;
                    it.nsplit = (int)((unsigned)e1.y >> 16);
                    it.g = e1.z & 0xffff;
                    it.split = (int)((unsigned)e1.z >> 16);
                    it.t0q = e1.w & ((1 << 30) - 1);
                    it.has1 = (e1.w >> 30) & 1;
                    if (it.T > 0) {
                        it.valid = 1;
                        break;
                    }
                }
                if (lane == 0) {
                    slots[sl].s = it.s;
                    slots[sl].row0 = it.row0;
                    slots[sl].n = it.n;
                    slots[sl].L = it.L;
                    slots[sl].t0q = it.t0q;
                    slots[sl].has1 = it.has1;
                    slots[sl].j0 = it.j0;
                    slots[sl].T = it.T;
                    slots[sl].nsplit = it.nsplit;
                    slots[sl].g = it.g;
                    slots[sl].split = it.split;
                    slots[sl].valid = it.valid;
                    mbar_arrive(bar(B_IFULL + sl));
                }
                __syncwarp();
                if (!it.valid) break;
                // Q of the item, once every QK^T product of the item before finished
                if (kq > 0 && !wait_w(bar(B_QFREE), (kq - 1) & 1)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(B_Q), (it.has1 ? 4 : 2) * p.q_box_bytes);
                    for (int gi = 0; gi < (it.has1 ? 2 : 1); ++gi) {
                        const int zq = it.row0 + (it.t0q + gi) * tpt;
                        tma_load_3d(sbase + SQ + gi * Q_TILE, &qmap, 0, it.g * G, zq, bar(B_Q));
                        tma_load_3d(sbase + SQ + gi * Q_TILE + 16384, &qmap, 64, it.g * G, zq, bar(B_Q));
                    }
                }
                ++kq;
            } else if (!read_item(k, it)) {
                break;
            }
            const int32_t *bt = p.block_tables + (size_t)it.s * p.max_blocks;
            const int nblk = (it.L + BS - 1) / BS;
            const int j0 = it.j0, T = it.T;
            if constexpr (FP8) {
                // e4m3 K and V of each block (one 2 KiB box each) into a staging stage;
                // the widening warps turn it into the operand tiles.  The block ids of
                // the next tile are read during the wait for a free stage.
                auto block_id8 = [&](int jj) -> int32_t {
                    const int b = (j0 + jj) * (BN / BS) + blk8;
                    return (lane < 8 && jj < T && b < nblk) ? __ldg(bt + b) : -1;
                };
                int32_t next_id = block_id8(0);
                for (int jj = 0; jj < T; ++jj, ++u) {
                    const int st = u % F8_STAGES;
                    const int32_t id = next_id;
                    next_id = block_id8(jj + 1);
                    if (u >= F8_STAGES && !wait_w(bar(B_F8E + st), ((u - F8_STAGES) / F8_STAGES) & 1)) {
                        failed = true;
                        break;
                    }
                    const int j = j0 + jj;
                    const bool in = lane < 8 && j * (BN / BS) + blk8 < nblk;
                    const bool valid = in && id >= 0 && id < p.num_blocks;
                    if (in && !valid && kv == 0) flag(ST_BAD_BLOCK);
                    const unsigned vm = __ballot_sync(0xffffffffu, valid);
                    if (lane == 0) {
                        fence_proxy_async_smem();
                        mbar_arrive_expect_tx(bar(B_F8F + st), __popc(vm) * 2048);
                    }
                    __syncwarp();
                    if (valid) {
                        const int y = (id * p.hkv + it.g) * BS;
                        const uint32_t dst = sbase + LY::SF8 + st * F8_STAGE_BYTES + kv * F8_V_OFF + blk8 * 2048;
                        tma_load_2d(dst, kv ? &vmap : &kmap, 0, y, bar(B_F8F + st));
                    }
                }
            } else {
                auto block_id = [&](int jj) -> int32_t {
                    const int b = (j0 + jj) * (BN / BS) + blk;
                    return (lane < BOX_LANES && jj < T && b < nblk) ? __ldg(bt + b) : -1;
                };
                int32_t next_id = block_id(0);
                for (int jj = 0; jj < T; ++jj, ++u) {
                    const int st = u % KV_STAGES;
                    const int32_t id = next_id;
                    next_id = block_id(jj + 1);
                    if (u >= KV_STAGES && !wait_w(bar(B_KVE + st), ((u - KV_STAGES) / KV_STAGES) & 1)) {
                        failed = true;
                        break;
                    }
                    const int j = j0 + jj;
                    const bool in = lane < BOX_LANES && j * (BN / BS) + blk < nblk;
                    const bool valid = in && id >= 0 && id < p.num_blocks;
                    if (in && !valid && is_v) flag(ST_BAD_BLOCK);
                    const unsigned vm = __ballot_sync(0xffffffffu, valid);
                    if (lane == 0 && role == 0) {
                        fence_proxy_async_smem();
                        constexpr unsigned K_MASK = (1u << K_LANES) - 1u;
                        // BIG: the V warp loads one 4 KiB box per valid block (2 K lanes each)
                        const unsigned vbytes =
                            BIG ? __popc(vm & K_MASK & 0x55555555u) * 4096 : __popc(vm & ~K_MASK) * 4096;
                        mbar_arrive_expect_tx(bar(B_KVF + st), __popc(vm & K_MASK) * 2048 + vbytes);
                    }
                    __syncwarp();
                    if (valid) {
                        const int y = (id * p.hkv + it.g) * BS;
                        const uint32_t stg = sbase + SKV + st * KV_STAGE_BYTES;
                        if (is_v) tma_load_3d(stg + V_OFF + blk * 4096, &vmap, 0, y, 0, bar(B_KVF + st));
                        else tma_load_2d(stg + opnd * KV_HALF + blk * 2048, &kmap, opnd * 64, y, bar(B_KVF + st));
                    }
                    const int first = it.L - j * BN;         // first row of the tile at or past L
                    if (!BIG && first < BN) {
                        // the 64-key layout: this warp zeroes the V rows past the context
                        // (see the tail warp) once the tile has landed
                        if (!wait_w(bar(B_KVF + st), (u / KV_STAGES) & 1)) {
                            failed = true;
                            ++u;
                            break;
                        }
                        zero_tail(st, first);
                    }
                }
            }
        }
        if (*abort_flag) {
            // let loads already in flight land before the CTA exits
            constexpr int RING = FP8 ? F8_STAGES : KV_STAGES;
            for (int uu = max(0, u - RING); uu < u; ++uu)
                (void)mbar_wait_bounded(bar((FP8 ? B_F8F : B_KVF) + uu % RING), (uu / RING) & 1);
            if (role == 0 && kq > 0) (void)mbar_wait_bounded(bar(B_Q), (kq - 1) & 1);
        }
    } else if (warp >= LY::W_MMA && warp < LY::W_MMA + LY::NG) {
        // ======================= MMA issuers: one warp per query tile
        const int gi = warp - LY::W_MMA;
        // shared-memory descriptors of stage 0; other stages and K steps are
        // constant byte offsets added to the start-address field (in 16-byte
        // units; shared memory is < 256 KiB, so the 14-bit field never carries)
        const uint64_t qdesc = sdesc_sw128(sbase + SQ + gi * Q_TILE, 16, 1024);
        const uint64_t kdesc0 = sdesc_sw128(sbase + SKV, 16, 1024);
        // V: bf16 cache [block][64-dim half][16 keys] (one 3-D box per block); fp8
        // cache [half][block][16 keys] (written by the widening warps)
        constexpr uint32_t V_LBO = FP8 ? KV_HALF : 2048, V_KSTEP = FP8 ? 2048 : 4096;
        const uint64_t vdesc0 = sdesc_sw128(sbase + SKV + V_OFF, V_LBO, 1024);
        const uint32_t to = tO(gi);
        // running positions, carried across items: the stage and phase parity of
        // the next K/V tile; the S buffer and its phase parity of this group's next
        // tile; items the group computed (drain and fp8 Q phases)
        int stg = 0;
        uint32_t kph = 0;
        int sbuf = 0;
        uint32_t sph = 0;
        int kg = 0;
        unsigned tailpar = 0;   // phase parity of each stage's tail barrier
        auto adv = [](int &st, uint32_t &ph) {
            if (++st == KV_STAGES) {
                st = 0;
                ph ^= 1u;
            }
        };
        bool ok = true;
        for (int k = 0; ok; ++k) {
            ItemSlot it;
            if (!read_item(k, it)) break;
            const int T = it.T;
            const int st0 = stg;
            const uint32_t ph0 = kph;
            {   // the ring position after the item's tiles
                const int tot = stg + T;
                stg = tot % KV_STAGES;
                kph ^= (uint32_t)(tot / KV_STAGES) & 1u;
            }
            // the tail tile (if any) is the item's last; both issuers follow its parity
            const int tail_st = (st0 + T - 1) % KV_STAGES;
            const bool tail = !FP8 && has_tail(it);
            if (gi == 1 && !it.has1) {                 // no second query tile in this item
                if (tail) tailpar ^= 1u << tail_st;
                continue;
            }
            // the partner issuer's releases, when the item has no second query tile
            const bool rel2 = LY::NG == 2 && !it.has1;
            // S = Q K^T for the tile in stage st into S buffer b: A = Q, B = K (K-major)
            auto issue_s = [&](int st, int b, bool last) {
                if (lane == 0) {
                    tc_fence_after();
                    const uint64_t kd = kdesc0 + (uint64_t)((st * KV_STAGE_BYTES) >> 4);
                    const uint32_t ts = tS(gi, b);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)   // D = 128 in steps of 16: 4 per 64-wide half
                        umma_f16(ts, qdesc + (uint64_t)((((kk >> 2) * 16384) + (kk & 3) * 32) >> 4),
                                 kd + (uint64_t)((((kk >> 2) * KV_HALF) + (kk & 3) * 32) >> 4),
                                 FP8 ? IDESC_S16 : (BIG ? IDESC_S128 : IDESC_S), kk > 0);
                    umma_commit(bar(B_S + 2 * gi + b));
                    if (last) {
                        // the item's last QK^T product: its Q tiles may be replaced once done
                        umma_commit(bar(B_QFREE));
                        if (rel2) umma_commit(bar(B_QFREE));
                    }
                }
                __syncwarp();
            };
            // O += P V for the tile in stage st: A = P from TMEM (S buffer b), B = V
            // (MN-major) from smem
            auto issue_pv = [&](int st, int b, bool first) {
                if (lane == 0) {
                    tc_fence_after();
                    const uint64_t vd = vdesc0 + (uint64_t)((st * KV_STAGE_BYTES) >> 4);
                    const uint32_t ts = tS(gi, b);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)   // the tile's keys in steps of 16
                        umma_f16_ts(to, ts + kk * 8, vd + (uint64_t)((kk * V_KSTEP) >> 4), FP8 ? IDESC_PV16 : IDESC_PV,
                                    (first && kk == 0) ? 0u : 1u);
                    umma_commit(bar(B_PVD + gi));
                    // the stage is released once both issuers' MMAs reading it are done
                    umma_commit(bar(B_KVE + st));
                    if (rel2) umma_commit(bar(B_KVE + st));
                }
                __syncwarp();
            };
            // S of the first two tiles up front; afterwards S(jj+2) follows PV(jj), so
            // each softmax finds its S computed while it worked on the tile before.
            // PV(jj-2) of the item before (or of this one) read the S buffer that
            // S(jj) overwrites; this thread issued it first, and P(jj-2) had arrived.
            // fp8 cache: Q is used once the softmax warps have turned it into f16
            ok = FP8 ? wait_w(bar(B_QC + gi), kg & 1) : wait_w(bar(B_Q), k & 1);
            int sx = st0;                              // the next tile to compute S for
            uint32_t px = ph0;                         // its KVF phase parity
            // the tail tile has landed: the tail warp may zero its rows past L (it
            // waits for this in item order, so its barrier phases cannot alias)
            auto tail_go = [&]() {
                if (BIG && tail && gi == 0 && lane == 0) mbar_arrive(bar(B_TGO + tail_st));
            };
            for (int jj = 0; ok && jj < min(2, T); ++jj) {
                if (!wait_w(bar(B_KVF + sx), px)) { ok = false; break; }
                if (jj == T - 1) tail_go();
                issue_s(sx, sbuf ^ jj, jj == T - 1);
                adv(sx, px);
            }
            int spv = st0;                             // the PV tile's stage
            for (int jj = 0; jj < T && ok; ++jj) {
                if (!wait_w(bar(B_P + 2 * gi + sbuf), sph)) { ok = false; break; }
                // a tile holding keys >= L is read by PV only after the producer zeroed
                // them (fp8 cache: the widening warps write those rows as zeros)
                if (tail && jj == T - 1) {
                    if (!wait_w(bar(B_TAIL + tail_st), (tailpar >> tail_st) & 1)) { ok = false; break; }
                    tailpar ^= 1u << tail_st;
                }
                // in issue order: PV(jj) reads P from its S buffer before S(jj+2)
                // overwrites it
                issue_pv(spv, sbuf, jj == 0);
                if (jj + 2 < T) {
                    if (!wait_w(bar(B_KVF + sx), px)) { ok = false; break; }
                    if (jj + 2 == T - 1) tail_go();
                    issue_s(sx, sbuf, jj + 2 == T - 1);
                    adv(sx, px);
                }
                if (++spv == KV_STAGES) spv = 0;
                sbuf ^= 1;
                if (sbuf == 0) sph ^= 1u;
            }
            // the item's every MMA finished: the softmax warps may read O
            if (lane == 0) umma_commit(bar(B_DRAIN + gi));
            __syncwarp();
            ++kg;
        }
        // every MMA this issuer started has finished before TMEM is released: its
        // last item's drain phase (a further commit could complete together with
        // that phase while the softmax warps still wait on it, and the two phases
        // would alias their parity)
        if (kg > 0) (void)mbar_wait_bounded(bar(B_DRAIN + gi), (kg - 1) & 1);
    } else if (warp == LY::W_TAIL) {
        // ======================= bf16 cache: an item's last tile may hold keys past
        // the context; their V rows may hold anything (never written, or not
        // loaded), and P is 0 there but 0 * NaN is NaN, so they are zeroed once the
        // tile has landed, before its PV product (which waits for B_TAIL) reads it
        // (the first issuer signals B_TGO once the tile has landed: this warp must
        // not wait on the stage's own barrier, which it could reach two phases early)
        int stg = 0;        // the ring position of the next item's first tile
        unsigned tgpar = 0; // phase parity of each stage's B_TGO
        for (int k = 0;; ++k) {
            ItemSlot it;
            if (!read_item(k, it)) break;
            const int T = it.T;
            const int st = (stg + T - 1) % KV_STAGES;  // the item's last tile
            stg = (stg + T) % KV_STAGES;
            if (!has_tail(it)) continue;
            if (!__all_sync(0xffffffffu, wait_bar_lazy(bar(B_TGO + st), (tgpar >> st) & 1, abort_flag))) break;
            tgpar ^= 1u << st;
            zero_tail(st, it.L - (it.j0 + T - 1) * BN);
        }
    } else if (warp >= LY::W_WIDEN) {
        // ======================= fp8 cache: widen each e4m3 K/V tile to f16 operand
        // tiles (exact), in the operand stages' 128-byte-swizzled layout; keys at
        // or past L and blocks outside the pool become zeros
        if constexpr (FP8) {
            // thread ct owns key row ct % 64 of every tile and the chunks of 16 e4m3
            // (d = 16c .. 16c+15) with c = ct / 64 + 2k, k = 0..3, of both K and V; the
            // lanes of a warp take consecutive keys, so the 8 lanes of each
            // quarter-warp access 8 distinct 16-byte bank groups (the 128-byte
            // swizzle XORs the chunk with the key's low 3 bits)
            const int ct = threadIdx.x - LY::W_WIDEN * 32;      // 0..127
            const int row = ct & (BN - 1), c0 = ct >> 6;
            int u = 0;      // tiles of the CTA's items so far: the stage ring positions
            bool failed = false;
            for (int k = 0; !failed; ++k) {
                ItemSlot it;
                if (!read_item(k, it)) break;
                const int32_t *bt = p.block_tables + (size_t)it.s * p.max_blocks;
                const int j0 = it.j0, T = it.T, L = it.L;
                // the row's key of tile jj lies inside the context and its block in the
                // pool (read one tile ahead, during the waits)
                auto row_ok = [&](int jj) -> bool {
                    const int key = (j0 + jj) * BN + row;
                    if (jj >= T || key >= L) return false;
                    const int32_t id = __ldg(bt + key / BS);
                    return id >= 0 && id < p.num_blocks;
                };
                bool next_ok = row_ok(0);
                for (int jj = 0; jj < T; ++jj, ++u) {
                    const int s8 = u % F8_STAGES, st = u % KV_STAGES;
                    const bool valid = next_ok;
                    next_ok = row_ok(jj + 1);
                    if (!wait_w(bar(B_F8F + s8), (u / F8_STAGES) & 1) ||
                        (u >= KV_STAGES && !wait_w(bar(B_KVE + st), ((u - KV_STAGES) / KV_STAGES) & 1))) {
                        failed = true;
                        break;
                    }
                    const uint32_t src = sbase + LY::SF8 + s8 * F8_STAGE_BYTES + row * 128;
                    const uint32_t dst = sbase + SKV + st * KV_STAGE_BYTES + row * 128;
                    // all eight 16-byte loads first, then the conversions and stores
                    uint32_t w[2][4][4];
#pragma unroll
                    for (int which = 0; which < 2; ++which)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const int c = c0 + 2 * kk;
                            if (valid)
                                lds128(src + which * F8_V_OFF + ((c ^ (row & 7)) << 4), w[which][kk][0],
                                       w[which][kk][1], w[which][kk][2], w[which][kk][3]);
                            else
                                w[which][kk][0] = w[which][kk][1] = w[which][kk][2] = w[which][kk][3] = 0u;
                        }
#pragma unroll
                    for (int which = 0; which < 2; ++which)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const int c = c0 + 2 * kk;
                            const uint32_t base = dst + which * V_OFF + (c >> 2) * KV_HALF;
                            const int q0 = (2 * c) & 7, q1 = (2 * c + 1) & 7;   // d 16c .. +7 and 16c+8 .. +15
                            const uint32_t *x = w[which][kk];
                            st_shared_v4(base + ((q0 ^ (row & 7)) << 4), e4m3x2_to_f16x2(x[0] & 0xffffu),
                                         e4m3x2_to_f16x2(x[0] >> 16), e4m3x2_to_f16x2(x[1] & 0xffffu),
                                         e4m3x2_to_f16x2(x[1] >> 16));
                            st_shared_v4(base + ((q1 ^ (row & 7)) << 4), e4m3x2_to_f16x2(x[2] & 0xffffu),
                                         e4m3x2_to_f16x2(x[2] >> 16), e4m3x2_to_f16x2(x[3] & 0xffffu),
                                         e4m3x2_to_f16x2(x[3] >> 16));
                        }
                    fence_proxy_async_smem();
                    mbar_arrive(bar(B_KVF + st));
                    mbar_arrive(bar(B_F8E + s8));
                }
            }
        }
    } else {
        // ======================= softmax warpgroups: thread = query row = TMEM lane
        const int gi = warp >> 2;                  // which query tile of the pair
        const int r = threadIdx.x - gi * 128;      // row of the tile, 0..127
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        int cs = 0;         // tiles the group computed: S buffers, P and PV phases
        int kg = 0;         // items the group computed: drain (and fp8 Q) phases
        bool ok = true;
        for (int k = 0; ok; ++k) {
            ItemSlot it;
            if (!read_item(k, it)) break;
            if (gi == 1 && !it.has1) continue;     // no second query tile in this item
            const int n = it.n, L = it.L, j0 = it.j0, T = it.T, g = it.g, row0 = it.row0;
            const int split = it.split, nsplit = it.nsplit;
            const int i0 = (it.t0q + gi) * tpt, i1 = min(n, i0 + tpt);
            const int i = i0 + r / G;
            const int head = g * G + r % G;
            const bool row_valid = i < i1;
            // last key this row may attend; rows past the chunk (computed only to fill
            // the tile, never stored) take the tile's last valid row, so no row ever
            // sees a key at or beyond L
            const int pos = row_valid ? L - n + i : L - n + i1 - 1;
            const int pos_min = L - n + i0;
            float m_ref = -INFINITY, l = 0.f;
            // fp8 cache: the k scale folds into the softmax scale, the v scale into O
            const float sl = FP8 ? p.scale_log2 * __ldg(p.k_scale + g) : p.scale_log2;
            const float vsc = FP8 ? __ldg(p.v_scale + g) : 1.f;
            if constexpr (FP8) {
                // the group's Q tile, bf16 -> f16 in place (exact for these values'
                // range but the smallest subnormals), before its first product
                ok = wait_w(bar(B_Q), k & 1);
                if (ok) {
                    const uint32_t qt = sbase + SQ + gi * Q_TILE;
                    for (int c = r; c < Q_TILE / 16; c += 128) {
                        uint32_t w0, w1, w2, w3;
                        lds128(qt + c * 16, w0, w1, w2, w3);
                        auto cv = [](uint32_t w) -> uint32_t {
                            return pack_f16(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
                        };
                        st_shared_v4(qt + c * 16, cv(w0), cv(w1), cv(w2), cv(w3));
                    }
                    fence_proxy_async_smem();
                }
                mbar_arrive(bar(B_QC + gi));
            }
            for (int jj = 0; jj < T && ok; ++jj) {
                const int t0 = (j0 + jj) * BN;
                const int sb = (cs + jj) & 1;           // the tile's S buffer
                if (!wait_w(bar(B_S + 2 * gi + sb), ((cs + jj) >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                float sv[BN];
#pragma unroll
                for (int h = 0; h < BN / 64; ++h)
                    tmem_ld64(tS(gi, sb) + lane_base + 64 * h, *reinterpret_cast<float(*)[64]>(sv + 64 * h));
                // raw scores; the scale (> 0) is applied inside the exponent's FFMA,
                // so the max is taken on the raw values
                if (t0 + BN - 1 > pos_min) {             // diagonal tile: causal mask
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (t0 + c > pos) sv[c] = -INFINITY;
                }
                // max over the 64 scores: four independent chains of 3-input maxima
                float mk[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) mk[k] = fmaxf(sv[k], sv[4 + k]);        // elements 0..7
#pragma unroll
                for (int c = 8; c < BN; c += 8) {                                      // elements c..c+7
#pragma unroll
                    for (int k = 0; k < 4; ++k) mk[k] = max3(mk[k], sv[c + k], sv[c + 4 + k]);
                }
                const float mraw = max3(mk[0], mk[1], fmaxf(mk[2], mk[3]));
                const float mx = mraw * sl;
                float alpha = 1.f;
                if (mx > m_ref + RESCALE_LOG2 || (m_ref == -INFINITY && mx != -INFINITY)) {
                    alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - mx);
                    m_ref = mx;
                }
                // With no visible key yet (m_ref = -inf) every score is -inf and the
                // reference 0 keeps the exponent at -inf, i.e. p = 0.
                const float mneg = m_ref == -INFINITY ? 0.f : -m_ref;
                // exponent argument and running sum on packed fp32 pairs
                const uint64_t sl2 = f2_pack(sl, sl), mn2 = f2_pack(mneg, mneg);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
                uint32_t pw[BN / 2];
#pragma unroll
                for (int e = 0; e < BN / 2; ++e) {
                    float y0, y1;
                    f2_unpack(f2_fma(f2_pack(sv[2 * e], sv[2 * e + 1]), sl2, mn2), y0, y1);
                    const float p0 = ex2(y0), p1 = ex2(y1);
                    acc[e & 3] = f2_add(acc[e & 3], f2_pack(p0, p1));
                    pw[e] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
                }
                const uint64_t a2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
                float s0, s1;
                f2_unpack(a2, s0, s1);
                const float sum = s0 + s1;
                l = l * alpha + sum;
                // PV(jj-2), which read the P columns about to be overwritten, finished
                // before S(jj) (issued after it by the same thread) completed.  O is
                // rescaled only once PV(jj-1) has accumulated into it; PV(jj) waits
                // for this warp's P, so it cannot start before the rescale is done.
                if (jj > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    if (!wait_w(bar(B_PVD + gi), (cs + jj - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float o[32];
                        tmem_ld32(tO(gi) + lane_base + c * 32, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= alpha;
                        tmem_st32(tO(gi) + lane_base + c * 32, o);
                    }
                }
                // P in bf16 pairs over the first 32 columns of the S buffer (the A
                // operand of PV)
#pragma unroll
                for (int h = 0; h < BN / 64; ++h)
                    tmem_st32u(tS(gi, sb) + lane_base + 32 * h, *reinterpret_cast<const uint32_t(*)[32]>(pw + 32 * h));
                tmem_wait_st();
                tc_fence_before();
                // one P barrier per S buffer: a warp reaches buffer b's next phase only
                // after S(jj+2) completed, which the issuer started only once all 128
                // rows had arrived for this phase -- arrivals never mix two tiles
                mbar_arrive(bar(B_P + 2 * gi + sb));
            }
            // every MMA of the group's item has finished (the issuer's per-item drain
            // commit: PV(T-2) may still run here, so a parity wait on the per-tile
            // barrier could alias)
            if (ok && !wait_w(bar(B_DRAIN + gi), kg & 1)) ok = false;
            if (ok) {
                tc_fence_after();
                const size_t rh = (size_t)(row0 + (row_valid ? i : i0)) * p.hq + head;
                const size_t pi = rh * p.max_splits + split;
                const float inv = ((nsplit == 1 && l > 0.f) ? 1.f / l : (nsplit == 1 ? 0.f : 1.f)) * vsc;
                float4 *dst = reinterpret_cast<float4 *>(nsplit == 1 ? p.out + rh * D : p.part_o + pi * D);
#pragma unroll
                for (int c = 0; c < 4; ++c) {       // 32 columns at a time (the load is warp-wide)
                    float o[32];
                    tmem_ld32(tO(gi) + lane_base + c * 32, o);
                    if (row_valid) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            dst[c * 8 + e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv,
                                                         o[4 * e + 2] * inv, o[4 * e + 3] * inv);
                    }
                }
                if (row_valid && nsplit > 1) {
                    p.part_ml[pi * 2] = l > 0.f ? m_ref : -INFINITY;
                    p.part_ml[pi * 2 + 1] = l;
                }
            }
            cs += T;
            ++kg;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);   // (both layouts allocate all 512 columns)
}

// Log-sum-exp merge of prefill partitions: one warp per (query row, head).
// (grid-stride; nothing to do when tile_prefix_kernel cut no key range)
// (512 threads: few CTAs to start and retire when there is nothing to merge)
constexpr int MERGE_WARPS = 16;
__global__ void __launch_bounds__(MERGE_WARPS * 32) prefill_reduce_kernel(const PrefillParams p)
{
    griddep_wait();   // launched with programmatic serialisation after the chunk kernel
    if (p.order_count[2] == 0) return;
    const int lane = threadIdx.x & 31;
    const long nw = (long)p.total_rows * p.hq;
    for (long wid = (long)blockIdx.x * MERGE_WARPS + (threadIdx.x >> 5); wid < nw;
         wid += (long)gridDim.x * MERGE_WARPS) {
        const int row = (int)(wid / p.hq), h = (int)(wid % p.hq);
        // the partitions of the query item the row belongs to (tile_prefix_kernel
        // wrote them; 0 for rows outside any chunk)
        const int ns = min(p.row_info[row], p.max_splits);
        if (ns <= 1) continue;
        const size_t base = ((size_t)row * p.hq + h) * p.max_splits;
        reinterpret_cast<float4 *>(p.out + ((size_t)row * p.hq + h) * D)[lane] =
            lse_merge_warp(p.part_ml + base * 2, p.part_o + base * D, ns, lane);
    }
}

constexpr int MAX_SPLIT_KEYS = 16384;           // keys per partition at most
constexpr int MIN_SPLIT_KEYS = 1024;            // and at least
constexpr int64_t NUM_SMS = 152;               // a chunk CTA holds a whole SM: waves of 152
constexpr double CTA_FIXED_TILES = 4.0;        // a CTA's Q load, set-up and epilogue, in tile-times
// HBM bytes moved while a CTA works through one 64-key tile (~0.86 us at ~6.5 TB/s)
constexpr double BYTES_PER_TILE_TIME = 5.6e6;
// bytes the decode kernel's CTAs on one SM (three of them) read while a chunk CTA
// works through one 64-key tile, with the chunk kernel on the other SMs.  Fitted
// on GB300 to the mixed batch (1,024-row chunk + 255 decode rows): the best
// whole call came with 140 chunk CTAs of 152 (bf16 cache), 3.098 ms, against
// 3.157-3.353 ms at 124-136 and 3.150-3.263 ms at 144-148; this rate makes the
// model take 139 (and 145 over an fp8 cache, whose decode rows read half the
// bytes: 3.150-3.155 ms at 140-148)
constexpr double DECODE_SM_BYTES_PER_TILE_TIME = 120.0 * 1024.0;

struct Plan {
    size_t decode_bytes, part_o_off, part_ml_off, tile_off_off, order_off, row_info_off, total;
    int max_splits, tiles_per_split;
    int64_t items_ub;    // bounds the query items: sum over chunks of ceil(n / tpt)
};

}  // namespace

namespace pkv_decode {
kv_status run(float *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens,
              const int32_t *cu_q_lens, int32_t total_rows, int32_t num_seqs, int32_t hq, int32_t hkv,
              int32_t num_blocks, float scale, kv_dtype dt, const float *k_scale, const float *v_scale,
              int32_t num_splits, void *workspace, size_t workspace_bytes_given, cudaStream_t st,
              int32_t multi_q_len, bool pdl, bool corun);
size_t workspace_bytes(int32_t num_seqs, int32_t hq, int32_t max_blocks, int32_t num_splits);
size_t workspace_bytes_multi(int32_t total_rows, int32_t num_seqs, int32_t hq, int32_t max_blocks,
                             int32_t num_splits);
bool make_maps(const void *k_cache, const void *v_cache, int32_t num_blocks, int32_t hkv, kv_dtype dt,
               CUtensorMap *km, CUtensorMap *vm);
void plan_splits(int32_t max_blocks, int32_t num_splits, int32_t num_seqs, int32_t hq, int32_t *part_blocks,
                 int32_t *splits);
}  // namespace pkv_decode

namespace {
// KV partitions of a chunk's keys.  Every CTA (one per pair of query tiles, KV
// head and partition) holds a whole SM, so the grid runs in waves of NUM_SMS
// CTAs, and the partitions of a key range are of equal length.  Their count s
// minimises a makespan model: waves(s) x (W / s + CTA_FIXED_TILES) tile-times,
// plus -- when s > 1 -- each partition's partial results written and merged
// (rows x heads x 130 floats, twice), converted to tile-times.  W is the longest
// key range in tiles, and the number of (pair, KV head) problems is estimated
// from host-visible sizes only: chunk sequences ~ total_q / max_q_len, each with
// ceil(ceil(max_q_len / tpt) / 2) pairs of query tiles.  Equal partitions alone
// can leave a last wave almost empty (768 CTAs = 5.05 waves), which the model
// avoids by taking one more partition.  Returns the partition length in tiles.
int plan_tiles_per_split(int32_t total_q, int32_t max_q_len, int32_t hq, int32_t hkv, int max_kv_tiles,
                         bool big)
{
    const int G = std::max(1, hq / std::max(1, hkv)), tpt = std::max(1, BM / G);
    const int64_t chunks = std::max<int64_t>(1, (int64_t)total_q / std::max(1, max_q_len));
    const int item = big ? 1 : 2;                       // query tiles per CTA
    const int64_t items = chunks * ((((int64_t)max_q_len + tpt - 1) / tpt + item - 1) / item);
    const int64_t problems = std::max<int64_t>(1, items * std::max(1, hkv));
    const int W = std::max(1, max_kv_tiles);
    const int tile_keys = big ? 128 : 64;              // W and the result are in tiles of tile_keys
    const int TILES_PER_SPLIT = MAX_SPLIT_KEYS / tile_keys, MIN_TILES_PER_SPLIT = MIN_SPLIT_KEYS / tile_keys;
    const double CTA_FIXED = CTA_FIXED_TILES * 64.0 / tile_keys;
    const double merge_per_split =
        (double)total_q * hq * (D + 2) * 4.0 * 2.0 / (BYTES_PER_TILE_TIME * tile_keys / 64.0);
    const int s_lo = (W + TILES_PER_SPLIT - 1) / TILES_PER_SPLIT;
    // (the partition count is the grid's z extent: at most 65,535)
    const int s_hi = std::max(s_lo, std::min(65535, (W + MIN_TILES_PER_SPLIT - 1) / MIN_TILES_PER_SPLIT));
    auto cost = [&](int s) {
        const int len = (W + s - 1) / s;
        const int splits = (W + len - 1) / len;        // what the kernel makes of len
        const int64_t waves = (problems * splits + NUM_SMS - 1) / NUM_SMS;
        return (double)waves * (len + CTA_FIXED) + (splits > 1 ? splits * merge_per_split : 0.0);
    };
    double best = cost(s_lo);
    for (int s = s_lo + 1; s <= s_hi; ++s) best = std::min(best, cost(s));
    // the model takes every key range as long as the longest; with several chunk
    // sequences the real ranges are ragged, which favours finer partitions: then
    // the most partitions within 2% of the best modelled cost
    const double slack = chunks > 1 ? 1.02 : 1.0;
    int pick = s_lo;
    for (int s = s_lo; s <= s_hi; ++s)
        if (cost(s) <= best * slack) pick = s;
    return (W + pick - 1) / pick;
}

Plan make_plan(int32_t num_seqs, int32_t total_q, int32_t max_q_len, int32_t hq, int32_t hkv, int32_t max_blocks,
               int32_t num_splits, bool big)
{
    Plan pl{};
    auto up = [](size_t v) { return (v + 255) & ~size_t(255); };
    pl.decode_bytes = up(pkv_decode::workspace_bytes(num_seqs, hq, max_blocks, num_splits));
    const int tile_keys = big ? 128 : 64;
    const int max_kv_tiles = (max_blocks * BS + tile_keys - 1) / tile_keys;
    pl.tiles_per_split = plan_tiles_per_split(total_q, max_q_len, hq, hkv, max_kv_tiles, big);
    pl.max_splits = max_q_len >= 2 ? (max_kv_tiles + pl.tiles_per_split - 1) / pl.tiles_per_split : 0;
    size_t off = pl.decode_bytes;
    pl.part_o_off = off;
    if (pl.max_splits > 1) off += up((size_t)total_q * hq * pl.max_splits * D * sizeof(float));
    pl.part_ml_off = off;
    if (pl.max_splits > 1) off += up((size_t)total_q * hq * pl.max_splits * 2 * sizeof(float));
    pl.tile_off_off = off;
    if (max_q_len >= 2) off += up((size_t)(num_seqs + 1) * sizeof(int32_t));
    // the work items in launch order (two int4 each), then their count and the
    // CTAs' fetch counter; then each query row's partition count
    const int G = std::max(1, hq / std::max(1, hkv)), tpt = std::max(1, BM / G);
    pl.items_ub = ((int64_t)total_q + tpt - 1) / tpt + std::min<int64_t>(num_seqs, total_q / 2);
    pl.order_off = off;
    if (max_q_len >= 2)
        off += up((size_t)pl.items_ub * hkv * std::max(1, pl.max_splits) * 2 * sizeof(int4)) + up(4 * sizeof(int32_t));
    pl.row_info_off = off;
    if (max_q_len >= 2) off += up((size_t)total_q * sizeof(int32_t));
    pl.total = off;
    return pl;
}

// Short chunks (a speculative draft being verified, a few rows per sequence)
// are memory-bound like decode: when every sequence's rows x the group's heads
// fit in MULTI_MAX_COLS columns, the whole batch runs in the decode kernel's
// multi-row mode, which streams each K/V tile once for all the rows of its
// sequence.  That is up to one MMA column tile (8 columns); measured on GB300,
// 16 columns (4-token drafts at G = 4) ran at 0.752 of HBM there against 0.775
// in the persistent tensor-core kernel.
#ifndef PKV_MULTI_MAX_COLS
#define PKV_MULTI_MAX_COLS 8
#endif
constexpr int64_t MULTI_MAX_COLS = PKV_MULTI_MAX_COLS;

bool use_multi(int32_t max_q_len, int32_t hq, int32_t hkv)
{
    return max_q_len >= 2 && hkv >= 1 && (int64_t)max_q_len * (hq / hkv) <= MULTI_MAX_COLS;
}

// The 128-key layout (one query tile per CTA) when every chunk's rows x heads
// fit one 128-row tile; bf16 cache.
bool use_big(kv_dtype dt, int32_t max_q_len, int32_t hq, int32_t hkv)
{
    return dt == KV_BF16 && hkv >= 1 && (int64_t)max_q_len * (hq / hkv) <= BM;
}
}  // namespace

namespace {
constexpr int MAX_DEVICES = 64;

// SMs of the current device (the persistent chunk grid's size)
int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return (int)NUM_SMS;
    return n;
}

}  // namespace

namespace {
// Tracing aid: CUDA events around the tensor-core chunk kernel of each call,
// per device, recorded only while enabled (not during stream capture).
struct Trace {
    cudaEvent_t start = nullptr, stop = nullptr;
    bool recorded = false;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
Trace g_trace[MAX_DEVICES];

Trace *trace_for_call()
{
    std::lock_guard<std::mutex> g(g_trace_mu);
    if (!g_trace_on) return nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
    Trace &t = g_trace[dev];
    if (!t.start && (cudaEventCreate(&t.start) != cudaSuccess || cudaEventCreate(&t.stop) != cudaSuccess))
        return nullptr;
    return &t;
}
}  // namespace

namespace pkv_prefill {
uint32_t take_status()
{
    uint32_t v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_status, &z, sizeof z);
    return v;
}
}  // namespace pkv_prefill

extern "C" {

size_t paged_attention_chunked_prefill_workspace_size(int32_t num_seqs, int32_t total_q_tokens,
                                                      int32_t max_q_len, int32_t num_q_heads,
                                                      int32_t num_kv_heads,
                                                      int32_t max_blocks_per_seq,
                                                      int32_t num_splits)
{
    if (num_seqs < 1 || total_q_tokens < 1 || max_q_len < 1 || num_q_heads < 1 || max_blocks_per_seq < 1 ||
        num_kv_heads < 1)
        return 0;
    // (the size query has no cache type: room for the plan of either layout)
    size_t t = make_plan(num_seqs, total_q_tokens, max_q_len, num_q_heads, num_kv_heads, max_blocks_per_seq,
                         num_splits, false).total;
    if (use_big(KV_BF16, max_q_len, num_q_heads, num_kv_heads))
        t = std::max(t, make_plan(num_seqs, total_q_tokens, max_q_len, num_q_heads, num_kv_heads,
                                  max_blocks_per_seq, num_splits, true).total);
    if (use_multi(max_q_len, num_q_heads, num_kv_heads))
        t = std::max(t, pkv_decode::workspace_bytes_multi(total_q_tokens, num_seqs, num_q_heads, max_blocks_per_seq,
                                                          num_splits));
    return t;
}

int32_t paged_attention_launch_count(int32_t num_seqs, int32_t total_q_tokens, int32_t max_q_len,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t max_blocks_per_seq,
                                     int32_t num_splits)
{
    if (num_seqs < 1 || total_q_tokens < 1 || max_q_len < 1 || num_q_heads < 1 || num_kv_heads < 1 ||
        max_blocks_per_seq < 1)
        return 0;
    // the decode kernel, plus its LSE merge when the context is partitioned
    int32_t pb = 0, s = 0;
    pkv_decode::plan_splits(max_blocks_per_seq, num_splits, num_seqs, num_q_heads, &pb, &s);
    const int32_t decode = 1 + (s > 1 ? 1 : 0);
    if (max_q_len < 2 || use_multi(max_q_len, num_q_heads, num_kv_heads)) return decode;
    // the decode rows (none when every query is max_q_len long), the work list,
    // the chunk tiles and their merge (the plan of a bf16 cache)
    const Plan pl = make_plan(num_seqs, total_q_tokens, max_q_len, num_q_heads, num_kv_heads, max_blocks_per_seq,
                              num_splits, use_big(KV_BF16, max_q_len, num_q_heads, num_kv_heads));
    const bool rows1 = (int64_t)total_q_tokens != (int64_t)num_seqs * max_q_len;
    return (rows1 ? decode : 0) + 2 + (pl.max_splits > 1 ? 1 : 0);
}

kv_status paged_attention_chunked_prefill(float *out, const void *q, const int32_t *cu_q_lens,
                                          const int32_t *context_lens, int32_t num_seqs,
                                          int32_t total_q_tokens, int32_t max_q_len,
                                          const void *k_cache, const void *v_cache,
                                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                                          int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t num_blocks, float scale, kv_dtype dtype,
                                          const float *k_scale, const float *v_scale,
                                          int32_t num_splits, void *workspace,
                                          size_t workspace_bytes, void *stream)
{
    PKV_NVTX_RANGE("paged_attention_chunked_prefill");
    if (num_seqs == 0 || total_q_tokens == 0) return KV_OK;
    if (num_seqs < 0 || total_q_tokens < 0 || max_q_len < 1 || !cu_q_lens || !context_lens || !out || !q ||
        !k_cache || !v_cache || !block_tables || num_q_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 1 ||
        num_blocks < 1 || num_q_heads % num_kv_heads)
        return KV_ERR_INVALID;
    const int G = num_q_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return KV_ERR_UNSUPPORTED;
    if (dtype != KV_BF16 && dtype != KV_FP8_E4M3) return KV_ERR_UNSUPPORTED;
    if (!(scale > 0.f) || num_seqs > 65535 || num_kv_heads > 65535) return KV_ERR_INVALID;
    if (!pkv_host::aligned(out, 16) || !pkv_host::aligned(q, 16)) return KV_ERR_INVALID;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (use_multi(max_q_len, num_q_heads, num_kv_heads)) {
        // short chunks: the decode kernel's multi-row mode for the whole batch
        return pkv_decode::run(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, cu_q_lens,
                               total_q_tokens, num_seqs, num_q_heads, num_kv_heads, num_blocks, scale, dtype,
                               k_scale, v_scale, num_splits, workspace, workspace_bytes, st, max_q_len, true,
                               false);
    }
    if (dtype == KV_FP8_E4M3 && (!k_scale || !v_scale)) return KV_ERR_INVALID;
    const bool big = use_big(dtype, max_q_len, num_q_heads, num_kv_heads);
    const Plan pl = make_plan(num_seqs, total_q_tokens, max_q_len, num_q_heads, num_kv_heads, max_blocks_per_seq,
                              num_splits, big);
    if (pl.total && (!workspace || workspace_bytes < pl.total || !pkv_host::aligned(workspace, 256)))
        return KV_ERR_INVALID;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    auto decode_rows = [&](cudaStream_t on, bool pdl, bool beside) {
        return pkv_decode::run(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, cu_q_lens,
                               total_q_tokens, num_seqs, num_q_heads, num_kv_heads, num_blocks, scale, dtype,
                               k_scale, v_scale, num_splits, pl.decode_bytes ? ws : nullptr, pl.decode_bytes, on,
                               0, pdl, beside);
    };
    if (max_q_len < 2) return decode_rows(st, true, false);   // decode rows only
    // decode rows (n = 1): none when total_q_tokens = num_seqs x max_q_len (every
    // query is max_q_len long; tile_prefix_kernel flags a row of 1 then)
    const bool rows1 = (int64_t)total_q_tokens != (int64_t)num_seqs * max_q_len;
    // prefill chunks (n >= 2)
    PrefillParams p{};
    p.out = out;
    p.q = static_cast<const uint16_t *>(q);
    p.cu_q_lens = cu_q_lens;
    p.context_lens = context_lens;
    p.block_tables = block_tables;
    p.tile_off = reinterpret_cast<int32_t *>(ws + pl.tile_off_off);
    p.order = reinterpret_cast<int4 *>(ws + pl.order_off);
    p.row_info = reinterpret_cast<int32_t *>(ws + pl.row_info_off);
    p.items_cap = (int)std::min<int64_t>(pl.items_ub, INT32_MAX);
    p.order_count = reinterpret_cast<int32_t *>(
        ws + pl.order_off + ((pl.items_ub * num_kv_heads * std::max(1, pl.max_splits) * 2 * sizeof(int4) + 255) & ~size_t(255)));
    p.part_o = pl.max_splits > 1 ? reinterpret_cast<float *>(ws + pl.part_o_off) : nullptr;
    p.part_ml = pl.max_splits > 1 ? reinterpret_cast<float *>(ws + pl.part_ml_off) : nullptr;
    p.max_blocks = max_blocks_per_seq;
    p.num_seqs = num_seqs;
    p.hq = num_q_heads;
    p.hkv = num_kv_heads;
    p.group = G;
    p.num_blocks = num_blocks;
    p.total_rows = total_q_tokens;
    p.tiles_per_split = pl.tiles_per_split;
    p.max_splits = std::max(1, pl.max_splits);
    p.scale_log2 = scale * LOG2E;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.item_tiles = big ? 1 : 2;
    p.tile_keys = big ? 128 : 64;
    p.num_sms = num_sms();
    p.rows1 = rows1 ? 1 : 0;
    p.max_q_len = max_q_len;
    p.bytes_per_tile = (float)(BYTES_PER_TILE_TIME * p.tile_keys / 64.0);
    Trace *tr = trace_for_call();
    // (a traced call times the chunk kernel alone: its decode rows run after it)
    p.corun = rows1 && !tr ? 1 : 0;
    p.decode_key_bytes = (float)num_kv_heads * D * 2 * (dtype == KV_FP8_E4M3 ? 1 : 2);
    p.decode_sm_bytes = (float)(DECODE_SM_BYTES_PER_TILE_TIME * p.tile_keys / 64.0);
    CUtensorMap qm, km, vm;
    const int tpt = BM / G;
    // the 128-key layout holds one query tile per sequence (max_q_len x G <= 128):
    // only its max_q_len rows are loaded; the tile's other rows keep what shared
    // memory held (their scores and outputs stay in their own rows, never stored)
    const int q_rows = big ? std::min(tpt, max_q_len) : tpt;
    p.q_box_bytes = q_rows * G * 128;
    if (!pkv_host::encode_tmap_3d(&qm, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, num_q_heads, total_q_tokens,
                                  (uint64_t)D * 2, (uint64_t)num_q_heads * D * 2, 64, G, q_rows,
                                  CU_TENSOR_MAP_SWIZZLE_128B))
        return KV_ERR_CUDA;
    if (!pkv_decode::make_maps(k_cache, v_cache, num_blocks, num_kv_heads, dtype, &km, &vm)) return KV_ERR_CUDA;
    const bool fp8 = dtype == KV_FP8_E4M3;
    // bf16 chunk tiles: the V of one (block, head) as one 3-D box holding both
    // 64-dim halves ([half][16 keys][64 dims] in shared memory): dims (64 dims,
    // rows, halves), strides (row 256 B, half 128 B)
    if (!fp8 && !pkv_host::encode_tmap_3d(&vm, v_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64,
                                          (uint64_t)num_blocks * num_kv_heads * BS, 2, (uint64_t)D * 2, 128,
                                          64, BS, 2, CU_TENSOR_MAP_SWIZZLE_128B))
        return KV_ERR_CUDA;
    const cudaError_t smem_ok =
        big   ? pkv_host::ensure_dynamic_smem<prefill_kernel<false, true>>(Lay<false, true>::SMEM_BYTES)
        : fp8 ? pkv_host::ensure_dynamic_smem<prefill_kernel<true, false>>(Lay<true>::SMEM_BYTES)
              : pkv_host::ensure_dynamic_smem<prefill_kernel<false, false>>(Lay<false>::SMEM_BYTES);
    if (smem_ok != cudaSuccess) return KV_ERR_CUDA;
    // one CTA per work item (query item, KV head, partition), in the order that
    // tile_prefix_kernel writes; the grid bounds their number
    const int64_t ctas_ub = pl.items_ub * num_kv_heads * p.max_splits;
    if (ctas_ub > INT32_MAX || p.max_splits > 65535 || num_kv_heads > 65535) return KV_ERR_UNSUPPORTED;
    p.grid_ctas = (int)std::min<int64_t>(ctas_ub, p.num_sms);
    // (a plain launch when there are decode rows: the decode CTAs, which start
    // while the chunk kernel runs, read their inputs without waiting, so every
    // kernel before this call must have finished)
    // (its block: a thread per sequence or per four query rows, 128 to 1,024.
    // The kernel is a chain of block-wide phases, so idle warps cost issue slots
    // at every one of them -- 1,024 threads took 7.4 us for 32 sequences of 8
    // rows -- while the per-row phase wants threads: 128 took 2.5 us longer than
    // 1,024 for 1,087 rows)
    const int64_t tp_want = std::max<int64_t>(num_seqs, ((int64_t)total_q_tokens + 3) / 4);
    const int tp_threads = (int)std::min<int64_t>(1024, std::max<int64_t>(128, (tp_want + 31) / 32 * 32));
    if (pkv_host::launch_ex(tile_prefix_kernel, dim3(1), dim3((unsigned)tp_threads), 0, st, !rows1, p) !=
        cudaSuccess)
        return KV_ERR_CUDA;
    // persistent: one CTA per SM (a CTA holds a whole SM), at most one per work item
    dim3 grid((unsigned)p.grid_ctas);
    if (tr) cudaEventRecord(tr->start, st);
    // programmatic serialisation: the CTAs' set-up overlaps tile_prefix_kernel
    // (trace events between the two only make the launch plain)
    const bool pdl = !tr;
    cudaError_t le;
    if (big)
        le = pkv_host::launch_ex(prefill_kernel<false, true>, grid, dim3(Lay<false, true>::THREADS),
                                 Lay<false, true>::SMEM_BYTES, st, pdl, qm, km, vm, p);
    else if (fp8)
        le = pkv_host::launch_ex(prefill_kernel<true, false>, grid, dim3(Lay<true>::THREADS), Lay<true>::SMEM_BYTES,
                                 st, pdl, qm, km, vm, p);
    else
        le = pkv_host::launch_ex(prefill_kernel<false, false>, grid, dim3(Lay<false>::THREADS),
                                 Lay<false>::SMEM_BYTES, st, pdl, qm, km, vm, p);
    if (le != cudaSuccess) return KV_ERR_CUDA;
    if (tr) {
        cudaEventRecord(tr->stop, st);
        tr->recorded = true;
    }
    if (cudaGetLastError() != cudaSuccess) return KV_ERR_CUDA;
    if (rows1) {
        // the decode rows, launched programmatically behind the chunk kernel: their
        // CTAs start on the SMs the chunk kernel leaves free while it runs (a chunk
        // CTA's shared memory leaves no room for one beside it), and on every SM
        // once it is done
        const kv_status r = decode_rows(st, true, p.corun != 0);
        if (r != KV_OK) return r;
    }
    if (p.max_splits > 1) {
        const int64_t warps = (int64_t)total_q_tokens * num_q_heads;
        if (pkv_host::launch_ex(prefill_reduce_kernel,
                                dim3((unsigned)std::min<int64_t>((warps + MERGE_WARPS - 1) / MERGE_WARPS,
                                                                 (int64_t)p.num_sms * 4)),
                                dim3(MERGE_WARPS * 32), 0, st, !tr, p) != cudaSuccess)
            return KV_ERR_CUDA;
    }
    return KV_OK;
}

kv_status kv_trace_prefill(int32_t enable)
{
    std::lock_guard<std::mutex> g(g_trace_mu);
    g_trace_on = enable != 0;
    return KV_OK;
}

double kv_trace_prefill_kernel_ms(void)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return -1.0;
    std::lock_guard<std::mutex> g(g_trace_mu);
    Trace &t = g_trace[dev];
    if (!t.recorded || cudaEventSynchronize(t.stop) != cudaSuccess) return -1.0;
    float ms = -1.f;
    if (cudaEventElapsedTime(&ms, t.start, t.stop) != cudaSuccess) return -1.0;
    t.recorded = false;
    return ms;
}

}  // extern "C"
