// decode.cu -- paged decode attention for sm_103a.
//
// One query token per sequence attends every key of its context, read
// through the block table ("Waste, and three ways to reclaim it", section
// "PagedAttention": a matching attention kernel that knows how to read from
// scattered blocks; "M.65 Inference serving", block management (d)).  Softmax
// is computed online: a running max and normaliser updated per 16-token block
// ("PagedAttention, chunked prefill, and the launch that cascades", section
// "FlashAttention").  GQA: the G query heads of one KV head share every K/V
// tile ("Kernel engineering": repeat_interleave grouping, h -> h / G).
//
// Design (GB300):
//  * Work item = (split partition, KV head, sequence): one CTA of 4 warps.  A
//    partition is a run of whole *logical* blocks; warp w takes blocks
//    w, w+4, ... of it.  Split points depend only on logical positions.
//  * Every (block, KV head) tile of K and of V is contiguous in HBM (4 KiB bf16,
//    2 KiB fp8).  Each warp owns a private ring of stages; its lane 0 issues
//    TMA tiled loads (128-byte swizzle) of the K and V tile of a future block
//    into a stage, completion counted on the stage's mbarrier.  Three CTAs per
//    SM keep ~190 KiB of loads in flight, which HBM3e needs at this tile size.
//  * Scores: S^T[16 tokens][8 heads] = K[16][128] . Q^T[128][8] on the tensor
//    cores (mma.sync m16n8k16, tokens on M, the GQA group on N) -- G = 8 fills
//    the tile exactly.  K comes from shared memory with ldmatrix (conflict-free
//    thanks to the swizzle); Q's B fragments stay in registers all kernel.
//  * P^T is transposed inside the warp with movmatrix and becomes the B operand
//    of O^T[128][8] += V^T[128][16] . P^T[16][8] (V via ldmatrix.trans).
//  * fp8 cache: e4m3 -> f16 is exact, so K/V are widened in registers and the
//    f16 MMA is used; k_scale folds into the softmax scale, v_scale into the
//    epilogue.  For fp8 V the transpose is done with 16-byte shared loads and
//    byte permutes; the D index is permuted consistently and undone at the end.
//  * The 4 warps merge their (max, sum, O) in shared memory; a partition that
//    covers the whole sequence writes the normalised output, otherwise it
//    writes its partial (max, sum, O) and a second kernel merges the
//    partitions with the log-sum-exp rule in fixed order -- no atomics, so the
//    result is bitwise independent of physical placement.
#include "common.cuh"
#include "trace.h"

#include <algorithm>
#include <mutex>

// ---- device code begin (hashed with the ncu counters of profiles/)
namespace {

__device__ uint32_t g_status;

using namespace pkv;

constexpr int WARPS = 4;
constexpr int THREADS = WARPS * 32;
constexpr float LOG2E = 1.4426950408889634f;

struct DecodeParams {
    float *out;
    const uint16_t *q;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *cu_q_lens;  // mixed batches: only sequences with one query row
    int total_rows;            // rows of q/out (mixed batches)
    int col_groups;            // multi-row mode: CTAs per (split, KV head, sequence) over the columns
    const float *k_scale;
    const float *v_scale;
    float *part_o;             // [B][Hq][S][128]   (B = rows in the multi-row mode)
    float *part_ml;            // [B][Hq][S][2]
    int max_blocks;
    int num_seqs;
    int hq;
    int hkv;
    int group;
    int num_blocks;
    int part_blocks;
    int num_splits;
    float scale_log2;          // softmax scale * log2(e)
    // launched programmatically right after the chunk-prefill kernel of the same
    // call, to run beside it: every input was written before that call's first
    // kernel, so only the first CTA waits for the chunk kernel (the grid then
    // completes after it, and the kernels behind it see both grids' results)
    int corun;
};

// Ring depth per warp and CTAs per SM (compile-time).  Measured on GB300:
// 2 bf16 stages (4 fp8) of 8 KiB per warp with 3 CTAs per SM beat deeper
// rings with fewer CTAs on every decode workload -- more CTAs hide each
// CTA's ramp-up, and 3 x 4 warps x 16 KiB still keeps ~190 KiB in flight.
#ifndef PKV_DECODE_STAGES_BF16
#define PKV_DECODE_STAGES_BF16 2
#endif
#ifndef PKV_DECODE_STAGES_FP8
#define PKV_DECODE_STAGES_FP8 4
#endif
#ifndef PKV_DECODE_MIN_CTAS
#define PKV_DECODE_MIN_CTAS 3
#endif

template <bool FP8>
struct Geo {
    static constexpr int TILE = FP8 ? 2048 : 4096;       // bytes of one K or V tile
    static constexpr int STAGE = 2 * TILE;               // K + V
    static constexpr int STAGES = FP8 ? PKV_DECODE_STAGES_FP8 : PKV_DECODE_STAGES_BF16;
    static constexpr int RING = STAGES * STAGE;
    static constexpr int SMEM = WARPS * RING + 1024 + 256;
};

__device__ __forceinline__ void flag(uint32_t bits) { atomicOr(&g_status, bits); }

// Multi-row mode: the context length of the sequence owning query row r of a
// mixed batch (binary search over cu_q_lens), 0 for a malformed batch.
__device__ __forceinline__ int row_seq_len(const DecodeParams &p, int r)
{
    const int32_t *cu = p.cu_q_lens;
    int lo = 0, hi = p.num_seqs;                 // cu[lo] <= r < cu[hi] if well formed
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= r) lo = mid;
        else hi = mid;
    }
    const int a = __ldg(cu + lo), b = __ldg(cu + lo + 1);
    if (r < a || r >= b) return 0;
    const int len = __ldg(p.context_lens + lo);
    return (b - a > len || len > p.max_blocks * BS) ? 0 : len;
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int32_t x, int32_t y,
                                                 uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

template <bool FP8>
__device__ __forceinline__ void issue_stage(uint32_t dst, uint32_t bar, const CUtensorMap *km,
                                            const CUtensorMap *vm, int32_t y, uint64_t pol)
{
    mbar_arrive_expect_tx(bar, Geo<FP8>::STAGE);
    if constexpr (FP8) {
        tma_load_2d_hint(dst, km, 0, y, bar, pol);
        tma_load_2d_hint(dst + Geo<FP8>::TILE, vm, 0, y, bar, pol);
    } else {
        tma_load_2d_hint(dst, km, 0, y, bar, pol);
        tma_load_2d_hint(dst + 2048, km, 64, y, bar, pol);
        tma_load_2d_hint(dst + 4096, vm, 0, y, bar, pol);
        tma_load_2d_hint(dst + 4096 + 2048, vm, 64, y, bar, pol);
    }
}

// MR (multi-row): one CTA covers CW = 8 NT columns of the (query row, head)
// pairs of one sequence and one KV head -- the n rows of a chunk x the G heads
// of the group, column c -> row c / G, head c % G -- so a short chunk (a
// speculative draft being verified) reads each K/V tile once for all its
// rows.  Row i of the chunk sees keys 0 .. L-n+i; longer chunks take several
// column groups (CTAs next to each other in the grid, sharing tiles in L2).
template <bool FP8, int NT, bool MR>
__global__ void __launch_bounds__(THREADS, PKV_DECODE_MIN_CTAS)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const DecodeParams p)
{
    using GE = Geo<FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + WARPS * GE::RING);

    constexpr int CW = NT * 8;               // columns of this CTA
    const int g = blockIdx.y;
    int split = blockIdx.x, cg = 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    // launched with programmatic serialisation: the CTA may be resident before
    // the previous kernel on the stream (typically the cache write) finished
    if (!p.corun || (blockIdx.x | blockIdx.y | blockIdx.z) == 0) griddep_wait();

    // s: sequence (block table); row: (first) row of q/out; wi: index of the
    // partials; nq: query rows of the sequence this CTA covers
    int s = blockIdx.z, row = s, wi = s, L, nq = 1;
    if constexpr (MR) {
        cg = split % p.col_groups;
        split /= p.col_groups;
        const int a = p.cu_q_lens[s], b = p.cu_q_lens[s + 1];
        nq = b - a;
        L = p.context_lens[s];
        if (nq == 0) return;
        // (nq x G > col_groups x CW: more rows than the caller's max_q_len allowed for)
        if (nq < 0 || a < 0 || b > p.total_rows || nq > L || L < 1 || L > p.max_blocks * BS ||
            nq * p.group > p.col_groups * CW) {
            if (split == 0 && cg == 0) {
                if (threadIdx.x == 0) flag(ST_BAD_LEN);
                if (nq > 0 && a >= 0 && b <= p.total_rows)
                    for (int i = threadIdx.x; i < nq * p.group * D; i += THREADS) {
                        const int r = i / (p.group * D), rem = i % (p.group * D);
                        p.out[((size_t)(a + r) * p.hq + g * p.group) * D + rem] = 0.f;
                    }
            }
            return;
        }
        if (cg * CW >= nq * p.group) return;
        row = a;
    } else {
        if (p.cu_q_lens) {
            int a = p.cu_q_lens[s], b = p.cu_q_lens[s + 1];
            if (b - a != 1) return;
            if (a < 0 || b > p.total_rows) {
                if (split == 0 && g == 0 && threadIdx.x == 0) flag(ST_BAD_LEN);
                return;
            }
            row = a;
        }
        L = p.context_lens[s];
    }
    if (L < 1 || L > p.max_blocks * BS) {
        if (split == 0) {
            if (threadIdx.x == 0) flag(ST_BAD_LEN);
            for (int i = threadIdx.x; i < p.group * D; i += THREADS)
                p.out[((size_t)row * p.hq + g * p.group) * D + i] = 0.f;
        }
        return;
    }
    const int nblk = (L + BS - 1) / BS;
    const int b0 = split * p.part_blocks;
    if (b0 >= nblk) return;
    const int b1 = min(nblk, b0 + p.part_blocks);
    const int nsplit_s = (nblk + p.part_blocks - 1) / p.part_blocks;
    const int32_t *bt = p.block_tables + (size_t)s * p.max_blocks;
    // blocks of this warp: b0 + warp + k * WARPS, k < count
    // (b1 - b0 >= 1 and warp <= 3, so the numerator is never negative)
    const int count = (b1 - b0 - warp + WARPS - 1) / WARPS;

    // L2 policy of the K/V loads.  A sequence's later partitions are read once,
    // so they are marked evict-first; its first partition keeps the normal
    // policy.  Blocks shared between sequences -- a common prompt prefix -- sit
    // at the start of every sharer's table, so they stay in L2 for the other
    // sharers instead of being pushed out by the read-once stream (measured on
    // the 128-sequence shared-prefix batch: 3.5% less time, the prefix's
    // re-reads no longer reaching DRAM).
    uint64_t l2pol;
    if (split > 0) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(l2pol));
    else asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(l2pol));
    const uint32_t ring = smem_u32(smem + warp * GE::RING);
    const uint32_t bar0 = smem_u32(bars + warp * GE::STAGES);
    if (lane == 0) {
        for (int i = 0; i < GE::STAGES; ++i) mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // block ids of this warp, 32 at a time: lane i holds the id of block k0 + i
    auto load_ids = [&](int k0) -> int32_t {
        int k = k0 + lane;
        return k < count ? __ldg(bt + b0 + warp + k * WARPS) : -1;
    };
    int32_t ids_cur = load_ids(0), ids_nxt = load_ids(32);
    int win = 0;  // window base of ids_cur

    auto block_id = [&](int k) -> int32_t {
        // k is in [win, win + 64)
        int32_t a = __shfl_sync(0xffffffffu, ids_cur, (k - win) & 31);
        int32_t b = __shfl_sync(0xffffffffu, ids_nxt, (k - win) & 31);
        return (k - win) < 32 ? a : b;
    };
    auto issue = [&](int k) {
        int32_t phys = block_id(k);
        const int st = k % GE::STAGES;
        if (lane == 0) {
            const uint32_t bar = bar0 + 8 * st;
            if (phys >= 0 && phys < p.num_blocks) {
                fence_proxy_async_smem();
                issue_stage<FP8>(ring + st * GE::STAGE, bar, &kmap, &vmap, (phys * p.hkv + g) * BS, l2pol);
            } else {
                flag(ST_BAD_BLOCK);
                mbar_arrive(bar);  // completes the phase without data
            }
        }
    };

    // ---- Q fragments (B operand of S^T = K . Q^T), kept in registers
    uint32_t qf[NT][8][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        // column -> (row offset, head of the group)
        const int gc = cg * CW + nt * 8 + gq;
        const int qi = MR ? gc / p.group : 0, hl = MR ? gc % p.group : gc;
        const bool hv = MR ? qi < nq : hl < p.group;
        const uint16_t *qr = p.q + ((size_t)(row + (hv ? qi : 0)) * p.hq + g * p.group + (hv ? hl : 0)) * D;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            if constexpr (!FP8) {
                uint32_t x0 = *reinterpret_cast<const uint32_t *>(qr + 16 * kk + 2 * cq);
                uint32_t x1 = *reinterpret_cast<const uint32_t *>(qr + 16 * kk + 2 * cq + 8);
                qf[nt][kk][0] = hv ? x0 : 0u;
                qf[nt][kk][1] = hv ? x1 : 0u;
            } else {
                uint2 x = *reinterpret_cast<const uint2 *>(qr + 16 * kk + 4 * cq);
                qf[nt][kk][0] = hv ? pack_f16(bf16_lo(x.x), bf16_hi(x.x)) : 0u;
                qf[nt][kk][1] = hv ? pack_f16(bf16_lo(x.y), bf16_hi(x.y)) : 0u;
            }
        }
    }
    // MR: keys visible to this lane's two columns of each n-tile (2 cq, 2 cq + 1):
    // row i sees keys < L - nq + i + 1; padding columns see everything (their Q
    // is zero and their output is never stored)
    int lim[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int qi = (cg * CW + nt * 8 + 2 * cq + e) / p.group;
            lim[nt][e] = (MR && qi < nq) ? L - nq + qi + 1 : L;
        }
    float sl = p.scale_log2;
    float vsc = 1.f;
    if constexpr (FP8) {
        sl *= __ldg(p.k_scale + g);
        vsc = __ldg(p.v_scale + g);
    }

    // ---- prologue
    const int pro = count < GE::STAGES ? count : GE::STAGES;
    for (int k = 0; k < pro; ++k) issue(k);

    float o[NT][8][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[nt][j][i] = 0.f;
    float m[NT][2], l[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
    }

    bool timed_out = false;
    int k = 0;
    for (; k < count; ++k) {
        const int st = k % GE::STAGES;
        const uint32_t par = (k / GE::STAGES) & 1;
        if (!mbar_wait_bounded(bar0 + 8 * st, par)) {
            timed_out = true;
            break;
        }
        const int32_t phys = block_id(k);
        const int blk = b0 + warp + k * WARPS;
        const int nvalid = min(BS, L - blk * BS);
        const uint32_t kb = ring + st * GE::STAGE;
        const uint32_t vb = kb + GE::TILE;
        if (phys >= 0 && phys < p.num_blocks) {
            // ---------------- S^T = K . Q^T
            float sacc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.f;
            if constexpr (!FP8) {
                const int mi = lane >> 3;
                const int tok = ((mi & 1) << 3) | (lane & 7);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int chunk = 2 * kk + (mi >> 1);
                    const uint32_t addr = kb + (chunk >> 3) * 2048 + tok * 128 +
                                          (((chunk & 7) ^ (tok & 7)) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16(sacc[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
                }
            } else {
                const int mi = lane >> 3;
                const int tok = ((mi & 1) << 3) | (lane & 7);
#pragma unroll
                for (int i2 = 0; i2 < 4; ++i2) {
                    const int chunk = 2 * i2 + (mi >> 1);
                    const uint32_t addr = kb + tok * 128 + ((chunk ^ (tok & 7)) << 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(addr, r0, r1, r2, r3);
                    // k step 2*i2 from chunks in r0/r1, step 2*i2+1 from r2/r3; the D
                    // order inside a step is permuted and Q's fragments match it
                    const uint32_t a0 = e4m3x2_to_f16x2(r0 & 0xffff), a2 = e4m3x2_to_f16x2(r0 >> 16);
                    const uint32_t a1 = e4m3x2_to_f16x2(r1 & 0xffff), a3 = e4m3x2_to_f16x2(r1 >> 16);
                    const uint32_t c0 = e4m3x2_to_f16x2(r2 & 0xffff), c2 = e4m3x2_to_f16x2(r2 >> 16);
                    const uint32_t c1 = e4m3x2_to_f16x2(r3 & 0xffff), c3 = e4m3x2_to_f16x2(r3 >> 16);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_f16(sacc[nt], a0, a1, a2, a3, qf[nt][2 * i2][0], qf[nt][2 * i2][1]);
                        mma_f16(sacc[nt], c0, c1, c2, c3, qf[nt][2 * i2 + 1][0], qf[nt][2 * i2 + 1][1]);
                    }
                }
            }
            // ---------------- online softmax (log2 domain), per head column
            uint32_t pb[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float x[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = gq + ((i >> 1) << 3);
                    const bool vis = MR ? blk * BS + t < lim[nt][i & 1] : t < nvalid;
                    x[i] = vis ? sacc[nt][i] * sl : -INFINITY;
                }
                float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
                // MR: a column may have seen no key yet (all masked): exponents are
                // taken against 0 then, so p = 0 and nothing becomes NaN
                const float r0 = (MR && mn0 == -INFINITY) ? 0.f : mn0;
                const float r1 = (MR && mn1 == -INFINITY) ? 0.f : mn1;
                const float al0 = ex2(m[nt][0] - r0), al1 = ex2(m[nt][1] - r1);
                m[nt][0] = mn0;
                m[nt][1] = mn1;
                const float p0 = ex2(x[0] - r0), p1 = ex2(x[1] - r1);
                const float p2 = ex2(x[2] - r0), p3 = ex2(x[3] - r1);
                l[nt][0] = l[nt][0] * al0 + (p0 + p2);
                l[nt][1] = l[nt][1] * al1 + (p1 + p3);
                // alpha is exactly 1 once a column's max stops growing: skipping the
                // multiplications then changes no bit
                if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        o[nt][j][0] *= al0;
                        o[nt][j][1] *= al1;
                        o[nt][j][2] *= al0;
                        o[nt][j][3] *= al1;
                    }
                }
                if constexpr (!FP8) {
                    pb[nt][0] = movmatrix_t(pack_bf16(p0, p1));
                    pb[nt][1] = movmatrix_t(pack_bf16(p2, p3));
                } else {
                    pb[nt][0] = movmatrix_t(pack_f16(p0, p1));
                    pb[nt][1] = movmatrix_t(pack_f16(p2, p3));
                }
            }
            // ---------------- O^T += V^T . P^T
            const bool tail = nvalid < BS;
            const uint32_t m01 = (2 * cq < nvalid ? 0x0000ffffu : 0u) | (2 * cq + 1 < nvalid ? 0xffff0000u : 0u);
            const uint32_t m23 = (2 * cq + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * cq + 9 < nvalid ? 0xffff0000u : 0u);
            if constexpr (!FP8) {
                const int mi = lane >> 3;
                const int tok = ((mi >> 1) << 3) | (lane & 7);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int chunk = 2 * j + (mi & 1);
                    const uint32_t addr = vb + (chunk >> 3) * 2048 + tok * 128 +
                                          (((chunk & 7) ^ (tok & 7)) << 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(addr, a0, a1, a2, a3);
                    if (tail) {
                        a0 &= m01;
                        a1 &= m01;
                        a2 &= m23;
                        a3 &= m23;
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_bf16(o[nt][j], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
            } else {
                uint32_t w[4][4];  // tokens 2c, 2c+1, 2c+8, 2c+9 ; 16 bytes of chunk gq each
#pragma unroll
                for (int ti = 0; ti < 4; ++ti) {
                    const int tok = 2 * cq + (ti & 1) + ((ti >> 1) << 3);
                    lds128(vb + tok * 128 + ((gq ^ (tok & 7)) << 4), w[ti][0], w[ti][1], w[ti][2], w[ti][3]);
                    if (tok >= nvalid) w[ti][0] = w[ti][1] = w[ti][2] = w[ti][3] = 0u;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t sel = (j & 1) ? 0x7362u : 0x5140u;
                    const uint32_t x01 = prmt(w[0][j >> 1], w[1][j >> 1], sel);
                    const uint32_t x23 = prmt(w[2][j >> 1], w[3][j >> 1], sel);
                    const uint32_t a0 = e4m3x2_to_f16x2(x01 & 0xffff), a1 = e4m3x2_to_f16x2(x01 >> 16);
                    const uint32_t a2 = e4m3x2_to_f16x2(x23 & 0xffff), a3 = e4m3x2_to_f16x2(x23 >> 16);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_f16(o[nt][j], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
            }
        }
        __syncwarp();
        // ---------------- refill this stage with the block STAGES ahead
        const int kn = k + GE::STAGES;
        if (kn < count) issue(kn);
        // advance the id window when the next refill would leave ids_cur/ids_nxt
        if (kn + 1 >= win + 64 && kn + 1 < count) {
            // kn + 1 is the next refill index; move the window forward by 32
            ids_cur = ids_nxt;
            win += 32;
            ids_nxt = load_ids(win + 32);
        }
    }
    if (timed_out) {
        flag(ST_TIMEOUT);
        // wait (bounded) for this warp's loads still in flight before leaving
        const int last = count < k + GE::STAGES ? count : k + GE::STAGES;
        for (int kk = k; kk < last; ++kk)
            (void)mbar_wait_bounded(bar0 + 8 * (kk % GE::STAGES), (kk / GE::STAGES) & 1);
    }

    // the LSE merge (next on the stream) may start scheduling now
    griddep_launch_dependents();
    // ---------------- merge the warps' partial softmax states
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float v = l[nt][e];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            l[nt][e] = v;
        }
    __syncthreads();  // every warp is done with its ring: reuse it for the merge
    constexpr int HL = NT * 8;
    float *sm_o = reinterpret_cast<float *>(smem);                 // [WARPS][HL][128]
    float *sm_m = sm_o + WARPS * HL * D;                           // [WARPS][HL]
    float *sm_l = sm_m + WARPS * HL;                               // [WARPS][HL]
    int *sm_to = reinterpret_cast<int *>(sm_l + WARPS * HL);       // [WARPS]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int hl = nt * 8 + 2 * cq + (i & 1);
                int d;
                if constexpr (!FP8) d = 16 * j + gq + ((i >> 1) << 3);
                else d = 16 * gq + 2 * j + (i >> 1);
                sm_o[(warp * HL + hl) * D + d] = o[nt][j][i];
            }
        if (gq == 0) {
            sm_m[warp * HL + nt * 8 + 2 * cq] = m[nt][0];
            sm_m[warp * HL + nt * 8 + 2 * cq + 1] = m[nt][1];
            sm_l[warp * HL + nt * 8 + 2 * cq] = l[nt][0];
            sm_l[warp * HL + nt * 8 + 2 * cq + 1] = l[nt][1];
        }
    }
    if (lane == 0) sm_to[warp] = timed_out ? 1 : 0;
    __syncthreads();
    const bool any_to = sm_to[0] | sm_to[1] | sm_to[2] | sm_to[3];
    const int G = p.group;
    const int ncols = MR ? min(CW, nq * G - cg * CW) : G;
    for (int idx = threadIdx.x; idx < ncols * D; idx += THREADS) {
        const int hl = idx / D, d = idx % D;      // column of this CTA
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) M = fmaxf(M, sm_m[w * HL + hl]);
        float Ls = 0.f, O = 0.f;
        if (M != -INFINITY && !any_to) {
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const float f = ex2(sm_m[w * HL + hl] - M);
                Ls += f * sm_l[w * HL + hl];
                O += f * sm_o[(w * HL + hl) * D + d];
            }
        }
        // MR: column -> (row of the chunk, head); partials are per row
        const int gc = cg * CW + hl;
        const int orow = MR ? row + gc / G : row, owi = MR ? orow : wi;
        const int h = g * G + (MR ? gc % G : hl);
        if (nsplit_s == 1) {
            p.out[((size_t)orow * p.hq + h) * D + d] = Ls > 0.f ? O * vsc / Ls : 0.f;
        } else {
            const size_t pi = ((size_t)owi * p.hq + h) * p.num_splits + split;
            p.part_o[pi * D + d] = O * vsc;
            if (d == 0) {
                p.part_ml[pi * 2] = (Ls > 0.f) ? M : -INFINITY;
                p.part_ml[pi * 2 + 1] = Ls;
            }
        }
    }
}

// Log-sum-exp merge of the split partitions: one warp per (sequence, q head),
// or per (row, q head) in the multi-row mode.
__global__ void __launch_bounds__(128) reduce_kernel(const DecodeParams p)
{
    // (the lengths were written before the decode kernel began, so they are read
    // before the wait for its partials)
    const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const bool per_row = p.col_groups > 0;
    if (wid >= (per_row ? p.total_rows : p.num_seqs) * p.hq) return;
    const int wi = wid / p.hq, h = wid % p.hq;   // wi: sequence, or row
    int row = wi, L;
    if (per_row) {
        // multi-row: the row's partitions are those of its sequence's whole context
        L = row_seq_len(p, row);
    } else {
        if (p.cu_q_lens) {
            int a = p.cu_q_lens[wi], b = p.cu_q_lens[wi + 1];
            if (b - a != 1 || a < 0 || b > p.total_rows) return;
            row = a;
        }
        L = p.context_lens[wi];
    }
    if (L < 1 || L > p.max_blocks * BS) return;
    const int nblk = (L + BS - 1) / BS;
    const int ns = (nblk + p.part_blocks - 1) / p.part_blocks;
    if (ns <= 1) return;
    griddep_wait();   // the partials come from the decode kernel just before
    const size_t base = ((size_t)wi * p.hq + h) * p.num_splits;
    const float4 r = lse_merge_warp(p.part_ml + base * 2, p.part_o + base * D, ns, lane);
    reinterpret_cast<float4 *>(p.out + ((size_t)row * p.hq + h) * D)[lane] = r;
}

// ---- device code end (hashed with the ncu counters of profiles/)
template <bool FP8, int NT, bool MR>
cudaError_t launch_one(const CUtensorMap &km, const CUtensorMap &vm, const DecodeParams &p,
                       cudaStream_t st, bool pdl)
{
    const cudaError_t e = pkv_host::ensure_dynamic_smem<decode_kernel<FP8, NT, MR>>(Geo<FP8>::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_splits * (MR ? p.col_groups : 1), p.hkv, p.num_seqs);
    return pkv_host::launch_ex(decode_kernel<FP8, NT, MR>, grid, dim3(THREADS), Geo<FP8>::SMEM, st, pdl, km, vm, p);
}

template <bool FP8>
cudaError_t launch_for(const CUtensorMap &km, const CUtensorMap &vm, const DecodeParams &p, int nt,
                       cudaStream_t st, bool pdl)
{
    if (p.col_groups > 0)
        return nt == 2 ? launch_one<FP8, 2, true>(km, vm, p, st, pdl) : launch_one<FP8, 1, true>(km, vm, p, st, pdl);
    return nt == 2 ? launch_one<FP8, 2, false>(km, vm, p, st, pdl) : launch_one<FP8, 1, false>(km, vm, p, st, pdl);
}

}  // namespace

// ---------------------------------------------------------------- host side
namespace pkv_decode {

// Chooses the partition length (blocks) and the number of partitions.  Auto
// mode lengthens partitions with the longest context (64 blocks up to 8K
// tokens, 128 up to 64K, 256 beyond): measured on GB300 this keeps enough
// CTAs for the short batches while long ones pay less per-CTA ramp-up and
// partial-merge traffic.  A batch with few (sequence, KV head) pairs --
// estimated as num_seqs x hq / 8 -- gets shorter partitions (down to 16
// blocks, four per warp) so that the grid holds about SMALL_TARGET CTAs: a
// handful of sequences is otherwise latency-bound on a few warps each.
// Measured on the 4-sequence tiny batch: 47 us with one partition, 16 us with
// 64-block partitions, 14 us with 16-block ones, 24 us with 4-block ones
// (the merge and the CTAs' fixed costs take over).
constexpr int64_t SMALL_TARGET = 2 * 3 * 152;

void plan_splits(int32_t max_blocks, int32_t num_splits, int32_t num_seqs, int32_t hq, int32_t *part_blocks,
                 int32_t *splits)
{
    int32_t auto_part = max_blocks <= 512 ? 64 : (max_blocks <= 4096 ? 128 : 256);
    const int64_t pairs = (int64_t)std::max(1, num_seqs) * std::max(1, hq / 8);
    const int64_t want = ((int64_t)max_blocks * pairs + SMALL_TARGET - 1) / SMALL_TARGET;
    auto_part = (int32_t)std::min<int64_t>(auto_part, std::max<int64_t>(16, want));
    int32_t s = num_splits > 0 ? num_splits : (max_blocks + auto_part - 1) / auto_part;
    s = std::max(1, std::min(s, max_blocks));
    int32_t pb = (max_blocks + s - 1) / s;
    *part_blocks = pb;
    *splits = (max_blocks + pb - 1) / pb;
}

static size_t partial_bytes(int32_t problems, int32_t hq, int32_t splits)
{
    if (splits <= 1) return 0;
    size_t n = (size_t)problems * hq * splits;
    size_t bytes = n * D * sizeof(float) + n * 2 * sizeof(float);
    return (bytes + 255) & ~size_t(255);
}

size_t workspace_bytes(int32_t num_seqs, int32_t hq, int32_t max_blocks, int32_t num_splits)
{
    if (num_seqs < 1 || hq < 1 || max_blocks < 1) return 0;
    int32_t pb, s;
    plan_splits(max_blocks, num_splits, num_seqs, hq, &pb, &s);
    return partial_bytes(num_seqs, hq, s);
}

// Multi-row mode: the decode partitioning, partials per row.
size_t workspace_bytes_multi(int32_t total_rows, int32_t num_seqs, int32_t hq, int32_t max_blocks,
                             int32_t num_splits)
{
    if (total_rows < 1 || hq < 1 || max_blocks < 1) return 0;
    int32_t pb, s;
    plan_splits(max_blocks, num_splits, num_seqs, hq, &pb, &s);
    return partial_bytes(total_rows, hq, s);
}

bool make_maps(const void *k_cache, const void *v_cache, int32_t num_blocks, int32_t hkv,
               kv_dtype dt, CUtensorMap *km, CUtensorMap *vm)
{
    const uint64_t rows = (uint64_t)num_blocks * hkv * BS;
    if (dt == KV_BF16)
        return pkv_host::encode_tmap_2d(km, k_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, rows, D * 2,
                                        64, BS, CU_TENSOR_MAP_SWIZZLE_128B) &&
               pkv_host::encode_tmap_2d(vm, v_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, rows, D * 2,
                                        64, BS, CU_TENSOR_MAP_SWIZZLE_128B);
    return pkv_host::encode_tmap_2d(km, k_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, D, rows, D, D, BS,
                                    CU_TENSOR_MAP_SWIZZLE_128B) &&
           pkv_host::encode_tmap_2d(vm, v_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, D, rows, D, D, BS,
                                    CU_TENSOR_MAP_SWIZZLE_128B);
}

// Validates host-visible arguments shared by decode and the decode rows of a
// mixed batch, then launches decode (+ reduce), with programmatic dependent
// launch when pdl is set (see pkv_host::launch_ex).  Needing cu_q_lens:
//  multi_q_len > 0 multi-row mode: every sequence's rows (at most multi_q_len)
//                  are covered by column groups of one CTA per KV tile stream.
// corun (with pdl): launched right behind a mixed batch's chunk-prefill kernel,
// whose inputs and these were all written before that call began; only the
// grid's first CTA waits for the chunk kernel, the others start beside it.
kv_status run(float *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens,
              const int32_t *cu_q_lens, int32_t total_rows, int32_t num_seqs, int32_t hq, int32_t hkv,
              int32_t num_blocks, float scale, kv_dtype dt, const float *k_scale, const float *v_scale,
              int32_t num_splits, void *workspace, size_t workspace_bytes_given, cudaStream_t st,
              int32_t multi_q_len, bool pdl, bool corun = false)
{
    const bool multi = multi_q_len > 0;
    if (multi && (!cu_q_lens || total_rows < 0)) return KV_ERR_INVALID;
    if (multi && total_rows == 0) return KV_OK;
    if (num_seqs == 0) return KV_OK;
    if (num_seqs < 0 || hq < 1 || hkv < 1 || num_blocks < 1 || max_blocks < 1) return KV_ERR_INVALID;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return KV_ERR_INVALID;
    if (hq % hkv) return KV_ERR_INVALID;
    const int32_t G = hq / hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return KV_ERR_UNSUPPORTED;
    if (dt != KV_BF16 && dt != KV_FP8_E4M3) return KV_ERR_UNSUPPORTED;
    if (dt == KV_FP8_E4M3 && (!k_scale || !v_scale)) return KV_ERR_INVALID;
    if (!(scale > 0.f) || num_seqs > 65535 || hkv > 65535) return KV_ERR_INVALID;
    if ((int64_t)num_blocks * hkv * BS > INT32_MAX) return KV_ERR_UNSUPPORTED;
    if (!pkv_host::aligned(k_cache, 16) || !pkv_host::aligned(v_cache, 16) ||
        !pkv_host::aligned(q, 16) || !pkv_host::aligned(out, 16))
        return KV_ERR_INVALID;
    DecodeParams p{};
    p.out = out;
    p.q = static_cast<const uint16_t *>(q);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.cu_q_lens = cu_q_lens;
    p.total_rows = cu_q_lens ? total_rows : num_seqs;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.max_blocks = max_blocks;
    p.num_seqs = num_seqs;
    p.hq = hq;
    p.hkv = hkv;
    p.group = G;
    p.num_blocks = num_blocks;
    p.scale_log2 = scale * LOG2E;
    p.corun = corun && pdl ? 1 : 0;
    plan_splits(max_blocks, num_splits, num_seqs, hq, &p.part_blocks, &p.num_splits);
    // columns of one sequence and KV head: its rows x the group's heads
    const int64_t cols = multi ? (int64_t)multi_q_len * G : G;
    const int nt = cols > 8 ? 2 : 1;
    if (multi) {
        const int64_t groups = (cols + 8 * nt - 1) / (8 * nt);
        if (groups * p.num_splits > INT32_MAX) return KV_ERR_UNSUPPORTED;
        p.col_groups = (int)groups;
    }
    if (p.num_splits > 65535) return KV_ERR_UNSUPPORTED;
    const int32_t problems = multi ? total_rows : num_seqs;
    const size_t need = multi ? workspace_bytes_multi(total_rows, num_seqs, hq, max_blocks, num_splits)
                              : workspace_bytes(num_seqs, hq, max_blocks, num_splits);
    if (need) {
        if (!workspace || workspace_bytes_given < need || !pkv_host::aligned(workspace, 256))
            return KV_ERR_INVALID;
        const size_t n = (size_t)problems * hq * p.num_splits;
        p.part_o = static_cast<float *>(workspace);
        p.part_ml = p.part_o + n * D;
    }
    CUtensorMap km, vm;
    if (!make_maps(k_cache, v_cache, num_blocks, hkv, dt, &km, &vm)) return KV_ERR_CUDA;
    const cudaError_t e =
        dt == KV_BF16 ? launch_for<false>(km, vm, p, nt, st, pdl) : launch_for<true>(km, vm, p, nt, st, pdl);
    if (e != cudaSuccess) return KV_ERR_CUDA;
    if (p.num_splits > 1) {
        const int64_t warps = (int64_t)problems * hq;
        if (pkv_host::launch_ex(reduce_kernel, dim3((unsigned)((warps + 3) / 4)), dim3(128), 0, st, pdl, p) !=
            cudaSuccess)
            return KV_ERR_CUDA;
    }
    return KV_OK;
}

uint32_t take_status()
{
    uint32_t v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_status, &z, sizeof z);
    return v;
}

}  // namespace pkv_decode

extern "C" {

size_t paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                      int32_t max_blocks_per_seq, int32_t num_splits)
{
    return pkv_decode::workspace_bytes(num_seqs, num_q_heads, max_blocks_per_seq, num_splits);
}

kv_status paged_attention_decode(float *out, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 int32_t max_blocks_per_seq, const int32_t *context_lens,
                                 int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t num_blocks, float scale, kv_dtype dtype,
                                 const float *k_scale, const float *v_scale, int32_t num_splits,
                                 void *workspace, size_t workspace_bytes, void *stream)
{
    PKV_NVTX_RANGE("paged_attention_decode");
    return pkv_decode::run(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                           nullptr, num_seqs, num_seqs, num_q_heads, num_kv_heads, num_blocks, scale, dtype,
                           k_scale, v_scale, num_splits, workspace, workspace_bytes,
                           static_cast<cudaStream_t>(stream), 0, true);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention:
// code running inside a memory pool or allocator hook of its own, a runtime
// that forbids allocation once it has started serving, or a host that links
// this library without any allocator.  For them the split-KV partials live in
// one file-scope device array instead of a caller workspace.  Its size is
// fixed (STATIC_SCRATCH_BYTES); every GPU that loads the library holds it until
// the process exits.  Calls whose partials would not fit are refused with
// KV_ERR_UNSUPPORTED.  All calls share the array, so calls that overlap on the
// GPU (different streams, or different host threads on one device) race on it;
// serialise them.  Nothing in it needs to start at zero: every partial that is
// read was written earlier in the same call.  The first call on a device looks
// up the array's device address (cudaGetSymbolAddress, with that device
// current); make that first call before any stream capture.  The address is
// remembered together with the device's current context, so a call after a
// device reset (a new primary context, a new copy of the array) looks it up
// again instead of using the old one; such a call again belongs outside any
// capture.
namespace {
constexpr size_t STATIC_SCRATCH_BYTES = size_t(32) << 20;
static __device__ __align__(256) uint8_t g_static_scratch[STATIC_SCRATCH_BYTES];
constexpr int MAX_DEVICES = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[MAX_DEVICES] = {};
void *g_scratch_ctx[MAX_DEVICES] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

CtxGetCurrentFn get_ctx_current()
{
    static CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    return fn;
}

kv_status static_scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KV_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES) return KV_ERR_UNSUPPORTED;
    CtxGetCurrentFn ctx_fn = get_ctx_current();
    if (!ctx_fn) return KV_ERR_CUDA;
    // null until the runtime has set up this device's primary context
    CUcontext ctx = nullptr;
    if (ctx_fn(&ctx) != CUDA_SUCCESS) return KV_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_scratch_mu);
    if (!g_scratch_addr[dev] || !ctx || g_scratch_ctx[dev] != static_cast<void *>(ctx)) {
        void *p = nullptr;
        // the lookup sets up the primary context when it is not yet current
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return KV_ERR_CUDA;
        if (ctx_fn(&ctx) != CUDA_SUCCESS) return KV_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return KV_OK;
}
}  // namespace

extern "C" {

size_t paged_attention_decode_static_scratch_bytes(void) { return STATIC_SCRATCH_BYTES; }

kv_status paged_attention_decode_static_scratch(float *out, const void *q, const void *k_cache,
                                                const void *v_cache, const int32_t *block_tables,
                                                int32_t max_blocks_per_seq, const int32_t *context_lens,
                                                int32_t num_seqs, int32_t num_q_heads,
                                                int32_t num_kv_heads, int32_t num_blocks, float scale,
                                                kv_dtype dtype, const float *k_scale,
                                                const float *v_scale, int32_t num_splits, void *stream)
{
    PKV_NVTX_RANGE("paged_attention_decode_static_scratch");
    const size_t need = pkv_decode::workspace_bytes(num_seqs, num_q_heads, max_blocks_per_seq, num_splits);
    if (need > STATIC_SCRATCH_BYTES) return KV_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (need) {
        kv_status st = static_scratch_address(&scratch);
        if (st != KV_OK) return st;
    }
    return pkv_decode::run(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                           nullptr, num_seqs, num_seqs, num_q_heads, num_kv_heads, num_blocks, scale, dtype,
                           k_scale, v_scale, num_splits, scratch, need ? STATIC_SCRATCH_BYTES : 0,
                           static_cast<cudaStream_t>(stream), 0, true);
}

}  // extern "C"
