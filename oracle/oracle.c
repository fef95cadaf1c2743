/*
 * oracle.c -- plain fp64 CPU oracle for paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so and is
 * loaded only by tests/, by __graft_entry__.smoke() and by the cpu-baseline leg
 * of bench.py.  The CUDA library never links, loads or calls it, and it shares
 * no code, header or table with the CUDA path.
 *
 * What it computes, and where the pages define it:
 *
 *  - The paged KV cache: K/V of every token live in fixed 16-token physical
 *    blocks; a per-sequence block table maps logical block t/16 to a physical
 *    block, offset t%16 inside it.
 *      ["PagedAttention, chunked prefill, and the launch that cascades",
 *       section "PagedAttention: an OS idea, not an ML one"];
 *      ["M.65 Inference serving", PagedAttention block management (a)-(d)].
 *  - Attention itself is unchanged by paging: the paged result equals the
 *    textbook result on contiguous K/V.
 *      ["Waste, and three ways to reclaim it" (Document 10 - Quick learn),
 *       section "PagedAttention - operating-system virtual memory, applied to
 *       attention", "And note what it does not change"].
 *    So the oracle gathers each sequence's blocks into contiguous K/V and runs
 *    textbook softmax attention: z_t = scale * q.k_t, w = softmax(z),
 *    o = sum_t w_t v_t, all in fp64.
 *  - GQA: query head h reads KV head floor(h / G), G = Hq / Hkv (the
 *    repeat_interleave broadcast).
 *      ["PagedAttention, chunked prefill, ...", section "Kernel engineering"].
 *  - Chunked prefill: a chunk of n query tokens of a sequence of length L
 *    occupies positions L-n .. L-1; query i attends keys 0 .. L-n+i.  Decode is
 *    n = 1.  ["PagedAttention, chunked prefill, ...", section "Serving
 *    systems"]; ["M.65 Inference serving", prefill vs decode (e)].
 *  - fp8 cache: one byte per element, E4M3 (1 sign, 4 exponent bits with bias
 *    7, 3 mantissa bits, no infinities, max finite 448).  ["Waste, and three
 *    ways to reclaim it", section "Quantising the cache"]; ["M.65 Inference
 *    serving", quantisation (b), (d)].  Encoding divides by the per-head scale
 *    in fp32 and rounds to nearest-even, clamping to +-448 (satfinite).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fast-math), so
 * every operation is an IEEE operation in program order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BF16 0
#define ORACLE_FP8 1

/* ---------------------------------------------------------------- formats */

double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* E4M3 decode from the format definition. */
double oracle_e4m3_to_f64(uint8_t q)
{
    int s = q >> 7, e = (q >> 3) & 0xF, m = q & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);          /* (m/8) * 2^(1-7) */
    else v = ldexp(8.0 + (double)m, e - 10);       /* (1+m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* E4M3 encode of an fp32 value: round to nearest, ties to even, clamp to the
 * largest finite magnitude 448 (anything at or above 448 maps to 448, which is
 * what rounding gives up to 464 and saturation gives beyond); NaN -> 0x7F. */
uint8_t oracle_e4m3_from_f32(float xf)
{
    double x = (double)xf;                 /* exact */
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    double step;
    if (a < ldexp(1.0, -6)) {
        step = ldexp(1.0, -9);             /* subnormal spacing */
    } else {
        int ex;
        frexp(a, &ex);                     /* a in [2^(ex-1), 2^ex) */
        step = ldexp(1.0, (ex - 1) - 3);   /* 3 mantissa bits */
    }
    double r = rint(a / step);             /* a/step exact; rint = nearest-even */
    double v = r * step;
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) return sign | (uint8_t)r;
    int ex;
    frexp(v, &ex);
    int e = ex - 1 + 7;
    int m = (int)(ldexp(v, -(ex - 1)) * 8.0) - 8;
    return sign | (uint8_t)(e << 3) | (uint8_t)m;
}

/* Bulk encode, used by the encoder's exhaustive check: out[i] = e4m3(x[i]). */
void oracle_e4m3_encode_array(const float *x, uint8_t *out, int64_t n)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_from_f32(x[i]);
}

/* ------------------------------------------------------------ cache write */

/* Cache layout: cache[block][kv_head][offset][d]; element bf16 (uint16 bits)
 * or e4m3 (uint8).  Token t with slot = slot_mapping[t] goes to block
 * slot / block_size, offset slot % block_size.  slot < 0 means "skip".
 * Returns 0, or -1 if a slot points outside the pool. */
int oracle_reshape_and_cache(const uint16_t *k, const uint16_t *v, void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, int T, int Hkv, int D, int block_size,
                             int64_t num_blocks, int dtype, const float *k_scale,
                             const float *v_scale)
{
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t blk = slot / block_size, off = slot % block_size;
        if (blk >= num_blocks) return -1;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t src = ((int64_t)t * Hkv + h) * D + d;
                int64_t dst = ((blk * Hkv + h) * block_size + off) * D + d;
                if (dtype == ORACLE_BF16) {
                    ((uint16_t *)k_cache)[dst] = k[src];
                    ((uint16_t *)v_cache)[dst] = v[src];
                } else {
                    float kx = bf16_to_f32(k[src]) / k_scale[h];   /* IEEE fp32 divide */
                    float vx = bf16_to_f32(v[src]) / v_scale[h];
                    ((uint8_t *)k_cache)[dst] = oracle_e4m3_from_f32(kx);
                    ((uint8_t *)v_cache)[dst] = oracle_e4m3_from_f32(vx);
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------- textbook attention */

/* One query row against contiguous K/V of one head.
 * q[D], k[L][kstride], v[L][kstride] (fp64); attends keys 0..p inclusive.
 * z_t = scale * sum_d q_d k_td ; w_t = exp(z_t - max z) / sum exp(z - max z) ;
 * o_d = sum_t w_t v_td.  z is scratch of length >= p+1. */
static void attend_row(double *o, const double *q, const double *k, const double *v,
                       int64_t kstride, int64_t p, int D, double scale, double *z)
{
    double zmax = -INFINITY;
    for (int64_t t = 0; t <= p; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[d] * k[t * kstride + d];
        z[t] = scale * acc;
        if (z[t] > zmax) zmax = z[t];
    }
    double denom = 0.0;
    for (int64_t t = 0; t <= p; ++t) {
        z[t] = exp(z[t] - zmax);
        denom += z[t];
    }
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t t = 0; t <= p; ++t) {
        double w = z[t] / denom;
        for (int d = 0; d < D; ++d) o[d] += w * v[t * kstride + d];
    }
}

/* Contiguous attention for one sequence.
 * q[n][Hq][D], k/v[L][Hkv][D], out[n][Hq][D], all fp64.  Query i sits at
 * position L-n+i and attends keys 0..L-n+i; head h reads KV head h/(Hq/Hkv).
 * Returns 0, or -1 on bad sizes. */
int oracle_contiguous_attention(double *out, const double *q, const double *k, const double *v,
                                int n, int64_t L, int Hq, int Hkv, int D, double scale,
                                int nthreads)
{
    if (n < 1 || L < n || Hkv < 1 || Hq % Hkv != 0) return -1;
    int G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    int bad = 0;
    #pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)L);
        if (!z) {
            #pragma omp atomic write
            bad = 1;
        } else {
            #pragma omp for schedule(dynamic, 1) collapse(2)
            for (int i = 0; i < n; ++i) {
                for (int h = 0; h < Hq; ++h) {
                    int g = h / G;
                    int64_t p = L - n + i;
                    attend_row(out + ((int64_t)i * Hq + h) * D, q + ((int64_t)i * Hq + h) * D,
                               k + (int64_t)g * D, v + (int64_t)g * D, (int64_t)Hkv * D, p, D,
                               scale, z);
                }
            }
            free(z);
        }
    }
    return bad ? -1 : 0;
}

/* Paged attention over a batch.
 *  out          fp64 [R][Hq][D], R = total query rows
 *  q            bf16 bits [R][Hq][D]
 *  k/v_cache    [num_blocks][Hkv][block_size][D], bf16 bits or e4m3 bytes
 *  k/v_scale    [Hkv] fp32 (fp8 only): stored value * scale is the key/value
 *  block_tables int32 [B][max_blocks]
 *  context_lens int32 [B] (tokens of the sequence, the query chunk included)
 *  cu_q_lens    int32 [B+1] or NULL (NULL: one query row per sequence)
 * For each sequence and KV head the blocks are gathered into contiguous K/V
 * (logical token t from block_tables[s][t/bs] at offset t%bs), then textbook
 * attention is computed for every query head of the group.
 * Returns 0, -1 on bad sizes, -2 if a table entry is outside the pool. */
int oracle_paged_attention(double *out, const uint16_t *q, const void *k_cache,
                           const void *v_cache, int dtype, const float *k_scale,
                           const float *v_scale, const int32_t *block_tables, int max_blocks,
                           const int32_t *context_lens, const int32_t *cu_q_lens, int B, int Hq,
                           int Hkv, int D, int block_size, int64_t num_blocks, double scale,
                           int nthreads)
{
    if (B < 0 || Hkv < 1 || Hq % Hkv != 0 || block_size < 1) return -1;
    int G = Hq / Hkv;
    for (int s = 0; s < B; ++s) {
        int n = cu_q_lens ? cu_q_lens[s + 1] - cu_q_lens[s] : 1;
        int64_t L = context_lens[s];
        /* a sequence may contribute no query rows (n = 0): it has no output */
        if (n < 0 || L < 1 || L < n || L > (int64_t)max_blocks * block_size) return -1;
        for (int64_t j = 0; j < (L + block_size - 1) / block_size; ++j) {
            int32_t b = block_tables[(int64_t)s * max_blocks + j];
            if (b < 0 || b >= num_blocks) return -2;
        }
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    int bad = 0;
    #pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int s = 0; s < B; ++s) {
        for (int g = 0; g < Hkv; ++g) {
            int n = cu_q_lens ? cu_q_lens[s + 1] - cu_q_lens[s] : 1;
            int64_t row0 = cu_q_lens ? cu_q_lens[s] : s;
            int64_t L = context_lens[s];
            double *K = (double *)malloc(sizeof(double) * (size_t)(L * D));
            double *V = (double *)malloc(sizeof(double) * (size_t)(L * D));
            double *z = (double *)malloc(sizeof(double) * (size_t)L);
            double *qd = (double *)malloc(sizeof(double) * (size_t)D);
            if (!K || !V || !z || !qd) {
                #pragma omp atomic write
                bad = 1;
            } else {
                /* gather through the block table */
                for (int64_t t = 0; t < L; ++t) {
                    int64_t blk = block_tables[(int64_t)s * max_blocks + t / block_size];
                    int64_t off = t % block_size;
                    int64_t base = ((blk * Hkv + g) * block_size + off) * D;
                    for (int d = 0; d < D; ++d) {
                        if (dtype == ORACLE_BF16) {
                            K[t * D + d] = oracle_bf16_to_f64(((const uint16_t *)k_cache)[base + d]);
                            V[t * D + d] = oracle_bf16_to_f64(((const uint16_t *)v_cache)[base + d]);
                        } else {
                            K[t * D + d] = oracle_e4m3_to_f64(((const uint8_t *)k_cache)[base + d]) *
                                           (double)k_scale[g];
                            V[t * D + d] = oracle_e4m3_to_f64(((const uint8_t *)v_cache)[base + d]) *
                                           (double)v_scale[g];
                        }
                    }
                }
                for (int hh = 0; hh < G; ++hh) {
                    int h = g * G + hh;
                    for (int i = 0; i < n; ++i) {
                        const uint16_t *qs = q + ((row0 + i) * Hq + h) * D;
                        for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(qs[d]);
                        attend_row(out + ((row0 + i) * Hq + h) * D, qd, K, V, D, L - n + i, D,
                                   scale, z);
                    }
                }
            }
            free(K);
            free(V);
            free(z);
            free(qd);
        }
    }
    return bad ? -1 : 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
