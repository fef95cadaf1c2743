// prefill.cu -- paged attention over mixed chunked-prefill / decode batches.
// (work in progress: decode rows only)
#include "common.cuh"

namespace {
__device__ uint32_t g_status;
}

namespace pkv_decode {
kv_status run(float *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, int32_t max_blocks, const int32_t *context_lens,
              const int32_t *cu_q_lens, int32_t total_rows, int32_t num_seqs, int32_t hq, int32_t hkv,
              int32_t num_blocks, float scale, kv_dtype dt, const float *k_scale, const float *v_scale,
              int32_t num_splits, void *workspace, size_t workspace_bytes_given, cudaStream_t st);
size_t workspace_bytes(int32_t num_seqs, int32_t hq, int32_t max_blocks, int32_t num_splits);
}  // namespace pkv_decode

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
    (void)total_q_tokens; (void)max_q_len; (void)num_kv_heads;
    return pkv_decode::workspace_bytes(num_seqs, num_q_heads, max_blocks_per_seq, num_splits);
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
    if (!cu_q_lens || total_q_tokens < 0 || max_q_len < 1) return KV_ERR_INVALID;
    if (max_q_len > 1) return KV_ERR_UNSUPPORTED;
    return pkv_decode::run(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                           cu_q_lens, total_q_tokens, num_seqs, num_q_heads, num_kv_heads, num_blocks, scale, dtype,
                           k_scale, v_scale, num_splits, workspace, workspace_bytes,
                           static_cast<cudaStream_t>(stream));
}

}  // extern "C"
