// attn_prefill_chunk: argument checks of the C ABI; the work runs in prefill_tc.cu.
//
// Source: chunked prefill of long audio prompts, 4096 tokens per scheduling step, each chunk
// attending to the KV cache of the earlier chunks plus its own tokens ("Optimizing ASR
// Models to Transcribe 90-Minute Multi-Speaker Audio", "Chunked Prefill for Long Audio";
// "MOSS-Transcribe-Diarize" cookbook, "Inference Pipeline").
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_common.cuh"

namespace pa {
pa_status launch_prefill_tc(int32_t hkv, const void* q, int32_t total_q, const int32_t* cu_q_lens,
                            const void* k_pool, const void* v_pool, int64_t num_pages,
                            const int32_t* block_table, int32_t bt_stride,
                            const int32_t* seq_lens, int32_t batch, int32_t max_q_len,
                            float softmax_scale, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, int32_t* status, cudaStream_t stream,
                            int32_t max_ctas);
size_t prefill_workspace_bytes(int batch);

namespace {
pa_status prefill_call(pa_dims dims, const void* q, const int32_t* cu_q_lens, int32_t total_q,
                       const void* k_pool, const void* v_pool, int64_t num_pages,
                       const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                       int32_t batch, int32_t max_q_len, int32_t max_seq_len,
                       float softmax_scale, void* out, float* lse, void* workspace,
                       size_t workspace_bytes, int32_t* status, pa_stream_t stream,
                       int32_t max_ctas) {
  if (!gqa_dims_supported(dims)) return PA_ERR_UNSUPPORTED;
  if (total_q < 0 || batch < 0 || bt_stride <= 0 || num_pages <= 0 || max_q_len < 0 ||
      max_seq_len < 0 || max_seq_len > 131072 || max_q_len > max_seq_len ||
      !(softmax_scale > 0.f) || !(softmax_scale < 1e30f) || max_ctas < 0)
    return PA_ERR_INVALID_ARG;
  if (batch == 0 || max_q_len == 0 || total_q == 0) return PA_OK;
  if (!q || !cu_q_lens || !k_pool || !v_pool || !block_table || !seq_lens || !out)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pool) |
       reinterpret_cast<uintptr_t>(v_pool) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return PA_ERR_INVALID_ARG;
  return launch_prefill_tc(dims.num_kv_heads, q, total_q, cu_q_lens, k_pool, v_pool, num_pages,
                           block_table, bt_stride, seq_lens, batch, max_q_len, softmax_scale, out,
                           lse, workspace, workspace_bytes, status,
                           reinterpret_cast<cudaStream_t>(stream), max_ctas);
}
}  // namespace
}  // namespace pa

extern "C" size_t pa_prefill_workspace_size(pa_dims dims, int32_t batch, int32_t max_q_len,
                                            int32_t max_seq_len) {
  (void)dims; (void)max_q_len; (void)max_seq_len;
  return pa::prefill_workspace_bytes(batch);
}

extern "C" pa_status attn_prefill_chunk(pa_dims dims, const void* q, const int32_t* cu_q_lens,
                                        int32_t total_q, const void* k_pool, const void* v_pool,
                                        int64_t num_pages, const int32_t* block_table,
                                        int32_t bt_stride, const int32_t* seq_lens,
                                        int32_t batch, int32_t max_q_len, int32_t max_seq_len,
                                        float softmax_scale, void* out, float* lse,
                                        void* workspace, size_t workspace_bytes,
                                        int32_t* status, pa_stream_t stream) {
  return pa::prefill_call(dims, q, cu_q_lens, total_q, k_pool, v_pool, num_pages, block_table,
                          bt_stride, seq_lens, batch, max_q_len, max_seq_len, softmax_scale, out,
                          lse, workspace, workspace_bytes, status, stream, 0);
}

extern "C" pa_status attn_prefill_chunk_ex(pa_dims dims, const void* q, const int32_t* cu_q_lens,
                                           int32_t total_q, const void* k_pool,
                                           const void* v_pool, int64_t num_pages,
                                           const int32_t* block_table, int32_t bt_stride,
                                           const int32_t* seq_lens, int32_t batch,
                                           int32_t max_q_len, int32_t max_seq_len,
                                           float softmax_scale, void* out, float* lse,
                                           void* workspace, size_t workspace_bytes,
                                           int32_t* status, pa_stream_t stream,
                                           const pa_launch_opts* opts) {
  return pa::prefill_call(dims, q, cu_q_lens, total_q, k_pool, v_pool, num_pages, block_table,
                          bt_stride, seq_lens, batch, max_q_len, max_seq_len, softmax_scale, out,
                          lse, workspace, workspace_bytes, status, stream,
                          opts != nullptr ? opts->max_ctas : 0);
}
