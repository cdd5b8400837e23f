// kv_append_paged: scatter the K/V rows of new tokens into their page slots (sm_103a).
//
// Source: prefill "builds its KV cache" and each decode step extends it by one token
// ("Optimizing ASR Models to Transcribe 90-Minute Multi-Speaker Audio", "ASR Model Primer";
// 4096-token chunks per step, "Chunked Prefill for Long Audio").
//
// One CTA per new token: 16 * Hkv threads move its K row (Hkv heads x 128 dims x 2 B; 2 KB for
// the decoder's 8 KV heads) and as many its V row, 16 bytes each, so every warp writes 512
// contiguous bytes of the destination slot. Bit-exact copy; the slot address comes from the
// block table.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kChunksPerHead = kHeadDim * 2 / 16;  // 16-byte pieces of one head's row (16)

struct AppendParams {
  int32_t row_chunks;  // 16-byte pieces of one token row: 16 * Hkv
  const uint8_t* k_new;
  const uint8_t* v_new;
  const int32_t* cu_new_lens;
  const int32_t* start_pos;
  int32_t batch;
  const int32_t* block_table;
  int32_t bt_stride;
  uint8_t* k_pool;
  uint8_t* v_pool;
  int64_t num_pages;
  int32_t* status;
};

__global__ void __launch_bounds__(2 * kChunksPerHead * kHkv) kv_append_kernel(const AppendParams p) {
  const int t = blockIdx.x;
  const int packed = p.cu_new_lens[p.batch];
  // more packed rows than the call's total_new: the rows past it would be lost silently
  if (t == 0 && threadIdx.x == 0 && packed > static_cast<int>(gridDim.x))
    flag_error(p.status, PA_DEV_ERR_LENGTH);
  if (t >= packed) return;  // rows past the packed total are not tokens
  int lo = 0, hi = p.batch;                  // largest b with cu[b] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.cu_new_lens[mid] <= t) lo = mid; else hi = mid;
  }
  const int b = lo;
  const bool leader = threadIdx.x == 0;
  if (t < p.cu_new_lens[b] || t >= p.cu_new_lens[b + 1]) {
    if (leader) flag_error(p.status, PA_DEV_ERR_LENGTH);
    return;
  }
  const int pos = p.start_pos[b] + (t - p.cu_new_lens[b]);
  if (pos < 0 || pos >= p.bt_stride * kPage) {
    if (leader) flag_error(p.status, PA_DEV_ERR_LENGTH);
    return;
  }
  const int page = p.block_table[static_cast<int64_t>(b) * p.bt_stride + pos / kPage];
  if (page < 0 || page >= p.num_pages) {
    if (leader) flag_error(p.status, PA_DEV_ERR_PAGE_OOB);
    return;
  }
  const int which = threadIdx.x / p.row_chunks;  // 0 = K, 1 = V
  const int chunk = threadIdx.x - which * p.row_chunks;
  const int64_t row_bytes = p.row_chunks * 16;
  const uint8_t* src = (which ? p.v_new : p.k_new) + static_cast<int64_t>(t) * row_bytes + chunk * 16;
  uint8_t* dst = (which ? p.v_pool : p.k_pool) +
                 (static_cast<int64_t>(page) * kPage + pos % kPage) * row_bytes + chunk * 16;
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
}

}  // namespace
}  // namespace pa

extern "C" pa_status kv_append_paged(pa_dims dims, const void* k_new, const void* v_new,
                                     int32_t total_new, const int32_t* cu_new_lens,
                                     const int32_t* start_pos, int32_t batch,
                                     const int32_t* block_table, int32_t bt_stride, void* k_pool,
                                     void* v_pool, int64_t num_pages, int32_t* status,
                                     pa_stream_t stream) {
  using namespace pa;
  if (!gqa_dims_supported(dims)) return PA_ERR_UNSUPPORTED;
  if (total_new < 0 || batch < 0 || bt_stride <= 0 || num_pages <= 0) return PA_ERR_INVALID_ARG;
  if (total_new == 0 || batch == 0) return PA_OK;
  if (!k_new || !v_new || !cu_new_lens || !start_pos || !block_table || !k_pool || !v_pool)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
       reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 15u)
    return PA_ERR_INVALID_ARG;
  AppendParams p;
  p.row_chunks = kChunksPerHead * dims.num_kv_heads;
  p.k_new = static_cast<const uint8_t*>(k_new);
  p.v_new = static_cast<const uint8_t*>(v_new);
  p.cu_new_lens = cu_new_lens;
  p.start_pos = start_pos;
  p.batch = batch;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.k_pool = static_cast<uint8_t*>(k_pool);
  p.v_pool = static_cast<uint8_t*>(v_pool);
  p.num_pages = num_pages;
  p.status = status;
  kv_append_kernel<<<total_new, 2 * p.row_chunks, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  PA_CHECK_LAUNCH("kv_append_kernel");
  return PA_OK;
}
