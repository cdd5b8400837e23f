// attn_prefill_chunk: causal attention of query chunks over a paged KV cache (sm_103a).
//
// Source: chunked prefill of long audio prompts, 4096 tokens per scheduling step, each chunk
// attending to the KV cache of the earlier chunks plus its own tokens ("Optimizing ASR
// Models to Transcribe 90-Minute Multi-Speaker Audio", "Chunked Prefill for Long Audio";
// "MOSS-Transcribe-Diarize" cookbook, "Inference Pipeline").
//
// CUDA-core tiled kernel: a CTA takes 64 query rows of one chunk and both query heads of one
// KV head (128 (row, head) pairs, two threads per pair, 64 dims each). Key tiles of 32 tokens
// are gathered from their pages, widened to fp32 once into shared memory, and consumed with an
// online softmax in the exp2 domain. Only the tiles up to the block's last visible key are
// visited; masking is applied per key on the diagonal.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kRows = 64;   // query rows per CTA
constexpr int kKeys = 32;   // keys per tile
constexpr int kThreads = kRows * kGroup * 2;
constexpr int kHalf = kHeadDim / 2;

struct PrefillParams {
  const uint16_t* q;
  const int32_t* cu_q_lens;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  int64_t num_pages;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  int32_t batch;
  float scale_log2;
  uint16_t* out;
  float* lse;
  int32_t* status;
};

struct PrefillSmem {
  float k[kKeys][kHeadDim];
  float v[kKeys][kHeadDim];
  int32_t page[kKeys / kPage + 1];
};

__global__ void __launch_bounds__(kThreads, 1) prefill_cc_kernel(const PrefillParams p) {
  __shared__ __align__(16) PrefillSmem s;
  const int b = blockIdx.z, g = blockIdx.y;
  const int q0 = p.cu_q_lens[b];
  const int n = p.cu_q_lens[b + 1] - q0;
  const int row0 = blockIdx.x * kRows;
  if (n <= 0 || row0 >= n) return;
  const int L = p.seq_lens[b];
  if (n > L || L > p.bt_stride * kPage) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && g == 0) flag_error(p.status, PA_DEV_ERR_LENGTH);
    return;
  }
  const int off = L - n;  // position of the chunk's first query
  const int tid = threadIdx.x;
  const int pair = tid >> 1, half = tid & 1;
  const int qi = row0 + (pair >> 1);
  const int head = kGroup * g + (pair & 1);
  const bool live = qi < n;
  const int qpos = off + qi;
  const int last_key = off + min(n, row0 + kRows) - 1;  // largest visible key of the block

  float2 q[kHalf / 2];
  {
    const int qr = live ? qi : 0;
    const uint4* src = reinterpret_cast<const uint4*>(
        p.q + (static_cast<int64_t>(q0 + qr) * kHq + head) * kHeadDim + half * kHalf);
#pragma unroll
    for (int i = 0; i < kHalf / 8; ++i) {
      const uint4 w = src[i];
      q[4 * i + 0] = make_float2(bf16lo(w.x) * p.scale_log2, bf16hi(w.x) * p.scale_log2);
      q[4 * i + 1] = make_float2(bf16lo(w.y) * p.scale_log2, bf16hi(w.y) * p.scale_log2);
      q[4 * i + 2] = make_float2(bf16lo(w.z) * p.scale_log2, bf16hi(w.z) * p.scale_log2);
      q[4 * i + 3] = make_float2(bf16lo(w.w) * p.scale_log2, bf16hi(w.w) * p.scale_log2);
    }
  }
  float2 o[kHalf / 2];
#pragma unroll
  for (int i = 0; i < kHalf / 2; ++i) o[i] = make_float2(0.f, 0.f);
  float m = -CUDART_INF_F, l = 0.f;

  const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
  for (int kt = 0; kt <= last_key; kt += kKeys) {
    __syncthreads();
    if (tid < kKeys / kPage) {
      int page = -1;  // table entries past the sequence's last page are never read
      if (kt + tid * kPage < L) {
        page = bt_row[kt / kPage + tid];
        if (page < 0 || page >= p.num_pages) {
          flag_error(p.status, PA_DEV_ERR_PAGE_OOB);
          page = 0;
        }
      }
      s.page[tid] = page;
    }
    __syncthreads();
    // gather + widen: 32 keys x 16 chunks of 8 dims, for K and V
    for (int e = tid; e < 2 * kKeys * (kHeadDim / 8); e += kThreads) {
      const int which = e / (kKeys * (kHeadDim / 8));
      const int r = e % (kKeys * (kHeadDim / 8));
      const int j = r / (kHeadDim / 8), c = r % (kHeadDim / 8);
      const int page = s.page[j / kPage];
      float* dst = which ? &s.v[j][8 * c] : &s.k[j][8 * c];
      if (page < 0 || kt + j >= L) {
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = 0.f;
      } else {
        const uint8_t* base = which ? p.v_pool : p.k_pool;
        const uint4 w = *reinterpret_cast<const uint4*>(
            base + ((static_cast<int64_t>(page) * kPage + (j % kPage)) * kHkv + g) * (kHeadDim * 2) + 16 * c);
        dst[0] = bf16lo(w.x); dst[1] = bf16hi(w.x);
        dst[2] = bf16lo(w.y); dst[3] = bf16hi(w.y);
        dst[4] = bf16lo(w.z); dst[5] = bf16hi(w.z);
        dst[6] = bf16lo(w.w); dst[7] = bf16hi(w.w);
      }
    }
    __syncthreads();
    float sc[kKeys];
#pragma unroll
    for (int j = 0; j < kKeys; ++j) {
      const float4* kr = reinterpret_cast<const float4*>(&s.k[j][half * kHalf]);
      float2 a = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kHalf / 4; ++i) {
        const float4 kk = kr[i];
        a = fma2(q[2 * i], make_float2(kk.x, kk.y), a);
        a = fma2(q[2 * i + 1], make_float2(kk.z, kk.w), a);
      }
      float d = a.x + a.y;
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      sc[j] = (live && kt + j <= qpos) ? d : -CUDART_INF_F;
    }
    float tm = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < kKeys; ++j) tm = fmaxf(tm, sc[j]);
    if (!live || tm == -CUDART_INF_F) continue;
    const float mn = fmaxf(m, tm);
    const float alpha = (m == -CUDART_INF_F) ? 0.f : fast_exp2(m - mn);
    const float2 aa = make_float2(alpha, alpha);
#pragma unroll
    for (int i = 0; i < kHalf / 2; ++i) o[i] = mul2(o[i], aa);
    l *= alpha;
    m = mn;
#pragma unroll
    for (int j = 0; j < kKeys; ++j) {
      const float pj = fast_exp2(sc[j] - m);
      l += pj;
      const float2 pp = make_float2(pj, pj);
      const float4* vr = reinterpret_cast<const float4*>(&s.v[j][half * kHalf]);
#pragma unroll
      for (int i = 0; i < kHalf / 4; ++i) {
        const float4 vv = vr[i];
        o[2 * i] = fma2(make_float2(vv.x, vv.y), pp, o[2 * i]);
        o[2 * i + 1] = fma2(make_float2(vv.z, vv.w), pp, o[2 * i + 1]);
      }
    }
  }
  if (!live) return;
  const float inv = 1.0f / l;
  uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(q0 + qi) * kHq + head) * kHeadDim + half * kHalf);
#pragma unroll
  for (int i = 0; i < kHalf / 8; ++i) {
    uint4 w;
    w.x = pack_bf16x2(o[4 * i].x * inv, o[4 * i].y * inv);
    w.y = pack_bf16x2(o[4 * i + 1].x * inv, o[4 * i + 1].y * inv);
    w.z = pack_bf16x2(o[4 * i + 2].x * inv, o[4 * i + 2].y * inv);
    w.w = pack_bf16x2(o[4 * i + 3].x * inv, o[4 * i + 3].y * inv);
    dst[i] = w;
  }
  if (half == 0 && p.lse != nullptr) p.lse[static_cast<int64_t>(q0 + qi) * kHq + head] = (m + log2f(l)) * kLn2;
}

}  // namespace
}  // namespace pa

extern "C" size_t pa_prefill_workspace_size(pa_dims dims, int32_t batch, int32_t max_q_len,
                                            int32_t max_seq_len) {
  (void)dims; (void)batch; (void)max_q_len; (void)max_seq_len;
  return 0;
}

extern "C" pa_status attn_prefill_chunk(pa_dims dims, const void* q, const int32_t* cu_q_lens,
                                        int32_t total_q, const void* k_pool, const void* v_pool,
                                        int64_t num_pages, const int32_t* block_table,
                                        int32_t bt_stride, const int32_t* seq_lens,
                                        int32_t batch, int32_t max_q_len, int32_t max_seq_len,
                                        float softmax_scale, void* out, float* lse,
                                        void* workspace, size_t workspace_bytes,
                                        int32_t* status, pa_stream_t stream) {
  using namespace pa;
  (void)workspace; (void)workspace_bytes;
  if (dims.num_q_heads != kHq || dims.num_kv_heads != kHkv || dims.head_dim != kHeadDim ||
      dims.page_size != kPage)
    return PA_ERR_UNSUPPORTED;
  if (total_q < 0 || batch < 0 || bt_stride <= 0 || num_pages <= 0 || max_q_len < 0 ||
      max_seq_len < 0 || max_seq_len > 131072 || max_q_len > max_seq_len ||
      !(softmax_scale == softmax_scale) || batch > 65535)
    return PA_ERR_INVALID_ARG;
  if (batch == 0 || max_q_len == 0 || total_q == 0) return PA_OK;
  if (!q || !cu_q_lens || !k_pool || !v_pool || !block_table || !seq_lens || !out)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pool) |
       reinterpret_cast<uintptr_t>(v_pool) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return PA_ERR_INVALID_ARG;
  PrefillParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.cu_q_lens = cu_q_lens;
  p.k_pool = static_cast<const uint8_t*>(k_pool);
  p.v_pool = static_cast<const uint8_t*>(v_pool);
  p.num_pages = num_pages;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.scale_log2 = softmax_scale * kLog2e;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.status = status;
  dim3 grid((max_q_len + kRows - 1) / kRows, kHkv, batch);
  prefill_cc_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  PA_CHECK_LAUNCH("prefill_cc_kernel");
  return PA_OK;
}
