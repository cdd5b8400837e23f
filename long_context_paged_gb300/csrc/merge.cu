// attn_merge_lse: combine attention results computed over disjoint key sets (sm_103a).
//
// With lse = ln sum_s exp(lse_s), the whole is o = sum_s exp(lse_s - lse) o_s: the exact
// recombination that split-KV decoding of long caches relies on. Parts whose lse is -inf are
// empty and carry no weight; their o_s is never read.
//
// One warp per (row, head); each lane owns 4 consecutive dims per 128-dim slice.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "pa_common.cuh"

namespace pa {
namespace {

struct MergeParams {
  int32_t num_parts, rows, heads, head_dim;
  const float* o_parts;
  const float* lse_parts;
  uint16_t* out;
  float* lse_out;
};

__global__ void __launch_bounds__(256) merge_lse_kernel(const MergeParams p) {
  const int64_t item = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t items = static_cast<int64_t>(p.rows) * p.heads;
  if (item >= items) return;
  float m = -CUDART_INF_F;
  for (int s = lane; s < p.num_parts; s += 32) m = fmaxf(m, p.lse_parts[s * items + item]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  uint16_t* orow = p.out + item * p.head_dim;
  if (m == -CUDART_INF_F) {
    for (int d = 4 * lane; d < p.head_dim; d += 128)
      *reinterpret_cast<uint2*>(orow + d) = make_uint2(0u, 0u);
    if (lane == 0 && p.lse_out != nullptr) p.lse_out[item] = -CUDART_INF_F;
    return;
  }
  float sum = 0.f;
  for (int d0 = 0; d0 < p.head_dim; d0 += 128) {
    const int d = d0 + 4 * lane;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    sum = 0.f;
    for (int s = 0; s < p.num_parts; ++s) {
      const float l = p.lse_parts[s * items + item];
      if (l == -CUDART_INF_F) continue;
      const float w = fast_exp2((l - m) * kLog2e);
      sum += w;
      if (d < p.head_dim) {
        const float4 o = *reinterpret_cast<const float4*>(p.o_parts + (s * items + item) * p.head_dim + d);
        acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
      }
    }
    if (d < p.head_dim) {
      const float inv = 1.0f / sum;
      *reinterpret_cast<uint2*>(orow + d) =
          make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
  }
  if (lane == 0 && p.lse_out != nullptr) p.lse_out[item] = m + logf(sum);
}

}  // namespace
}  // namespace pa

extern "C" pa_status attn_merge_lse(int32_t num_parts, int32_t rows, int32_t heads,
                                    int32_t head_dim, const float* o_parts,
                                    const float* lse_parts, void* out, float* lse_out,
                                    pa_stream_t stream) {
  using namespace pa;
  if (num_parts < 0 || rows < 0 || heads < 0 || head_dim <= 0) return PA_ERR_INVALID_ARG;
  if (head_dim % 4 != 0 || head_dim > 1024) return PA_ERR_UNSUPPORTED;
  const int64_t items = static_cast<int64_t>(rows) * heads;
  if (items == 0) return PA_OK;
  if (!out || (num_parts > 0 && (!o_parts || !lse_parts))) return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(o_parts) & 15u) || (reinterpret_cast<uintptr_t>(out) & 7u))
    return PA_ERR_INVALID_ARG;
  if (items > (static_cast<int64_t>(1) << 34)) return PA_ERR_INVALID_ARG;
  MergeParams p{num_parts, rows, heads, head_dim, o_parts, lse_parts,
                static_cast<uint16_t*>(out), lse_out};
  const int64_t blocks = (items + 7) / 8;
  if (blocks > 0x7fffffff) return PA_ERR_INVALID_ARG;
  merge_lse_kernel<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  PA_CHECK_LAUNCH("merge_lse_kernel");
  return PA_OK;
}
