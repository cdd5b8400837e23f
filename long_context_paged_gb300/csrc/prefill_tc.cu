// attn_prefill_chunk on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Source: chunked prefill of long audio prompts, 4096 tokens per scheduling step, each chunk
// attending causally to the KV cache of the earlier chunks plus its own tokens ("Optimizing
// ASR Models to Transcribe 90-Minute Multi-Speaker Audio", "Chunked Prefill for Long Audio";
// "MOSS-Transcribe-Diarize" cookbook, "Inference Pipeline"). QK^T and PV are dense
// contractions here (thousands of queries per KV read), so they run on tcgen05.mma.
//
// One CTA = 128 queries of one chunk x both query heads of one KV head (GQA 16/8), i.e. two
// 128-row M tiles that share every K/V tile read. Per 128-key tile j:
//   S_t = Q_t K_j^T         tcgen05.mma, A = Q_t (smem), B = K_j (smem), D = S_t (TMEM fp32)
//   P_t = softmax part      4 warps per M tile, one thread per row: tcgen05.ld S_t, mask the
//                           diagonal, exp2, row sum; P_t written back over S_t as bf16
//   O_t += P_t V_j          tcgen05.mma, A = P_t (TMEM), B = V_j (smem, MN-major), D = O_t
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
// Warp roles: 0-3 softmax of M tile 0, 4-7 softmax of M tile 1, 8 TMA producer, 9 MMA issuer.
// K/V tiles arrive by tiled TMA straight from the page pools: one 16-token page x 64 dims per
// copy (a 3-D tensor map over [tokens][kv heads][dims] with 128-byte swizzle), so the block
// table is applied per page without any gather pass. Pages past the sequence are fetched at an
// out-of-range coordinate and arrive as zeros; V rows of the last partial page are zeroed in
// shared memory before use, so unwritten slots can never reach P*V.
// The running row max is moved only when a tile exceeds it by more than 8 (log2 units); O is
// then rescaled in TMEM by its owning warps, after the previous P*V has completed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <mutex>

#include "pa_common.cuh"
#include "tc_common.cuh"

namespace pa {
namespace {

constexpr int kTileM = 128;   // queries per CTA (per head)
constexpr int kTileN = 128;   // keys per K/V tile
constexpr int kThreads = 320; // 8 softmax warps + producer + MMA
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kBlockBytes = 128 * 128;  // 128 rows x 64 bf16 (one swizzled 64-dim block)
constexpr uint32_t kTileBytes = 2 * kBlockBytes;
constexpr float kRescaleThreshold = 8.0f;

struct __align__(1024) PrefillTcSmem {
  uint8_t q[2][2][kBlockBytes];   // [M tile][64-dim block]
  uint8_t k[2][2][kBlockBytes];   // [stage][64-dim block]
  uint8_t v[2][2][kBlockBytes];
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], o_ready[2];
  uint64_t mma_done;
  uint32_t tmem_base;
};

struct PrefillTcParams {
  const int32_t* cu_q_lens;
  const int32_t* seq_lens;
  const int32_t* block_table;
  int32_t bt_stride;
  int64_t num_pages;
  float scale_log2;
  uint16_t* out;
  float* lse;
  int32_t* status;
};

__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_wait_bounded(bar, parity)) return true;
  flag_error(status, PA_DEV_ERR_TIMEOUT);
  return false;
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                  const __grid_constant__ CUtensorMap k_map,
                  const __grid_constant__ CUtensorMap v_map, const PrefillTcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  PrefillTcSmem& s = *reinterpret_cast<PrefillTcSmem*>(base);

  const int b = blockIdx.z, g = blockIdx.y, qt = blockIdx.x;
  const int q0 = p.cu_q_lens[b];
  const int n = p.cu_q_lens[b + 1] - q0;
  const int row0 = qt * kTileM;
  if (n <= 0 || row0 >= n) return;
  const int L = p.seq_lens[b];
  if (n > L || L > p.bt_stride * kPage) {
    if (threadIdx.x == 0 && qt == 0 && g == 0) flag_error(p.status, PA_DEV_ERR_LENGTH);
    return;
  }
  const int off = L - n;                                  // position of the chunk's first query
  const int last_key = off + min(n, row0 + kTileM) - 1;   // largest key any row here sees
  const int J = last_key / kTileN + 1;                    // K/V tiles to visit

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
      mbar_init(&s.o_ready[i], 1);
    }
    mbar_init(&s.mma_done, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tc::tmem_alloc<512>(&s.tmem_base);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s.tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ TMA producer
    const int oob_token = static_cast<int>(p.num_pages * kPage);  // zero-filled coordinate
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
    auto page_token = [&](int j) {
      int tok = oob_token;
      const int key0 = j * kTileN + kPage * lane;
      if (lane < kTileN / kPage && key0 < L) {
        const int e = bt_row[key0 / kPage];
        if (e < 0 || e >= p.num_pages) {
          flag_error(p.status, PA_DEV_ERR_PAGE_OOB);
          tok = 0;
        } else {
          tok = e * kPage;
        }
      }
      return tok;
    };
    bool ok = true;
    if (lane == 0) {
      mbar_arrive_expect_tx(&s.q_full, 4 * kBlockBytes);
      for (int t = 0; t < 2; ++t)
        for (int kb = 0; kb < 2; ++kb)
          tc::tma_load_3d(s.q[t][kb], &q_map, kb * 64, 2 * g + t, q0 + row0, &s.q_full);
    }
    int tok = page_token(0);
    for (int j = 0; j < J && ok; ++j) {
      const int st = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      const int tok_next = (j + 1 < J) ? page_token(j + 1) : 0;
      if (lane == 0) ok = wait_or_flag(&s.k_empty[st], ph ^ 1u, p.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&s.k_full[st], kTileBytes);
#pragma unroll
      for (int pg = 0; pg < kTileN / kPage; ++pg) {
        const int t = __shfl_sync(0xffffffffu, tok, pg);
        if (lane == 0) {
          tc::tma_load_3d(s.k[st][0] + pg * 2048, &k_map, 0, g, t, &s.k_full[st]);
          tc::tma_load_3d(s.k[st][1] + pg * 2048, &k_map, 64, g, t, &s.k_full[st]);
        }
      }
      if (lane == 0) ok = wait_or_flag(&s.v_empty[st], ph ^ 1u, p.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&s.v_full[st], kTileBytes);
#pragma unroll
      for (int pg = 0; pg < kTileN / kPage; ++pg) {
        const int t = __shfl_sync(0xffffffffu, tok, pg);
        if (lane == 0) {
          tc::tma_load_3d(s.v[st][0] + pg * 2048, &v_map, 0, g, t, &s.v_full[st]);
          tc::tma_load_3d(s.v[st][1] + pg * 2048, &v_map, 64, g, t, &s.v_full[st]);
        }
      }
      tok = tok_next;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t id_s = tc::idesc_bf16(128, kTileN, 0, 0);    // S = Q K^T
    constexpr uint32_t id_o = tc::idesc_bf16(128, 128, 0, 1);       // O = P V, V MN-major
    auto issue_s = [&](int t, int st) {
      const uint32_t qa = smem_addr(s.q[t][0]), kb = smem_addr(s.k[st][0]);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off_b = (kk >> 2) * kBlockBytes + (kk & 3) * 32;
        tc::mma_ss(tmem + t * 128, tc::smem_desc_sw128(qa + off_b, 16, 1024),
                   tc::smem_desc_sw128(kb + off_b, 16, 1024), id_s, kk > 0);
      }
    };
    auto issue_pv = [&](int t, int st, bool acc) {
      const uint32_t vb = smem_addr(s.v[st][0]);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        tc::mma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                   tc::smem_desc_sw128(vb + kk * 2048, kBlockBytes, 1024), id_o,
                   (acc || kk > 0) ? 1u : 0u);
      }
    };
    bool ok = true;
    if (lane == 0) {
      ok = wait_or_flag(&s.q_full, 0, p.status) && wait_or_flag(&s.k_full[0], 0, p.status);
      if (ok) {
        tc::fence_after_sync();
        issue_s(0, 0);
        tc::mma_commit(&s.s_full[0]);
        issue_s(1, 0);
        tc::mma_commit(&s.s_full[1]);
        tc::mma_commit(&s.k_empty[0]);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    for (int j = 0; j < J && ok; ++j) {
      const int st = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (lane == 0) ok = wait_or_flag(&s.v_full[st], ph, p.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int first_bad = L - j * kTileN;  // V rows at or past this row are not keys
      if (first_bad < kTileN) {
        // zero them so that P = 0 there cannot meet an unwritten (possibly NaN) slot
        const int r0 = max(first_bad, 0);
        for (int e = r0 * 16 + lane; e < kTileN * 16; e += 32) {
          const int r = e >> 4, c = e & 15;   // row, 16-byte chunk (8 per 64-dim block)
          *reinterpret_cast<uint4*>(s.v[st][c >> 3] + r * 128 + (c & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        ok = wait_or_flag(&s.p_full[0], j & 1, p.status);
        if (ok) {
          tc::fence_after_sync();
          issue_pv(0, st, j > 0);
          tc::mma_commit(&s.o_ready[0]);
          if (j + 1 < J) {
            const int st1 = (j + 1) & 1;
            ok = wait_or_flag(&s.k_full[st1], ((j + 1) >> 1) & 1, p.status);
            if (ok) {
              tc::fence_after_sync();
              issue_s(0, st1);
              tc::mma_commit(&s.s_full[0]);
            }
          }
        }
        if (ok) ok = wait_or_flag(&s.p_full[1], j & 1, p.status);
        if (ok) {
          tc::fence_after_sync();
          issue_pv(1, st, j > 0);
          tc::mma_commit(&s.o_ready[1]);
          tc::mma_commit(&s.v_empty[st]);
          if (j + 1 < J) {
            const int st1 = (j + 1) & 1;
            issue_s(1, st1);
            tc::mma_commit(&s.s_full[1]);
            tc::mma_commit(&s.k_empty[st1]);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    // every MMA this thread issued must have finished before TMEM is released
    if (lane == 0) {
      tc::mma_commit(&s.mma_done);
      wait_or_flag(&s.mma_done, 0, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax warps
    const int t = warp >> 2;                       // M tile = query head 2g + t
    const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;             // row of the tile
    const int qrow = row0 + r;
    const int qpos = off + qrow;                   // absolute position of this query
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_bits + t * 128;
    const uint32_t t_o = tmem + lane_bits + 256 + t * 128;
    float m_used = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    for (int j = 0; j < J; ++j) {
      ok = __all_sync(0xffffffffu, wait_or_flag(&s.s_full[t], j & 1, p.status));
      if (!ok) break;
      tc::fence_after_sync();
      float sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rr[32];
        tc::tmem_ld32(t_s + c * 32, rr);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(rr[i]);
      }
      const int k0 = j * kTileN;
      if (k0 + kTileN - 1 > qpos) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (k0 + c > qpos) sv[c] = -CUDART_INF_F;
      }
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < 128; ++c) mx = fmaxf(mx, sv[c]);
      const float mx2 = mx * p.scale_log2;
      const bool grow = mx2 > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, grow)) {
        const float m_new = grow ? mx2 : m_used;
        const float alpha = (m_used == -CUDART_INF_F) ? 0.f : fast_exp2(m_used - m_new);
        if (j > 0) {
          // O_t holds the sum through tile j-1 once the previous P*V has completed
          ok = __all_sync(0xffffffffu, wait_or_flag(&s.o_ready[t], (j - 1) & 1, p.status));
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t rr[32];
            tc::tmem_ld32(t_o + c * 32, rr);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
            tc::tmem_st32(t_o + c * 32, rr);
          }
          tc::tmem_wait_st();
        }
        l *= alpha;
        m_used = m_new;
      }
      // probabilities (bf16) over S's first 64 columns
      const float neg_m = -m_used;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = fast_exp2(fmaf(sv[c * 64 + 2 * i], p.scale_log2, neg_m));
          const float p1 = fast_exp2(fmaf(sv[c * 64 + 2 * i + 1], p.scale_log2, neg_m));
          l += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tc::tmem_st32(t_s + c * 32, pk);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(&s.p_full[t]);
    }
    // epilogue: O / l -> bf16 rows, LSE
    if (ok) ok = __all_sync(0xffffffffu, wait_or_flag(&s.o_ready[t], (J - 1) & 1, p.status));
    if (ok) {
      tc::fence_after_sync();
      const bool live = qrow < n;
      const float inv = 1.0f / l;
      uint16_t* dst = p.out + (static_cast<int64_t>(q0 + qrow) * kHq + 2 * g + t) * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t rr[32];
        tc::tmem_ld32(t_o + c * 32, rr);
        tc::tmem_wait_ld();
        if (live) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(rr[8 * i + 0]) * inv, __uint_as_float(rr[8 * i + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(rr[8 * i + 2]) * inv, __uint_as_float(rr[8 * i + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(rr[8 * i + 4]) * inv, __uint_as_float(rr[8 * i + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(rr[8 * i + 6]) * inv, __uint_as_float(rr[8 * i + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + 8 * i) = w;
          }
        }
      }
      if (live && p.lse != nullptr)
        p.lse[static_cast<int64_t>(q0 + qrow) * kHq + 2 * g + t] = (m_used + log2f(l)) * kLn2;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc<512>(tmem);
  }
}

// ---------------------------------------------------------------------------------------------
// host side: tensor maps (driver entry point looked up once), launch
// ---------------------------------------------------------------------------------------------
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 3-D bf16 view [outer][heads][128 dims] (dims innermost), box = 64 dims x 1 head x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* map, const void* base, uint64_t outer, uint64_t heads, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), heads, outer};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim * 2), heads * kHeadDim * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

pa_status launch_prefill_tc(const void* q, int32_t total_q, const int32_t* cu_q_lens,
                            const void* k_pool, const void* v_pool, int64_t num_pages,
                            const int32_t* block_table, int32_t bt_stride,
                            const int32_t* seq_lens, int32_t batch, int32_t max_q_len,
                            float softmax_scale, void* out, float* lse, int32_t* status,
                            cudaStream_t stream) {
  if (num_pages * kPage >= (int64_t(1) << 31) || total_q >= (1 << 30)) return PA_ERR_UNSUPPORTED;
  CUtensorMap qm, km, vm;
  if (!make_map(&qm, q, static_cast<uint64_t>(total_q), kHq, kTileM) ||
      !make_map(&km, k_pool, static_cast<uint64_t>(num_pages) * kPage, kHkv, kPage) ||
      !make_map(&vm, v_pool, static_cast<uint64_t>(num_pages) * kPage, kHkv, kPage)) {
    snprintf_error("cuTensorMapEncodeTiled failed for the prefill operands");
    return PA_ERR_CUDA;
  }
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  const int smem = static_cast<int>(sizeof(PrefillTcSmem)) + 1024;
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return record_cuda_error(e, "cudaFuncSetAttribute(prefill_tc)");
    configured_device = dev;
  }
  PrefillTcParams p;
  p.cu_q_lens = cu_q_lens;
  p.seq_lens = seq_lens;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.num_pages = num_pages;
  p.scale_log2 = softmax_scale * kLog2e;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.status = status;
  dim3 grid((max_q_len + kTileM - 1) / kTileM, kHkv, batch);
  prefill_tc_kernel<<<grid, kThreads, smem, stream>>>(qm, km, vm, p);
  PA_CHECK_LAUNCH("prefill_tc_kernel");
  return PA_OK;
}

}  // namespace pa
