// adaptor_mlp_merge4: the audio-text bridge in front of the decoder (sm_103a).
//
// Source: "Optimizing ASR Models to Transcribe 90-Minute Multi-Speaker Audio", "ASR Model
// Primer" (encoder bullet and component table: 4x frame merge, then an FFN adapter
// Linear -> SiLU -> Linear -> LayerNorm, 4096 -> 1024); "MOSS-Transcribe-Diarize 0.9B",
// "Model Architecture" (4x temporal merge + MLP adaptor). Hidden width read as 1024:
//   x = frames viewed as [T, 4096] (row t = frames 4t..4t+3 side by side: no copy)
//   h = SiLU(x W1^T + b1)            [T, 1024]  bf16 (workspace)
//   y = LayerNorm(h W2^T + b2)       [T, 1024]  bf16 (out; pre-norm values staged in out)
//
// The two linears run on one persistent tcgen05 GEMM kernel over CTA pairs (clusters of 2,
// .cta_group::2): a pair owns a 256-row x 256-column output tile, K in 64-element blocks
// through a 6-stage TMA ring per CTA (its 128 A rows, 16 KB, and 128 of the tile's 256 weight
// rows, 16 KB; 128-byte swizzle), fp32 accumulators in two 256-column TMEM buffers per CTA so
// the epilogue of one tile overlaps the MMAs of the next. Warps: 0-3 epilogue (bias, SiLU,
// bf16, store), 4 TMA producer, 5 MMA issuer (even CTA). Tiles are numbered row tile by row
// tile, so the pairs that run the column tiles of one row tile at the same time read its A rows
// from L2 once they are in; the weights (8 MB and 2 MB) stay in L2 throughout.
// LayerNorm is a row-wise pass (one warp per row) over the staged pre-norm rows.
#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "cluster_common.cuh"
#include "pa_common.cuh"
#include "tc_common.cuh"
#include "tc_pair.cuh"

namespace pa {

bool make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                 uint64_t row_stride_bytes, uint32_t box_rows);

namespace {

constexpr int kDModel = 1024;
constexpr int kMerge = 4;
constexpr int kIn = kDModel * kMerge;  // 4096
constexpr int kHidden = 1024;
constexpr int kOut = 1024;

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kGemmThreads = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB

struct GemmParams {
  int32_t M, N, K;
  const float* bias;   // [N]
  uint16_t* c;         // bf16 [M][N]
  int32_t silu;        // apply SiLU after the bias
  int32_t* status;
};

__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_wait_bounded(bar, parity)) return true;
  flag_error(status, PA_DEV_ERR_TIMEOUT);
  return false;
}

// One M = 256 MMA issued by the even CTA covers a pair's whole tile, each CTA's 128 accumulator
// rows landing in its own TMEM. Per SM that is 8 KB of shared-memory operand reads per
// 128x256x16 step and 32 KB of copies per K block, against 12 KB and 48 KB for a 1-CTA
// 128 x 256 tile, and each weight tile crosses from L2 once per pair.
constexpr int kPairBM = 256;
constexpr int kPairStages = 6;
constexpr uint32_t kHalfBBytes = 128 * kBK * 2;  // 16 KB
constexpr int kEpilogueWarps = 4;

struct PairGemmSmem {  // placed at a 1024-byte aligned address; the same layout in both CTAs
  uint8_t a[kPairStages][kABytes];
  uint8_t b[kPairStages][kHalfBBytes];
  uint64_t full[kPairStages], empty[kPairStages];   // full: used in the even CTA only
  uint64_t acc_full[2], acc_empty[2];                // acc_empty: used in the even CTA only
  uint64_t mma_done;
  uint32_t tmem_base;
};
static_assert(sizeof(PairGemmSmem) + 1024 <= 232448, "pair GEMM shared memory over the 227 KB limit");

__device__ __forceinline__ bool wait_cl_or_flag(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_wait_cluster_bounded(bar, parity)) return true;
  flag_error(status, PA_DEV_ERR_TIMEOUT);
  return false;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_bias_act_kernel(const __grid_constant__ CUtensorMap a_map,
                 const __grid_constant__ CUtensorMap b_map, const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  PairGemmSmem& s = *reinterpret_cast<PairGemmSmem*>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int m_tiles = (p.M + kPairBM - 1) / kPairBM, n_tiles = p.N / kBN;
  // unit u = row tile u / n_tiles x column tile u % n_tiles; pair c takes units c, c + G, ...
  const int units = m_tiles * n_tiles;
  const int k_blocks = p.K / kBK;
  const int cl = static_cast<int>(blockIdx.x >> 1), n_cl = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPairStages; ++i) {
      mbar_init(&s.full[i], 1);    // the even CTA's producer (+ both CTAs' bytes)
      mbar_init(&s.empty[i], 1);   // the issuer's commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.acc_full[i], 1);
      mbar_init(&s.acc_empty[i], 2 * kEpilogueWarps);  // one arrive per epilogue warp of each CTA
    }
    mbar_init(&s.mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 5) tc::tmem_alloc_pair<512>(&s.tmem_base);
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any arrive reaches them
  tc::fence_after_sync();
  const uint32_t tmem = s.tmem_base;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer (both)
    if (lane == 0) {
      const uint32_t full0 = map_to_rank(&s.full[0], 0);
      uint32_t it = 0;
      bool ok = true;
      for (int u = cl; u < units && ok; u += n_cl) {
        const int m0 = (u / n_tiles) * kPairBM + static_cast<int>(rank) * kBM;
        const int n0 = (u % n_tiles) * kBN + static_cast<int>(rank) * (kBN / 2);
        for (int kb = 0; kb < k_blocks && ok; ++kb, ++it) {
          const uint32_t st = it % kPairStages;
          ok = wait_cl_or_flag(&s.empty[st], ((it / kPairStages) & 1) ^ 1u, p.status);
          if (!ok) break;
          if (rank == 0) mbar_arrive_expect_tx(&s.full[st], 2 * (kABytes + kHalfBBytes));
          tc::tma_load_2d_pair(s.a[st], &a_map, kb * kBK, m0, full0 + 8u * st);
          tc::tma_load_2d_pair(s.b[st], &b_map, kb * kBK, n0, full0 + 8u * st);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer (even CTA)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16(kPairBM, kBN, 0, 0);
      const uint32_t empty_me = smem_addr(&s.empty[0]), empty_peer = map_to_rank(&s.empty[0], 1);
      const uint32_t accf_me = smem_addr(&s.acc_full[0]), accf_peer = map_to_rank(&s.acc_full[0], 1);
      uint32_t it = 0, tc_n = 0;
      bool ok = true;
      for (int u = cl; u < units && ok; u += n_cl, ++tc_n) {
        const uint32_t acc = tc_n & 1;
        ok = wait_cl_or_flag(&s.acc_empty[acc], ((tc_n >> 1) & 1) ^ 1u, p.status);
        if (!ok) break;
        tc::fence_after_sync();
        for (int kb = 0; kb < k_blocks && ok; ++kb, ++it) {
          const uint32_t st = it % kPairStages;
          ok = wait_cl_or_flag(&s.full[st], (it / kPairStages) & 1, p.status);
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t aa = smem_addr(s.a[st]), bb = smem_addr(s.b[st]);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc::mma_ss_pair(tmem + acc * kBN, tc::smem_desc_sw128(aa + kk * 32, 16, 1024),
                            tc::smem_desc_sw128(bb + kk * 32, 16, 1024), idesc,
                            (kb > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit_pair(empty_me + 8u * st);
          tc::mma_commit_pair(empty_peer + 8u * st);
        }
        if (ok) {
          tc::mma_commit_pair(accf_me + 8u * acc);
          tc::mma_commit_pair(accf_peer + 8u * acc);
        }
      }
      tc::mma_commit_pair(smem_addr(&s.mma_done));
      wait_or_flag(&s.mma_done, 0, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue warps 0-3
    const int r = warp * 32 + lane;  // row of this CTA's half tile = TMEM lane
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t acc_empty0 = map_to_rank(&s.acc_empty[0], 0);
    uint32_t tc_n = 0;
    for (int u = cl; u < units; u += n_cl, ++tc_n) {
      const uint32_t acc = tc_n & 1;
      if (!__all_sync(0xffffffffu, wait_cl_or_flag(&s.acc_full[acc], (tc_n >> 1) & 1, p.status)))
        break;
      tc::fence_after_sync();
      const int m0 = (u / n_tiles) * kPairBM + static_cast<int>(rank) * kBM, n0 = (u % n_tiles) * kBN;
      const int row = m0 + r;
      uint16_t* dst = p.c + static_cast<int64_t>(row) * p.N + n0;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + lane_bits + acc * kBN + c * 32, v);
        tc::tmem_wait_ld();
        const float bias_lane = __ldg(p.bias + n0 + c * 32 + lane);
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float x = __uint_as_float(v[i]) + __shfl_sync(0xffffffffu, bias_lane, i);
          if (p.silu) x = __fdividef(x, 1.0f + __expf(-x));
          f[i] = x;
        }
        if (row < p.M) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_bf16x2(f[8 * i + 0], f[8 * i + 1]);
            w.y = pack_bf16x2(f[8 * i + 2], f[8 * i + 3]);
            w.z = pack_bf16x2(f[8 * i + 4], f[8 * i + 5]);
            w.w = pack_bf16x2(f[8 * i + 6], f[8 * i + 7]);
            *reinterpret_cast<uint4*>(dst + c * 32 + 8 * i) = w;
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(&s.acc_empty[acc]);
        else mbar_arrive_cluster(acc_empty0 + 8u * acc);
      }
    }
  }

  // Neither CTA releases TMEM or leaves while the pair's MMAs may still read its shared memory
  // or write its TMEM: the issuer has seen all of them complete before it gets here, and every
  // stage either CTA loaded was consumed by an MMA.
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  tc::fence_after_sync();
  if (warp == 5) tc::tmem_dealloc_pair<512>(tmem);
}

// Row-wise LayerNorm over kOut columns, in place on bf16 rows; one warp per row.
__global__ void __launch_bounds__(256) layernorm_rows_kernel(uint16_t* y, int32_t rows,
                                                             const float* gamma,
                                                             const float* beta, float eps) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= rows) return;
  uint16_t* p = y + static_cast<int64_t>(row) * kOut;
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // lane owns columns 8 * (lane + 32 i) .. + 7
    const uint4 w = *reinterpret_cast<const uint4*>(p + 8 * (lane + 32 * i));
    v[8 * i + 0] = bf16lo(w.x); v[8 * i + 1] = bf16hi(w.x);
    v[8 * i + 2] = bf16lo(w.y); v[8 * i + 3] = bf16hi(w.y);
    v[8 * i + 4] = bf16lo(w.z); v[8 * i + 5] = bf16hi(w.z);
    v[8 * i + 6] = bf16lo(w.w); v[8 * i + 7] = bf16hi(w.w);
  }
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) sum += v[i];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float mean = sum * (1.0f / kOut);
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float d = v[i] - mean;
    sq += d * d;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  const float rstd = rsqrtf(sq * (1.0f / kOut) + eps);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int col = 8 * (lane + 32 * i);
    // the scale and shift of these 8 columns as two 16-byte loads each
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma + col));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma + col + 4));
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(beta + col));
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(beta + col + 4));
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    float o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = (v[8 * i + k] - mean) * rstd * g[k] + bb[k];
    uint4 w;
    w.x = pack_bf16x2(o[0], o[1]);
    w.y = pack_bf16x2(o[2], o[3]);
    w.z = pack_bf16x2(o[4], o[5]);
    w.w = pack_bf16x2(o[6], o[7]);
    *reinterpret_cast<uint4*>(p + col) = w;
  }
}

// Pairs of the persistent pair grid: as many clusters of 2 as can be resident at once, computed
// once per device (0 when the query fails).
int gemm_pairs(int dev) {
  static std::mutex mu;
  static int cached[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  const int smem = static_cast<int>(sizeof(PairGemmSmem)) + 1024;
  if (cudaFuncSetAttribute(gemm_bias_act_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * std::max(1, sm_count_current_device() / 2));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_bias_act_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 0;
  }
  cached[dev] = n;
  return n;
}

pa_status launch_gemm(const void* a, int64_t lda_bytes, const void* b, int M, int N, int K,
                      const float* bias, void* c, bool silu, int32_t* status,
                      cudaStream_t stream) {
  CUtensorMap am, bm;
  if (!make_map_2d(&am, a, static_cast<uint64_t>(M), static_cast<uint64_t>(K),
                   static_cast<uint64_t>(lda_bytes), kBM) ||
      !make_map_2d(&bm, b, static_cast<uint64_t>(N), static_cast<uint64_t>(K),
                   static_cast<uint64_t>(K) * 2, kBN / 2)) {
    snprintf_error("cuTensorMapEncodeTiled failed for the adaptor operands");
    return PA_ERR_CUDA;
  }
  int dev = 0;
  cudaGetDevice(&dev);
  const int pairs = gemm_pairs(dev);
  if (pairs <= 0) {
    snprintf_error("adaptor: no cluster of 2 CTAs fits on this device");
    return PA_ERR_CUDA;
  }
  GemmParams p{M, N, K, bias, static_cast<uint16_t*>(c), silu ? 1 : 0, status};
  const int units = (M + kPairBM - 1) / kPairBM * (N / kBN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * std::min(pairs, units));   // one CTA per SM, in pairs
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = sizeof(PairGemmSmem) + 1024;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_bias_act_kernel, am, bm, p);
  if (e != cudaSuccess) return record_cuda_error(e, "gemm_bias_act_kernel");
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" size_t pa_adaptor_workspace_size(int32_t num_frames) {
  if (num_frames < 0) return 0;
  return static_cast<size_t>(num_frames / pa::kMerge) * pa::kHidden * 2 + 256;
}

extern "C" pa_status adaptor_mlp_merge4(int32_t num_frames, const void* frames, const void* w1,
                                        const float* b1, const void* w2, const float* b2,
                                        const float* gamma, const float* beta, float eps,
                                        void* out, void* workspace, size_t workspace_bytes,
                                        int32_t* status, pa_stream_t stream) {
  using namespace pa;
  if (num_frames < 0 || num_frames % kMerge != 0 || !(eps >= 0.f)) return PA_ERR_INVALID_ARG;
  if (num_frames == 0) return PA_OK;
  if (num_frames / kMerge >= (1 << 24)) return PA_ERR_UNSUPPORTED;
  if (!frames || !w1 || !b1 || !w2 || !b2 || !gamma || !beta || !out || !workspace)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(frames) | reinterpret_cast<uintptr_t>(w1) |
       reinterpret_cast<uintptr_t>(w2) | reinterpret_cast<uintptr_t>(out) |
       reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(gamma) |
       reinterpret_cast<uintptr_t>(beta)) & 15u)
    return PA_ERR_INVALID_ARG;
  if (workspace_bytes < pa_adaptor_workspace_size(num_frames)) return PA_ERR_WORKSPACE_TOO_SMALL;
  const int T = num_frames / kMerge;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // h = SiLU(x W1^T + b1), x = frames viewed as [T][4096]
  pa_status r = launch_gemm(frames, static_cast<int64_t>(kIn) * 2, w1, T, kHidden, kIn, b1,
                            workspace, true, status, st);
  if (r != PA_OK) return r;
  // pre-norm y = h W2^T + b2, staged in out
  r = launch_gemm(workspace, static_cast<int64_t>(kHidden) * 2, w2, T, kOut, kHidden, b2, out,
                  false, status, st);
  if (r != PA_OK) return r;
  layernorm_rows_kernel<<<(T + 7) / 8, 256, 0, st>>>(static_cast<uint16_t*>(out), T, gamma, beta,
                                                      eps);
  PA_CHECK_LAUNCH("layernorm_rows_kernel");
  return PA_OK;
}
