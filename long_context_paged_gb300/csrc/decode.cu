// attn_decode_paged: split-KV decode attention over a paged KV cache (sm_103a).
//
// Source: the autoregressive decode step of the Qwen3 text decoder (GQA 16/8, head_dim 128)
// that "Optimizing ASR Models to Transcribe 90-Minute Multi-Speaker Audio" ("Where Time Is
// Spent: Profiling") and the "MOSS-Transcribe-Diarize" cookbook ("Where Time Is Spent",
// "Inference Pipeline" item 3) name as the dominant cost on long audio: one query token per
// sequence reads the whole cached K/V of every layer, so the step is bound by HBM reads.
//
// Design (GB300):
//  * Persistent grid, one CTA per SM. The pages of all sequences are laid end to end and cut
//    into contiguous page ranges: by default one equal range per CTA, so a ragged batch
//    (375 .. 70,000 tokens) is balanced to within one page; with an explicit split size the
//    ranges are that many pages and CTA c takes ranges c, c + G, ... A sequence cut by a range
//    boundary yields one partial (o, lse) per range that touches it; a second small kernel
//    merges them by log-sum-exp.
//  * A page holds 16 tokens x 8 KV heads x 128 dims of K (32 KB, contiguous) and the same of
//    V. A producer warp streams whole pages into a 3-stage shared-memory ring with bulk
//    asynchronous copies (cp.async.bulk + mbarrier transaction counts): 64 KB per stage,
//    up to 192 KB in flight per SM. Block-table entries are fetched 32 at a time.
//  * Sixteen consumer warps, two per KV head, each taking 8 of a page's 16 tokens; each serves
//    BOTH query heads of its GQA group from one read of the K/V rows. Lane (c, th) holds dims
//    8c..8c+7 of 4 tokens. Scores are reduce-scattered across the 16 lanes of a half-warp
//    (8 shuffles per page for 8 scores), so each lane ends with one (token, head) score. The
//    two warps of a head keep their own running max and sums and merge once per (sequence,
//    range) through shared memory.
//  * fp32 math on bf16 loads, paired fp32 FMAs (fma.rn.f32x2). The running max is only moved
//    when a page exceeds it by more than 8 (log2 units), so the accumulators are rescaled
//    rarely; probabilities stay <= 2^8 and the result is exact up to rounding.
#include <algorithm>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "cluster_common.cuh"
#include "pa_common.cuh"

namespace pa {
namespace {

// Two consumer warps per (KV head, page slot) pair, each taking half of every page's tokens: with
// one warp per pair a CTA consumed a 64 KB stage in ~2,100 cycles (two warps per SMSP, bound by
// their dependent latencies), which capped it at ~61 GB/s however few CTAs shared the HBM.
constexpr int kPairs = 8;
constexpr int kConsumerWarps = 2 * kPairs;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
// A ring stage holds K (or V) of 16 tokens x 8 KV heads: one page of the decoder's pools, or
// 8 / Hkv consecutive pages of a call with Hkv < 8 KV heads.
constexpr uint32_t kStageBytes = kPage * kHkv * kHeadDim * 2;
constexpr int kMaxBatch = 4096;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Fewest pages per range by default: a short batch is spread one page per SM (two or four
// pages per CTA measured 0.9 and 2.4-2.9 us slower for one sequence of 1,000 keys).
constexpr int kMinPagesPerCta = 1;

struct DecodeSmem {
  uint8_t kv[kStages][2][kStageBytes];
  alignas(16) float2 p2[kConsumerWarps][16];  // probabilities, each as a (p, p) pair
  // hand-off of a (sequence, range)'s second token half to the first: per warp pair, lane l's
  // 8 accumulator values and each head's max and sum
  alignas(16) float xo[kPairs][32][8];
  float xm[kPairs][2];
  float xl[kPairs][2];
  uint64_t xfull[kPairs];
  uint64_t xempty[kPairs];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int32_t warp_tot[kThreads / 32];
  int32_t total;
  int32_t prefix[kMaxBatch + 1];
};
static_assert(sizeof(DecodeSmem) <= 227 * 1024, "decode shared memory beyond the per-CTA limit");

struct DecodeParams {
  int32_t hq;           // query heads of the call (2 x its KV heads)
  int32_t stage_pages;  // pages per ring stage: 8 / KV heads
  const uint16_t* q;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  int64_t num_pages;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t max_seq_len;
  int32_t split_pages;  // pages per range; 0 = an equal share per CTA
  int32_t max_ranges;   // ranges the workspace has records for (the grid size by default)
  float scale_log2;
  uint16_t* out;
  float* lse;
  int32_t* ws_header;  // [0] = pages per range (W), [1] = total pages, [2] = grid size
  int32_t* ws_prefix;  // [batch + 1]
  float* ws_lse;       // [records][Hq], record (b + range) * stage_pages + page slot
  float* ws_o;         // [records][Hq][D]
  int32_t* status;
  uint64_t wait_limit_ns;  // bound of every mbarrier wait
  int32_t starve;          // test hook: CTA 0 never fills its first ring stage
};

// Maximum of v over the 32 lanes of the warp, in every lane (redux.sync on fp32, sm_100 and
// later; like fmaxf, a NaN operand is ignored when another lane holds a number).
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Keys of sequence b as the kernels use them: negative -> 0, more than the table row covers
// -> cut to bt_stride * 16 (both flagged).
__device__ __forceinline__ int clamp_len(const DecodeParams& p, int b, bool report) {
  int L = p.seq_lens[b];
  const int cap = p.bt_stride * kPage;
  if (L < 0 || L > cap || L > p.max_seq_len) {
    if (report) flag_error(p.status, PA_DEV_ERR_LENGTH);
    L = L < 0 ? 0 : (L > cap ? cap : L);
  }
  return L;
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// prefix[b] = first global page of sequence b, prefix[batch] = total pages.
__device__ void build_prefix(const DecodeParams& p, DecodeSmem& s) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (p.batch + kThreads - 1) / kThreads;
  const int b0 = min(p.batch, tid * per), b1 = min(p.batch, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += (clamp_len(p, b, blockIdx.x == 0) + kPage - 1) / kPage;
  const int incl = warp_incl_scan(local, lane);
  if (lane == 31) s.warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = lane < kThreads / 32 ? s.warp_tot[lane] : 0;
    int sc = warp_incl_scan(v, lane);
    if (lane < kThreads / 32) s.warp_tot[lane] = sc - v;
    if (lane == 31) s.total = sc;
  }
  __syncthreads();
  int run = s.warp_tot[warp] + incl - local;
  for (int b = b0; b < b1; ++b) {
    s.prefix[b] = run;
    run += (clamp_len(p, b, false) + kPage - 1) / kPage;
  }
  if (tid == 0) s.prefix[p.batch] = s.total;
  __syncthreads();
}

// Last b with prefix[b] <= x (prefix non-decreasing, prefix[0] = 0 <= x < prefix[batch]).
__device__ __forceinline__ int find_seq(const int32_t* prefix, int batch, int x) {
  int lo = 0, hi = batch;  // invariant: prefix[lo] <= x < prefix[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// kHkvT: KV heads of the call (8 for the decoder; 1, 2 or 4 for a device's share of them).
// Consumer warp w serves KV head (w % 8) % kHkvT of page slot (w % 8) / kHkvT of each stage, tokens
// 8 * (w / 8) .. +7 of each page.
template <int kHkvT>
__global__ void __launch_bounds__(kThreads, 1) decode_splitkv_kernel(const DecodeParams p) {
  constexpr int kSlots = kHkv / kHkvT;                        // pages per stage
  constexpr int kHqT = kGroup * kHkvT;
  constexpr uint32_t kPageBytes = kPage * kHkvT * kHeadDim * 2;  // K (or V) of one page
  constexpr int kTokenBytes = kHkvT * kHeadDim * 2;             // one token's row in a page
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DecodeSmem& s = *reinterpret_cast<DecodeSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], kConsumerWarps);
    }
    for (int i = 0; i < kPairs; ++i) {
      mbar_init(&s.xfull[i], 32);
      mbar_init(&s.xempty[i], 32);
    }
    fence_mbar_init();
  }
  // This kernel is launched as a programmatic dependent of whatever precedes it on the stream,
  // so its launch and the barrier set-up above overlap the tail of that kernel; nothing written
  // by earlier work is read before this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the merge kernel only reads this grid's results after its own griddepcontrol.wait (full
  // completion), so it may be launched as soon as every CTA of this grid has got here (the
  // lengths it reads before that wait are final by now)
  asm volatile("griddepcontrol.launch_dependents;");
  // pages per range: an equal share per CTA (at least kMinPagesPerCta) unless a split size was
  // given; never fewer than the workspace has records for. A short batch is spread over as many
  // SMs as it has pages: one SM ingests a 32 KB page in well under a microsecond, so a
  // single-sequence decode is latency-bound, and its partials merge in parallel per head.
  const int base = p.split_pages > 0 ? p.split_pages : kMinPagesPerCta;
  // One sequence (a single long request): if its length fills the host's bound to the page,
  // the producer's first block-table entries follow from the bound alone, so they are loaded
  // beside the length instead of after it, and used only once the length confirms them.
  const int total_spec = (p.max_seq_len + kPage - 1) / kPage;
  int spec_entry = 0;
  if (p.batch == 1 && warp == kConsumerWarps) {
    const int W_s = max((total_spec + p.max_ranges - 1) / p.max_ranges, base);
    const int P0_s = static_cast<int>(blockIdx.x) * W_s;
    if (lane < min(W_s, total_spec - P0_s) && P0_s + lane < p.bt_stride)
      spec_entry = p.block_table[P0_s + lane];
  }
  build_prefix(p, s);  // ends with __syncthreads(), which also publishes the barrier init

  const int total = s.total;
  const int W = max((total + p.max_ranges - 1) / p.max_ranges, base);
  if (blockIdx.x == 0) {
    if (tid == 0) {
      p.ws_header[0] = W;
      p.ws_header[1] = total;
      p.ws_header[2] = gridDim.x;
    }
    for (int b = tid; b <= p.batch; b += kThreads) p.ws_prefix[b] = s.prefix[b];
  }
  if (total == 0) return;
  const int n_ranges = (total + W - 1) / W;  // <= max_ranges
  if (static_cast<int>(blockIdx.x) >= n_ranges) return;

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer warp
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    bool ok = true;
    bool starve = p.starve != 0 && blockIdx.x == 0;
    for (int rg = blockIdx.x; ok && rg < n_ranges; rg += gridDim.x) {
      const int P0 = rg * W, P1 = min(total, P0 + W);
      const int b_first = find_seq(s.prefix, p.batch, P0);
      for (int b = b_first; ok && b < p.batch && s.prefix[b] < P1; ++b) {
        const int lp0 = max(P0, s.prefix[b]) - s.prefix[b];
        const int lp1 = min(P1, s.prefix[b + 1]) - s.prefix[b];
        const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
        for (int lp = lp0; ok && lp < lp1; lp += 32) {
          const int n = min(32, lp1 - lp);
          // the entries loaded before the length are this CTA's first 32 when the length gave
          // the same page count as the bound (then W and this range are the ones assumed)
          const bool spec = p.batch == 1 && total == total_spec && rg == static_cast<int>(blockIdx.x) &&
                            lp == lp0;
          int entry = 0;
          if (lane < n) {
            entry = spec ? spec_entry : bt_row[lp + lane];
            if (entry < 0 || entry >= p.num_pages) {
              flag_error(p.status, PA_DEV_ERR_PAGE_OOB);
              entry = 0;
            }
          }
          // one stage = kSlots consecutive pages of this sequence (32 is a multiple of kSlots,
          // so the stages line up with the consumers' page groups)
          for (int i = 0; i < n; i += kSlots) {
            const int n_st = min(kSlots, n - i);
            int page[kSlots];
#pragma unroll
            for (int j = 0; j < kSlots; ++j) page[j] = __shfl_sync(0xffffffffu, entry, min(i + j, 31));
            if (lane == 0) {
              if (starve) {
                starve = false;  // this stage stays empty: its consumers' waits run out
              } else if (!mbar_wait_bounded(&s.empty[stage], phase ^ 1u, p.wait_limit_ns)) {
                flag_error(p.status, PA_DEV_ERR_TIMEOUT);
                ok = false;
              } else {
                mbar_arrive_expect_tx(&s.full[stage], 2 * n_st * kPageBytes);
#pragma unroll
                for (int j = 0; j < kSlots; ++j) {
                  if (j < n_st) {
                    bulk_g2s(s.kv[stage][0] + j * kPageBytes,
                             p.k_pool + static_cast<int64_t>(page[j]) * kPageBytes, kPageBytes,
                             &s.full[stage]);
                    bulk_g2s(s.kv[stage][1] + j * kPageBytes,
                             p.v_pool + static_cast<int64_t>(page[j]) * kPageBytes, kPageBytes,
                             &s.full[stage]);
                  }
                }
                ++issued;
              }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
          }
        }
      }
    }
    // Do not leave while copies into this CTA's shared memory may still be landing (the last
    // `issued` ring positions; a stage left empty by the test hook is the first one, never
    // among them).
    if (lane == 0) {
      int st = stage;
      uint32_t ph = phase;
      for (int k = 0; k < min(issued, kStages); ++k) {
        if (--st < 0) { st = kStages - 1; ph ^= 1u; }
        if (!mbar_wait_bounded(&s.full[st], ph, p.wait_limit_ns)) flag_error(p.status, PA_DEV_ERR_TIMEOUT);
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  // Warp w serves (KV head, page slot) pair w % 8 and tokens 8 * (w / 8) .. +7 of each page; the
  // two warps of a pair keep their own running max, sums and accumulators and are merged once
  // per (sequence, range) through shared memory.
  const int pair = warp & 7;
  const int half = warp >> 3;
  const int g = pair % kHkvT;   // KV head
  const int slot = pair / kHkvT;  // page of each stage
  const int c = lane & 15;      // dims 8c .. 8c+7
  const int th = lane >> 4;     // tokens tok0 .. tok0+3 of each page
  const int tok0 = 8 * half + 4 * th;
  // after the scatter lane c owns the score of token tok0 + (c & 3), head c >> 2 & 1 (lanes c and
  // c ^ 8 hold the same one)
  const bool hi_head = (c & 4) != 0;
  int stage = 0;
  uint32_t phase = 0;
  uint32_t xphase = 0;  // hand-offs between the two warps of the pair so far, mod 2

  for (int rg = blockIdx.x; rg < n_ranges; rg += gridDim.x) {
    const int P0 = rg * W, P1 = min(total, P0 + W);
    const int b_first = find_seq(s.prefix, p.batch, P0);
    for (int b = b_first; b < p.batch && s.prefix[b] < P1; ++b) {
      const int n_pages = s.prefix[b + 1] - s.prefix[b];
      const int lp0 = max(P0, s.prefix[b]) - s.prefix[b];
      const int lp1 = min(P1, s.prefix[b + 1]) - s.prefix[b];
      if (lp0 >= lp1) continue;
      const int L = clamp_len(p, b, false);

      // q of the two heads in this lane's order: its own head (the one whose score it keeps
      // after the scatter) first
      float2 qa[4], qb[4];
      {
        const uint16_t* qrow = p.q + (static_cast<int64_t>(b) * kHqT + 2 * g) * kHeadDim + 8 * c;
        const uint4 ra = *reinterpret_cast<const uint4*>(qrow + (hi_head ? kHeadDim : 0));
        const uint4 rb = *reinterpret_cast<const uint4*>(qrow + (hi_head ? 0 : kHeadDim));
        const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          qa[i] = make_float2(bf16lo(wa[i]) * p.scale_log2, bf16hi(wa[i]) * p.scale_log2);
          qb[i] = make_float2(bf16lo(wb[i]) * p.scale_log2, bf16hi(wb[i]) * p.scale_log2);
        }
      }
      float2 acc_a[4], acc_b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc_a[i] = acc_b[i] = make_float2(0.f, 0.f);
      float m_a = -CUDART_INF_F, m_b = -CUDART_INF_F;  // max used for the exponent, per head
      float l_part = 0.f;                               // this lane's share of its head's sum

      bool all_ok = true;
      for (int lp0s = lp0; lp0s < lp1; lp0s += kSlots) {
        const int lp = lp0s + slot;               // this warp's page of the stage
        const bool active = lp < lp1;             // (a stage may hold fewer than kSlots pages)
        const int n_valid = active ? min(kPage, L - lp * kPage) : 0;
        bool ok = true;
        if (!mbar_wait_bounded(&s.full[stage], phase, p.wait_limit_ns)) {
          flag_error(p.status, PA_DEV_ERR_TIMEOUT);
          ok = false;
        }
        if (!__all_sync(0xffffffffu, ok)) {
          all_ok = false;
          break;
        }
        const uint8_t* Ks = s.kv[stage][0] + slot * kPageBytes + g * (kHeadDim * 2) + c * 16;
        const uint8_t* Vs = s.kv[stage][1] + slot * kPageBytes + g * (kHeadDim * 2) + c * 16;
        // One page of this warp's tokens; kFull: all of them are keys (every page but a sequence's
        // last), so no token is masked or skipped.
        auto page = [&](auto full_tag) {
          constexpr bool kFull = decltype(full_tag)::value;
          // ---- scores: partial dot products over this lane's 8 dims, for 4 tokens x 2 heads.
          //      Register i holds value k = i ^ (c & 7) (k = head * 4 + token, head 0 = 2g): the
          //      lane visits its tokens as j ^ (c & 3) and its own head first, so that every lane
          //      keeps the low half of its values and sends the high half in each scatter round.
          float v[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 kr = lds128(Ks + (tok0 + (j ^ (c & 3))) * kTokenBytes);
            const float2 k0 = make_float2(bf16lo(kr.x), bf16hi(kr.x));
            const float2 k1 = make_float2(bf16lo(kr.y), bf16hi(kr.y));
            const float2 k2 = make_float2(bf16lo(kr.z), bf16hi(kr.z));
            const float2 k3 = make_float2(bf16lo(kr.w), bf16hi(kr.w));
            float2 sa = mul2(qa[0], k0), sb = mul2(qb[0], k0);
            sa = fma2(qa[1], k1, sa); sb = fma2(qb[1], k1, sb);
            sa = fma2(qa[2], k2, sa); sb = fma2(qb[2], k2, sb);
            sa = fma2(qa[3], k3, sa); sb = fma2(qb[3], k3, sb);
            v[j] = sa.x + sa.y;
            v[4 + j] = sb.x + sb.y;
          }
          // ---- reduce-scatter over lanes c & 7 of the half-warp (register i of lane c and
          //      register w + i of lane c ^ w hold the same value), then add the other 8 dims'
          //      lanes: lane c keeps the full score of value c & 7 (token tok0 + (c & 3), head
          //      (c >> 2) & 1)
#pragma unroll
          for (int w = 4; w >= 1; w >>= 1) {
#pragma unroll
            for (int i = 0; i < w; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[w + i], w);
          }
          v[0] += __shfl_xor_sync(0xffffffffu, v[0], 8);
          const float sc = (kFull || tok0 + (c & 3) < n_valid) ? v[0] : -CUDART_INF_F;

          // ---- page max per head over this warp's 8 tokens (one warp-wide max reduction per
          //      head), lazily moved running max
          const float pmax_a = warp_max(hi_head ? -CUDART_INF_F : sc);
          const float pmax_b = warp_max(hi_head ? sc : -CUDART_INF_F);
          if (pmax_a > m_a + kRescaleThreshold || pmax_b > m_b + kRescaleThreshold) {
            const float na = fmaxf(m_a, pmax_a), nb = fmaxf(m_b, pmax_b);
            const float al_a = (m_a == -CUDART_INF_F) ? 0.f : fast_exp2(m_a - na);
            const float al_b = (m_b == -CUDART_INF_F) ? 0.f : fast_exp2(m_b - nb);
            const float2 fa = make_float2(al_a, al_a), fb = make_float2(al_b, al_b);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc_a[i] = mul2(acc_a[i], fa);
              acc_b[i] = mul2(acc_b[i], fb);
            }
            l_part *= hi_head ? al_b : al_a;
            m_a = na;
            m_b = nb;
          }
          // (a warp may have seen only masked tokens so far when its half of a partial page is
          // empty: its max is still -inf and the probability is 0; on a full page the max is
          // finite by now)
          const float mh = hi_head ? m_b : m_a;
          const float pr = (!kFull && sc == -CUDART_INF_F) ? 0.f : fast_exp2(sc - mh);
          l_part += pr;

          // ---- hand probabilities to the lanes that own the V dims, each stored twice (the
          //      paired FMAs take it as both halves): p2[th * 8 + head * 4 + j]
          if (c < 8) s.p2[warp][th * 8 + c] = make_float2(pr, pr);
          __syncwarp();
          float2 ppa[4], ppb[4];
#pragma unroll
          for (int j = 0; j < 4; j += 2) {
            const float4 a4 = *reinterpret_cast<const float4*>(&s.p2[warp][th * 8 + j]);
            const float4 b4 = *reinterpret_cast<const float4*>(&s.p2[warp][th * 8 + 4 + j]);
            ppa[j] = make_float2(a4.x, a4.y);
            ppa[j + 1] = make_float2(a4.z, a4.w);
            ppb[j] = make_float2(b4.x, b4.y);
            ppb[j + 1] = make_float2(b4.z, b4.w);
          }

          // ---- o += p v over this lane's 4 tokens (invalid slots of a partial page skipped)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (kFull || tok0 + j < n_valid) {
              const uint4 vr = lds128(Vs + (tok0 + j) * kTokenBytes);
              const float2 v0 = make_float2(bf16lo(vr.x), bf16hi(vr.x));
              const float2 v1 = make_float2(bf16lo(vr.y), bf16hi(vr.y));
              const float2 v2 = make_float2(bf16lo(vr.z), bf16hi(vr.z));
              const float2 v3 = make_float2(bf16lo(vr.w), bf16hi(vr.w));
              acc_a[0] = fma2(v0, ppa[j], acc_a[0]); acc_b[0] = fma2(v0, ppb[j], acc_b[0]);
              acc_a[1] = fma2(v1, ppa[j], acc_a[1]); acc_b[1] = fma2(v1, ppb[j], acc_b[1]);
              acc_a[2] = fma2(v2, ppa[j], acc_a[2]); acc_b[2] = fma2(v2, ppb[j], acc_b[2]);
              acc_a[3] = fma2(v3, ppa[j], acc_a[3]); acc_b[3] = fma2(v3, ppb[j], acc_b[3]);
            }
          }
        };
        if (n_valid == kPage) {
          page(std::true_type{});
        } else if (active) {
          page(std::false_type{});
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.empty[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!all_ok) return;

      // ---- finish this warp's half: sums over its 8 tokens (lanes c and c ^ 8 hold the same
      //      probabilities, so they are not added together) and over the two token quarters
      float l_m = l_part;
      l_m += __shfl_xor_sync(0xffffffffu, l_m, 1);
      l_m += __shfl_xor_sync(0xffffffffu, l_m, 2);
      l_m += __shfl_xor_sync(0xffffffffu, l_m, 16);
      const float l_o = __shfl_xor_sync(0xffffffffu, l_m, 4);
      float l_a = hi_head ? l_o : l_m;
      float l_b = hi_head ? l_m : l_o;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc_a[i].x += __shfl_xor_sync(0xffffffffu, acc_a[i].x, 16);
        acc_a[i].y += __shfl_xor_sync(0xffffffffu, acc_a[i].y, 16);
        acc_b[i].x += __shfl_xor_sync(0xffffffffu, acc_b[i].x, 16);
        acc_b[i].y += __shfl_xor_sync(0xffffffffu, acc_b[i].y, 16);
      }
      // lanes 0..15 finish head 2g, lanes 16..31 head 2g+1
      const int head = 2 * g + th;
      float m_h = th ? m_b : m_a;
      float l_h = th ? l_b : l_a;
      float o[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = th ? acc_b[i] : acc_a[i];
        o[2 * i] = a.x;
        o[2 * i + 1] = a.y;
      }

      // ---- the second half hands its (max, sum, accumulator) to the first, which merges them
      bool xok = true;
      if (half == 1) {
        if (!mbar_wait_bounded(&s.xempty[pair], xphase ^ 1u, p.wait_limit_ns)) xok = false;
        if (xok) {
          float4* dst = reinterpret_cast<float4*>(s.xo[pair][lane]);
          dst[0] = make_float4(o[0], o[1], o[2], o[3]);
          dst[1] = make_float4(o[4], o[5], o[6], o[7]);
          if (c == 0) {
            s.xm[pair][th] = m_h;
            s.xl[pair][th] = l_h;
          }
          mbar_arrive(&s.xfull[pair]);
        }
      } else {
        if (!mbar_wait_bounded(&s.xfull[pair], xphase, p.wait_limit_ns)) xok = false;
        if (xok) {
          const float4* src = reinterpret_cast<const float4*>(s.xo[pair][lane]);
          const float4 u0 = src[0], u1 = src[1];
          const float m1 = s.xm[pair][th], l1 = s.xl[pair][th];
          mbar_arrive(&s.xempty[pair]);
          const float mm = fmaxf(m_h, m1);
          const float al0 = (m_h == -CUDART_INF_F) ? 0.f : fast_exp2(m_h - mm);
          const float al1 = (m1 == -CUDART_INF_F) ? 0.f : fast_exp2(m1 - mm);
          const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = o[i] * al0 + u[i] * al1;
          l_h = l_h * al0 + l1 * al1;
          m_h = mm;
        }
      }
      xphase ^= 1u;
      if (!__all_sync(0xffffffffu, xok)) {
        flag_error(p.status, PA_DEV_ERR_TIMEOUT);
        return;
      }
      if (half == 1) continue;

      // (with several pages per stage a warp pair may have seen no page of this range: l = 0,
      // and its record is o = 0, lse = -inf, which the merge weighs by 0)
      const float inv = (kSlots == 1 || l_h > 0.f) ? 1.0f / l_h : 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] *= inv;
      const float lse_h = (m_h + log2f(l_h)) * kLn2;
      if (kSlots == 1 && lp0 == 0 && lp1 == n_pages) {
        uint4 w;
        w.x = pack_bf16x2(o[0], o[1]);
        w.y = pack_bf16x2(o[2], o[3]);
        w.z = pack_bf16x2(o[4], o[5]);
        w.w = pack_bf16x2(o[6], o[7]);
        *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(b) * kHqT + head) * kHeadDim + 8 * c) = w;
        if (c == 0 && p.lse != nullptr) p.lse[b * kHqT + head] = lse_h;
      } else {
        // unique per (sequence, range, page slot): the records of sequence b are
        // b * kSlots + k for k = range * kSlots + slot over the ranges that touch it
        const int64_t r = (static_cast<int64_t>(b) + rg) * kSlots + slot;
        float* dst = p.ws_o + (r * kHqT + head) * kHeadDim + 8 * c;
        reinterpret_cast<float4*>(dst)[0] = make_float4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(o[4], o[5], o[6], o[7]);
        if (c == 0) p.ws_lse[r * kHqT + head] = lse_h;
      }
    }
  }
}

// Merge the partial results of sequences that crossed a CTA range boundary; also writes the
// result of empty sequences (o = 0, lse = -inf). One CTA per (sequence, head) of kWarps warps:
// each warp takes every kWarps-th partial (a lane holds 4 of the 128 dims) in one online pass
// with its own running maximum, four partials' loads in flight at a time, and the warps combine
// through shared memory. When sequences are cut into more partials than 4 warps take in one round
// (few sequences over many CTAs), 32 warps are used, so that a sequence split over ~128 CTAs is
// merged in one round of loads (16 warps, three rounds for one sequence over all 152 SMs,
// measured 1-2 us slower per call); beyond 64 partials decode_merge_dims_kernel takes over.
// Launched as a programmatic dependent of decode_splitkv_kernel: its CTAs may start while the
// split kernel is still running and wait (griddepcontrol.wait) until that grid has completed
// and its writes are visible, which hides this launch behind the split kernel.
constexpr int kMergeWarpsSmall = 32, kMergeWarpsLarge = 4;
constexpr int kMergePrefixBatch = 64;  // batches this small: page range computed before the wait

// Sequence b's first and past-last global page and the split's range size W, as the split kernel
// computed them. For a small batch every warp derives them from the lengths with the split
// kernel's own arithmetic while the split kernel still runs; a large batch reads them from the
// workspace after the wait. Contains the grid dependency wait.
__device__ __forceinline__ void merge_seq_range(const DecodeParams& p, int b, int lane, int& p0,
                                                int& p1, int& W) {
  p0 = p1 = W = 0;
  const bool early = p.batch <= kMergePrefixBatch;
  if (early) {
    const int n0 = lane < p.batch ? (clamp_len(p, lane, false) + kPage - 1) / kPage : 0;
    const int n1 = lane + 32 < p.batch ? (clamp_len(p, lane + 32, false) + kPage - 1) / kPage : 0;
    int before = (lane < b ? n0 : 0) + (lane + 32 < b ? n1 : 0), total = n0 + n1;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      total += __shfl_xor_sync(0xffffffffu, total, o);
    }
    const int mine = b < 32 ? __shfl_sync(0xffffffffu, n0, b) : __shfl_sync(0xffffffffu, n1, b - 32);
    p0 = before;
    p1 = before + mine;
    const int base = p.split_pages > 0 ? p.split_pages : kMinPagesPerCta;
    W = max((total + p.max_ranges - 1) / p.max_ranges, base);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!early) {
    p0 = p.ws_prefix[b];
    p1 = p.ws_prefix[b + 1];
    W = p.ws_header[0];
  }
}

template <int kWarps>
__global__ void __launch_bounds__(kWarps * 32) decode_merge_kernel(const DecodeParams p) {
  // the next kernel on the stream may launch now; it waits for this grid before reading anything
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ float red_m[kWarps], red_w[kWarps];
  __shared__ float4 red_o[kWarps][32];
  const int b = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = p.hq, slots = p.stage_pages;
  int p0, p1, W;
  merge_seq_range(p, b, lane, p0, p1, W);
  uint16_t* orow = p.out + (static_cast<int64_t>(b) * hq + h) * kHeadDim + 4 * lane;
  if (p1 == p0) {
    if (warp == 0) {
      *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
      if (lane == 0 && p.lse != nullptr) p.lse[b * hq + h] = -CUDART_INF_F;
    }
    return;
  }
  const int r0 = p0 / W, r1 = (p1 - 1) / W;
  if (r0 == r1 && slots == 1) return;  // finished inside one CTA
  // partials c0 .. c1: record b * slots + c, c = range * slots + page slot
  const int c0 = r0 * slots, c1 = r1 * slots + slots - 1;
  // this warp's partials c0 + warp, c0 + warp + kWarps, ..., four at a time: sum of
  // 2^(lse_c - m) o_c (lse in log2 units) against a running maximum m, rescaled when m moves
  const float* lse_src = p.ws_lse + static_cast<int64_t>(b) * slots * hq + h;
  const float* o_src = p.ws_o + (static_cast<int64_t>(b) * slots * hq + h) * kHeadDim + 4 * lane;
  float m = -CUDART_INF_F, wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = c0 + warp; c <= c1; c += 4 * kWarps) {
    float l2[4];
    float4 o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int cu = c + u * kWarps;
      l2[u] = cu <= c1 ? lse_src[static_cast<int64_t>(cu) * hq] * kLog2e : -CUDART_INF_F;
      o[u] = cu <= c1 ? *reinterpret_cast<const float4*>(o_src + static_cast<int64_t>(cu) * hq * kHeadDim)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float mn = fmaxf(fmaxf(m, fmaxf(l2[0], l2[1])), fmaxf(l2[2], l2[3]));
    const float ms = mn == -CUDART_INF_F ? 0.f : mn;  // no finite partial yet: weights all 0
    const float sc = fast_exp2(m - ms);
    acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
    wsum *= sc;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = fast_exp2(l2[u] - ms);
      wsum += w;
      acc.x += w * o[u].x; acc.y += w * o[u].y; acc.z += w * o[u].z; acc.w += w * o[u].w;
    }
    m = mn;
  }
  red_o[warp][lane] = acc;
  if (lane == 0) {
    red_m[warp] = m;
    red_w[warp] = wsum;
  }
  __syncthreads();
  if (warp != 0) return;
  float M = red_m[0];
#pragma unroll
  for (int k = 1; k < kWarps; ++k) M = fmaxf(M, red_m[k]);
  const float Ms = M == -CUDART_INF_F ? 0.f : M;
  acc = make_float4(0.f, 0.f, 0.f, 0.f);
  wsum = 0.f;
#pragma unroll
  for (int k = 0; k < kWarps; ++k) {
    const float s = fast_exp2(red_m[k] - Ms);  // a warp with no partial has m = -inf: s = 0
    const float4 o = red_o[k][lane];
    acc.x += s * o.x; acc.y += s * o.y; acc.z += s * o.z; acc.w += s * o.w;
    wsum += s * red_w[k];
  }
  const float inv = 1.0f / wsum;
  *reinterpret_cast<uint2*>(orow) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (lane == 0 && p.lse != nullptr) p.lse[b * hq + h] = (M + log2f(wsum)) * kLn2;
}

// The same merge for sequences cut into many partials (more than 64: a few sequences over all
// SMs). Each head's 128 dims are split over kMergeDimParts CTAs of 32 warps, a lane holding one
// dim, so a CTA reads 32 dims of every partial (a quarter of what one CTA per head would), and
// each warp keeps eight partials' loads in flight: up to 256 partials in one round of loads.
constexpr int kMergeDimParts = 4;
constexpr int kMergeManyPartials = 64;
__global__ void __launch_bounds__(kMergeWarpsSmall * 32) decode_merge_dims_kernel(const DecodeParams p) {
  constexpr int kWarps = kMergeWarpsSmall, kInFlight = 8;
  asm volatile("griddepcontrol.launch_dependents;");
  __shared__ float red_m[kWarps], red_w[kWarps];
  __shared__ float red_o[kWarps][32];
  const int b = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = blockIdx.z * 32 + lane;  // this lane's dim
  const int hq = p.hq, slots = p.stage_pages;
  int p0, p1, W;
  merge_seq_range(p, b, lane, p0, p1, W);
  uint16_t* orow = p.out + (static_cast<int64_t>(b) * hq + h) * kHeadDim;
  if (p1 == p0) {
    if (warp == 0) {
      orow[d] = 0;
      if (blockIdx.z == 0 && lane == 0 && p.lse != nullptr) p.lse[b * hq + h] = -CUDART_INF_F;
    }
    return;
  }
  const int r0 = p0 / W, r1 = (p1 - 1) / W;
  if (r0 == r1 && slots == 1) return;  // finished inside one CTA
  const int c0 = r0 * slots, c1 = r1 * slots + slots - 1;
  const float* lse_src = p.ws_lse + static_cast<int64_t>(b) * slots * hq + h;
  const float* o_src = p.ws_o + (static_cast<int64_t>(b) * slots * hq + h) * kHeadDim + d;
  float m = -CUDART_INF_F, wsum = 0.f, acc = 0.f;
  for (int c = c0 + warp; c <= c1; c += kInFlight * kWarps) {
    float l2[kInFlight], o[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int cu = c + u * kWarps;
      l2[u] = cu <= c1 ? lse_src[static_cast<int64_t>(cu) * hq] * kLog2e : -CUDART_INF_F;
      o[u] = cu <= c1 ? o_src[static_cast<int64_t>(cu) * hq * kHeadDim] : 0.f;
    }
    float mn = m;
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) mn = fmaxf(mn, l2[u]);
    const float ms = mn == -CUDART_INF_F ? 0.f : mn;  // no finite partial yet: weights all 0
    const float sc = fast_exp2(m - ms);
    acc *= sc;
    wsum *= sc;
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const float w = fast_exp2(l2[u] - ms);
      wsum += w;
      acc += w * o[u];
    }
    m = mn;
  }
  red_o[warp][lane] = acc;
  if (lane == 0) {
    red_m[warp] = m;
    red_w[warp] = wsum;
  }
  __syncthreads();
  if (warp != 0) return;
  float M = red_m[0];
#pragma unroll
  for (int k = 1; k < kWarps; ++k) M = fmaxf(M, red_m[k]);
  const float Ms = M == -CUDART_INF_F ? 0.f : M;
  float a = 0.f;
  wsum = 0.f;
#pragma unroll
  for (int k = 0; k < kWarps; ++k) {
    const float sk = fast_exp2(red_m[k] - Ms);  // a warp with no partial has m = -inf: s = 0
    a += sk * red_o[k][lane];
    wsum += sk * red_w[k];
  }
  orow[d] = static_cast<uint16_t>(pack_bf16x2(a / wsum, 0.f) & 0xffffu);
  if (blockIdx.z == 0 && lane == 0 && p.lse != nullptr) p.lse[b * hq + h] = (M + log2f(wsum)) * kLn2;
}

// ---------------------------------------------------------------------------------------------
// Short batches in one launch (decode_cluster_kernel). When every (sequence, KV head) pair of
// the batch can have a resident cluster of C CTAs (C a power of two <= 8; see small_path) and
// each CTA then holds few pages, the split above is latency-bound: a prefix pass, a dependent
// block-table load, one page per SM, partials through L2 and a second kernel that waits for the
// first to complete. Here CTA rank c of the cluster of pair (b, g) takes pages
// [cP/C, (c+1)P/C) of sequence b (P = its pages) for KV head g only (two heads, four warps each,
// when the batch has more pairs than resident clusters); its warps take one page each in turn,
// each lane copying its own pieces of the K/V rows of head g into its warp's 3-stage ring
// (16-byte cp.async, two pages in flight ahead of the one computed); the warps combine through
// shared memory, the ranks write their partial (o, max, sum) into rank 0's shared memory
// (distributed shared memory of the cluster) and rank 0 merges them and writes the output.
// ---------------------------------------------------------------------------------------------
constexpr int kSmallWarps = 8;
constexpr int kSmallThreads = kSmallWarps * 32;
constexpr int kSmallMaxCluster = 8;
constexpr int kSmallPreload = 256;  // block-table entries loaded beside the length (Pmax <= this)
constexpr int kSmallMaxPagesPerCta = 64;  // beyond this the full-grid split streams faster

constexpr int kRingStages = 3;                  // pages in flight per warp (incl. the current)
constexpr int kRowBytes = kHeadDim * 2;         // one token's row of one head
constexpr int kSlice = kPage * kRowBytes;       // one page of one head: K (or V) rows

struct SmallSmem {  // dynamic shared memory, 128-byte aligned
  uint8_t ring[kSmallWarps][kRingStages][2][kSlice];  // per warp: its lanes' K and V pieces
  int32_t pages[kSmallPreload];              // the sequence's block-table entries (preloaded)
  float p[kSmallWarps][32];                  // probabilities handed to the V lanes
  float red_o[kSmallWarps][2][kHeadDim];     // per warp: unnormalised o of both heads
  float red_m[kSmallWarps][2], red_l[kSmallWarps][2];
  float slot_o[kSmallMaxCluster][4][kHeadDim];  // rank 0: each rank's partial (query heads)
  float slot_m[kSmallMaxCluster][4], slot_l[kSmallMaxCluster][4];
  uint64_t full;                             // rank 0: the other ranks' partials have landed
};

// kHpc KV heads per CTA (1, or 2 when a batch has more (sequence, KV head) pairs than resident
// clusters allow): warp w serves the CTA's head w / (8 / kHpc).
template <int kHkvT, int kHpc>
__global__ void __launch_bounds__(kSmallThreads, 1) decode_cluster_kernel(const DecodeParams p) {
  static_assert(kHpc == 1 || kHpc == 2, "one or two KV heads per CTA");
  constexpr int kHqT = kGroup * kHkvT;
  constexpr int kWph = kSmallWarps / kHpc;  // warps per KV head
  constexpr int64_t kPageBytes = kPage * kHkvT * kHeadDim * 2;  // K (or V) of one page
  constexpr int kTokenBytes = kHkvT * kHeadDim * 2;             // one token's row in a page
  extern __shared__ __align__(128) uint8_t small_smem_raw[];
  SmallSmem& s = *reinterpret_cast<SmallSmem*>(small_smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t C = cluster_nctarank(), rank = cluster_ctarank();
  const int pair = static_cast<int>(blockIdx.x / C);  // (sequence, group of kHpc KV heads)
  const int b = pair / (kHkvT / kHpc);
  const int g0 = (pair % (kHkvT / kHpc)) * kHpc;      // the CTA's first KV head
  const int hh = warp / kWph, g = g0 + hh;            // this warp's KV head
  if (tid == 0) {
    if (rank == 0) mbar_init(&s.full, (C - 1) * kSmallThreads);
    fence_mbar_init();
  }
  cluster_sync_all();  // rank 0's barrier is initialised before any rank can arrive on it
  // a programmatic dependent of the previous kernel on the stream: nothing it wrote is read
  // before this wait; the next kernel may launch now and waits for this grid's completion
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
  const int pmax = min((p.max_seq_len + kPage - 1) / kPage, p.bt_stride);
  const bool preload = pmax <= kSmallPreload;
  if (preload)
    for (int i = tid; i < pmax; i += kSmallThreads) s.pages[i] = bt_row[i];
  const int L = clamp_len(p, b, rank == 0 && g0 == 0 && tid == 0);
  const int P = (L + kPage - 1) / kPage;
  const int p0 = static_cast<int>(static_cast<int64_t>(rank) * P / C);
  const int p1 = static_cast<int>(static_cast<int64_t>(rank + 1) * P / C);

  // ---- this lane's share of the group's two query rows (dims 8c .. 8c+7), in log2 units
  const int c = lane & 15, th = lane >> 4;
  const bool hi_head = (c & 8) != 0;
  // q of the two heads in this lane's order: its own head (the one whose score it keeps after the
  // scatter) first
  float2 qa[4], qb[4];
  {
    const uint16_t* qrow = p.q + (static_cast<int64_t>(b) * kHqT + 2 * g) * kHeadDim + 8 * c;
    const uint4 ra = *reinterpret_cast<const uint4*>(qrow + (hi_head ? kHeadDim : 0));
    const uint4 rb = *reinterpret_cast<const uint4*>(qrow + (hi_head ? 0 : kHeadDim));
    const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qa[i] = make_float2(bf16lo(wa[i]) * p.scale_log2, bf16hi(wa[i]) * p.scale_log2);
      qb[i] = make_float2(bf16lo(wb[i]) * p.scale_log2, bf16hi(wb[i]) * p.scale_log2);
    }
  }
  __syncthreads();  // the preloaded block-table entries

  auto cp_async16 = [](void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
  };
  auto page_entry = [&](int lp) {
    int e = preload ? s.pages[lp] : bt_row[lp];
    if (e < 0 || e >= p.num_pages) {
      if (lane == 0) flag_error(p.status, PA_DEV_ERR_PAGE_OOB);
      e = 0;
    }
    return e;
  };
  // This warp's pages are p0 + wl, p0 + wl + kWph, ...; its k-th page goes to ring stage
  // k % kRingStages. Each lane copies (16-byte cp.async) exactly the K and V pieces it reads
  // later, tokens th*8 .. th*8+7, dims 8c .. 8c+7, into slots of its own, so no lane waits for
  // another: one commit group per page, and a wait for all but the pages still ahead.
  const int wl = warp % kWph;
  const int n_my = p1 - p0 > wl ? (p1 - p0 - wl + kWph - 1) / kWph : 0;
  const int64_t lane_off = static_cast<int64_t>(th * 8) * kTokenBytes + g * kRowBytes + c * 16;
  auto slot = [&](int st, int kv, int j) {
    return s.ring[warp][st][0] + ((kv * 8 + j) * 32 + lane) * 16;
  };
  auto issue = [&](int k) {
    const int e = page_entry(p0 + wl + k * kWph);
    const int st = k % kRingStages;
    const uint8_t* kp = p.k_pool + static_cast<int64_t>(e) * kPageBytes + lane_off;
    const uint8_t* vp = p.v_pool + static_cast<int64_t>(e) * kPageBytes + lane_off;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      cp_async16(slot(st, 0, j), kp + j * kTokenBytes);
      cp_async16(slot(st, 1, j), vp + j * kTokenBytes);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  for (int k = 0; k < n_my && k < kRingStages; ++k) issue(k);

  float2 acc_a[4], acc_b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc_a[i] = acc_b[i] = make_float2(0.f, 0.f);
  float m_a = -CUDART_INF_F, m_b = -CUDART_INF_F;  // max used for the exponent, per head
  float l_part = 0.f;                               // this lane's share of its head's sum
  for (int k = 0; k < n_my; ++k) {
    const int st = k % kRingStages, lp = p0 + wl + k * kWph;
    // page k has landed once at most the pages issued after it are still pending
    const int ahead = min(n_my - 1 - k, kRingStages - 1);
    if (ahead >= 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
    else if (ahead == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else asm volatile("cp.async.wait_group 0;" ::: "memory");
    const int n_valid = min(kPage, L - lp * kPage);
    // ---- scores: partial dot products over this lane's 8 dims, for 8 tokens x 2 heads.
    //      Register i holds value k = i ^ (c & 15) (k = head * 8 + token, head 0 = 2g): the lane
    //      visits its tokens as j ^ (c & 7) and its own head first, so that every lane keeps the
    //      low half of its values and sends the high half in each scatter round.
    float v[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 kr = lds128(slot(st, 0, j ^ (c & 7)));
      const float2 k0 = make_float2(bf16lo(kr.x), bf16hi(kr.x));
      const float2 k1 = make_float2(bf16lo(kr.y), bf16hi(kr.y));
      const float2 k2 = make_float2(bf16lo(kr.z), bf16hi(kr.z));
      const float2 k3 = make_float2(bf16lo(kr.w), bf16hi(kr.w));
      float2 sa = mul2(qa[0], k0), sb = mul2(qb[0], k0);
      sa = fma2(qa[1], k1, sa); sb = fma2(qb[1], k1, sb);
      sa = fma2(qa[2], k2, sa); sb = fma2(qb[2], k2, sb);
      sa = fma2(qa[3], k3, sa); sb = fma2(qb[3], k3, sb);
      v[j] = sa.x + sa.y;
      v[8 + j] = sb.x + sb.y;
    }
    // ---- reduce-scatter over the 16 lanes of the half-warp (register i of lane c and register
    //      w + i of lane c ^ w hold the same value): lane c keeps the full score of token
    //      th*8 + (c & 7), head (c >> 3)
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
      for (int i = 0; i < w; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[w + i], w);
    }
    const float sc = (th * 8 + (c & 7) < n_valid) ? v[0] : -CUDART_INF_F;
    // ---- page max per head (one warp-wide max reduction per head), lazily moved running max
    //      (at least one key of a page is valid)
    const float pmax_a = warp_max(hi_head ? -CUDART_INF_F : sc);
    const float pmax_b = warp_max(hi_head ? sc : -CUDART_INF_F);
    if (pmax_a > m_a + kRescaleThreshold || pmax_b > m_b + kRescaleThreshold) {
      const float na = fmaxf(m_a, pmax_a), nb = fmaxf(m_b, pmax_b);
      const float al_a = (m_a == -CUDART_INF_F) ? 0.f : fast_exp2(m_a - na);
      const float al_b = (m_b == -CUDART_INF_F) ? 0.f : fast_exp2(m_b - nb);
      const float2 fa = make_float2(al_a, al_a), fb = make_float2(al_b, al_b);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc_a[i] = mul2(acc_a[i], fa);
        acc_b[i] = mul2(acc_b[i], fb);
      }
      l_part *= hi_head ? al_b : al_a;
      m_a = na;
      m_b = nb;
    }
    const float pr = fast_exp2(sc - (hi_head ? m_b : m_a));
    l_part += pr;
    // ---- hand probabilities to the lanes that own the V dims
    s.p[warp][lane] = pr;
    __syncwarp();
    const float4 pa0 = *reinterpret_cast<const float4*>(&s.p[warp][th * 16 + 0]);
    const float4 pa1 = *reinterpret_cast<const float4*>(&s.p[warp][th * 16 + 4]);
    const float4 pb0 = *reinterpret_cast<const float4*>(&s.p[warp][th * 16 + 8]);
    const float4 pb1 = *reinterpret_cast<const float4*>(&s.p[warp][th * 16 + 12]);
    __syncwarp();  // read before the next page overwrites them
    const float pav[8] = {pa0.x, pa0.y, pa0.z, pa0.w, pa1.x, pa1.y, pa1.z, pa1.w};
    const float pbv[8] = {pb0.x, pb0.y, pb0.z, pb0.w, pb1.x, pb1.y, pb1.z, pb1.w};
    // ---- o += p v over this lane's 8 tokens (invalid slots of a partial page skipped)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (th * 8 + j < n_valid) {
        const uint4 vr = lds128(slot(st, 1, j));
        const float2 ppa = make_float2(pav[j], pav[j]);
        const float2 ppb = make_float2(pbv[j], pbv[j]);
        const float2 v0 = make_float2(bf16lo(vr.x), bf16hi(vr.x));
        const float2 v1 = make_float2(bf16lo(vr.y), bf16hi(vr.y));
        const float2 v2 = make_float2(bf16lo(vr.z), bf16hi(vr.z));
        const float2 v3 = make_float2(bf16lo(vr.w), bf16hi(vr.w));
        acc_a[0] = fma2(v0, ppa, acc_a[0]); acc_b[0] = fma2(v0, ppb, acc_b[0]);
        acc_a[1] = fma2(v1, ppa, acc_a[1]); acc_b[1] = fma2(v1, ppb, acc_b[1]);
        acc_a[2] = fma2(v2, ppa, acc_a[2]); acc_b[2] = fma2(v2, ppb, acc_b[2]);
        acc_a[3] = fma2(v3, ppa, acc_a[3]); acc_b[3] = fma2(v3, ppb, acc_b[3]);
      }
    }
    // this lane has read its slots of the stage: refill them with the page kRingStages ahead
    if (k + kRingStages < n_my) issue(k + kRingStages);
  }

  // ---- this warp's (m, sum, unnormalised o) per head: lanes 0..15 head 2g, 16..31 head 2g+1
  float l_m = l_part;
  l_m += __shfl_xor_sync(0xffffffffu, l_m, 1);
  l_m += __shfl_xor_sync(0xffffffffu, l_m, 2);
  l_m += __shfl_xor_sync(0xffffffffu, l_m, 4);
  l_m += __shfl_xor_sync(0xffffffffu, l_m, 16);
  const float l_o = __shfl_xor_sync(0xffffffffu, l_m, 8);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc_a[i].x += __shfl_xor_sync(0xffffffffu, acc_a[i].x, 16);
    acc_a[i].y += __shfl_xor_sync(0xffffffffu, acc_a[i].y, 16);
    acc_b[i].x += __shfl_xor_sync(0xffffffffu, acc_b[i].x, 16);
    acc_b[i].y += __shfl_xor_sync(0xffffffffu, acc_b[i].y, 16);
  }
  {
    float* dst = &s.red_o[warp][th][8 * c];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = th ? acc_b[i] : acc_a[i];
      dst[2 * i] = a.x;
      dst[2 * i + 1] = a.y;
    }
    if (c == 0) {
      s.red_m[warp][th] = th ? m_b : m_a;
      s.red_l[warp][th] = th ? (hi_head ? l_m : l_o) : (hi_head ? l_o : l_m);
    }
  }
  __syncthreads();

  // ---- this CTA's partial per query head: thread tid + 256k takes dim d of the CTA's query head
  //      qh = 2 hh + h2 (head 2 g0 + qh), combining the warps that served KV head g0 + hh
  float o[kHpc], l[kHpc], M[kHpc];
#pragma unroll
  for (int k = 0; k < kHpc; ++k) {
    const int qh = (tid + k * kSmallThreads) >> 7, d = tid & (kHeadDim - 1);
    const int wh = qh >> 1, h2 = qh & 1;
    float m = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kWph; ++w) m = fmaxf(m, s.red_m[wh * kWph + w][h2]);
    const float ms = m == -CUDART_INF_F ? 0.f : m;  // a warp without pages weighs 0
    float oo = 0.f, ll = 0.f;
#pragma unroll
    for (int w = 0; w < kWph; ++w) {
      const int ww = wh * kWph + w;
      const float sw = fast_exp2(s.red_m[ww][h2] - ms);
      oo += sw * s.red_o[ww][h2][d];
      ll += sw * s.red_l[ww][h2];
    }
    o[k] = oo;
    l[k] = ll;
    M[k] = m;
  }
  if (C > 1) {
    if (rank != 0) {
      // into rank 0's slot for this rank, then one arrive per thread on rank 0's barrier
#pragma unroll
      for (int k = 0; k < kHpc; ++k) {
        const int qh = (tid + k * kSmallThreads) >> 7, d = tid & (kHeadDim - 1);
        st_cluster_f32(map_to_rank(&s.slot_o[rank][qh][d], 0), o[k]);
        if (d == 0) {
          st_cluster_f32(map_to_rank(&s.slot_m[rank][qh], 0), M[k]);
          st_cluster_f32(map_to_rank(&s.slot_l[rank][qh], 0), l[k]);
        }
      }
      mbar_arrive_cluster(map_to_rank(&s.full, 0));
      return;
    }
    if (!mbar_wait_cluster_bounded(&s.full, 0, p.wait_limit_ns)) {
      flag_error(p.status, PA_DEV_ERR_TIMEOUT);
      return;
    }
#pragma unroll
    for (int k = 0; k < kHpc; ++k) {
      const int qh = (tid + k * kSmallThreads) >> 7, d = tid & (kHeadDim - 1);
      float mc = M[k];
      for (uint32_t r = 1; r < C; ++r) mc = fmaxf(mc, s.slot_m[r][qh]);
      const float ms = mc == -CUDART_INF_F ? 0.f : mc;
      const float s0 = fast_exp2(M[k] - ms);
      float oo = o[k] * s0, ll = l[k] * s0;
      for (uint32_t r = 1; r < C; ++r) {
        const float sr = fast_exp2(s.slot_m[r][qh] - ms);
        oo += sr * s.slot_o[r][qh][d];
        ll += sr * s.slot_l[r][qh];
      }
      o[k] = oo;
      l[k] = ll;
      M[k] = mc;
    }
  }
  // an empty sequence has l = 0, M = -inf: o = 0 and lse = -inf
#pragma unroll
  for (int k = 0; k < kHpc; ++k) {
    const int qh = (tid + k * kSmallThreads) >> 7, d = tid & (kHeadDim - 1);
    const int head = 2 * g0 + qh;
    const float inv = l[k] > 0.f ? 1.0f / l[k] : 0.f;
    p.out[(static_cast<int64_t>(b) * kHqT + head) * kHeadDim + d] =
        static_cast<uint16_t>(pack_bf16x2(o[k] * inv, 0.f) & 0xffffu);
    if (d == 0 && p.lse != nullptr) p.lse[b * kHqT + head] = (M[k] + log2f(l[k])) * kLn2;
  }
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t header, prefix, lse, o, total;
};

// Records: (batch + ranges) x pages per stage, each [Hq] lse and [Hq][128] o. For a call with
// Hkv < 8 KV heads there are 8 / Hkv page slots per range but only 2 Hkv query heads, so the
// workspace is never larger than the decoder's.
WsLayout ws_layout(int batch, int64_t ranges, int hkv) {
  WsLayout w;
  const int hq = kGroup * hkv, slots = kHkv / hkv;
  const size_t records = (static_cast<size_t>(batch) + static_cast<size_t>(ranges)) * slots;
  w.header = 0;
  w.prefix = 256;
  w.lse = align_up(w.prefix + sizeof(int32_t) * (batch + 1), 256);
  w.o = align_up(w.lse + sizeof(float) * records * hq, 256);
  w.total = align_up(w.o + sizeof(float) * records * hq * kHeadDim, 256);
  return w;
}

// With an explicit split size, at most this many ranges per SM (the split is raised beyond
// that, which bounds the workspace: 64 ranges x 152 SMs x 8 KB of partials = 80 MB).
constexpr int64_t kMaxRangesPerSm = 64;

// Launch plan of one call, from host arguments only (so that it can be captured in a graph).
struct DecodePlan {
  int grid;          // CTAs
  int split_pages;   // 0 = an equal share per CTA
  int max_ranges;    // ranges of the launch (records = batch + max_ranges)
  int64_t ws_ranges; // ranges the workspace must hold records for
};

DecodePlan decode_plan(int batch, int max_seq_len, int split_tokens, int sm_grid) {
  DecodePlan d;
  // pages the batch can have at most
  const int64_t page_bound = std::max<int64_t>(
      1, static_cast<int64_t>(batch) * ((static_cast<int64_t>(max_seq_len) + kPage - 1) / kPage));
  if (split_tokens == 0) {
    // one CTA per SM, but no more CTAs than the batch can have pages (a short batch then
    // launches only the CTAs that get work); the workspace size does not depend on max_seq_len
    d.grid = static_cast<int>(std::min<int64_t>(sm_grid, page_bound));
    d.split_pages = 0;
    d.max_ranges = d.grid;
    d.ws_ranges = sm_grid;
  } else {
    const int64_t pages = (static_cast<int64_t>(split_tokens) + kPage - 1) / kPage;
    const int64_t ranges = std::min<int64_t>((page_bound + pages - 1) / pages, kMaxRangesPerSm * sm_grid);
    d.split_pages = static_cast<int>(pages);
    d.max_ranges = static_cast<int>(ranges);
    d.grid = static_cast<int>(std::min<int64_t>(sm_grid, ranges));
    d.ws_ranges = ranges;
  }
  return d;
}

// Clusters of decode_cluster_kernel of size C (1, 2, 4 or 8) that the current device can hold
// at once, from the occupancy calculator (0 if it cannot say: the split path then serves the
// call); cached per device and size.
// The single-launch kernels' shared memory is above the 48 KB default: allowed once per device
// for every instance (under the capacity cache's lock).
bool configure_small_kernels_locked(int dev) {
  static bool done[64] = {};
  if (done[dev]) return true;
  const int bytes = static_cast<int>(sizeof(SmallSmem));
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(decode_cluster_kernel<8, 1>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_cluster_kernel<8, 2>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_cluster_kernel<4, 1>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_cluster_kernel<4, 2>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_cluster_kernel<2, 1>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_cluster_kernel<2, 2>, a, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_cluster_kernel<1, 1>, a, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  done[dev] = true;
  return true;
}

int small_cluster_capacity(int C, int hpc) {
  static std::mutex mu;
  static int cache[64][2][4];
  static bool known[64][2][4] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int k = C == 1 ? 0 : (C == 2 ? 1 : (C == 4 ? 2 : 3)), h = hpc == 2 ? 1 : 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!configure_small_kernels_locked(dev)) return 0;  // the split path serves the call
  if (!known[dev][h][k]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C * 256));
    cfg.blockDim = dim3(kSmallThreads);
    cfg.dynamicSmemBytes = sizeof(SmallSmem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    // the instances for other KV-head counts use the same registers and shared memory
    const cudaError_t e = hpc == 2
        ? cudaOccupancyMaxActiveClusters(&n, decode_cluster_kernel<8, 2>, &cfg)
        : cudaOccupancyMaxActiveClusters(&n, decode_cluster_kernel<8, 1>, &cfg);
    if (e != cudaSuccess) {
      cudaGetLastError();  // not sticky: clear it; the split path serves this call, and the
      return 0;            // query is repeated on the next call
    }
    cache[dev][h][k] = n;
    known[dev][h][k] = true;
  }
  return cache[dev][h][k];
}

// Test hook (pa_debug_decode_starve): the calling thread's next launches leave one ring stage
// of CTA 0 empty and bound every wait by 1 ms.
thread_local bool g_debug_starve = false;

// How a call is served: the single-launch path with clusters of C CTAs of hpc KV heads each, or
// (C = 0) the split path (split kernel + merge). The single launch is taken with the automatic
// split when every (sequence, group of hpc KV heads) can have a resident cluster of C CTAs (the
// largest such C <= 8; one head per CTA first, two if the batch has more pairs than that) and a
// CTA then holds at most kSmallMaxPagesPerCta pages; the bounded-wait test hook keeps the split
// path, whose ring it exercises.
struct SmallPath {
  int C = 0, hpc = 0;
};
SmallPath small_path(int hkv, int batch, int max_seq_len, int split_tokens) {
  SmallPath r;
  if (split_tokens != 0 || g_debug_starve || batch <= 0) return r;
  const int64_t pmax = (static_cast<int64_t>(max_seq_len) + kPage - 1) / kPage;
  for (int hpc = 1; hpc <= 2 && hkv % hpc == 0; hpc *= 2) {
    const int64_t pairs = static_cast<int64_t>(batch) * (hkv / hpc);
    // the largest cluster size whose clusters can all be resident at once (a cluster must fit
    // in one GPC, so this can be fewer than SMs / C)
    int C = kSmallMaxCluster;
    while (C > 1 && pairs > small_cluster_capacity(C, hpc)) C >>= 1;
    if (pairs <= small_cluster_capacity(C, hpc) && (pmax + C - 1) / C <= kSmallMaxPagesPerCta) {
      r.C = C;
      r.hpc = hpc;
      return r;
    }
  }
  return r;
}
constexpr uint64_t kDebugWaitLimitNs = 1000000ull;

}  // namespace

int decode_grid_size() { return sm_count_current_device(); }

}  // namespace pa

extern "C" size_t pa_decode_workspace_size(pa_dims dims, int32_t batch, int32_t max_seq_len,
                                           int32_t split_tokens) {
  if (!pa::gqa_dims_supported(dims) || batch < 0 || max_seq_len < 0 || split_tokens < 0) return 0;
  const int sm_grid = pa::decode_grid_size();
  if (sm_grid <= 0) return 0;
  return pa::ws_layout(batch, pa::decode_plan(batch, max_seq_len, split_tokens, sm_grid).ws_ranges,
                       dims.num_kv_heads).total;
}

extern "C" pa_status pa_debug_decode_starve(int32_t enable) {
  pa::g_debug_starve = enable != 0;
  return PA_OK;
}

extern "C" int32_t pa_decode_kernels_per_call(pa_dims dims, int32_t batch, int32_t max_seq_len,
                                              int32_t split_tokens) {
  if (!pa::gqa_dims_supported(dims) || batch <= 0 || max_seq_len < 0 || split_tokens < 0)
    return 0;
  return pa::small_path(dims.num_kv_heads, batch, max_seq_len, split_tokens).C > 0 ? 1 : 2;
}

namespace pa {
namespace {
// attn_decode_paged with a cap on the grid (max_ctas > 0; 0 = one CTA per SM)
pa_status decode_call(pa_dims dims, const void* q, const void* k_pool, const void* v_pool,
                      int64_t num_pages, const int32_t* block_table, int32_t bt_stride,
                      const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                      float softmax_scale, int32_t split_tokens, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, int32_t* status,
                      pa_stream_t stream, int32_t max_ctas) {
  if (!gqa_dims_supported(dims)) return PA_ERR_UNSUPPORTED;
  if (batch < 0 || batch > kMaxBatch || bt_stride <= 0 || num_pages <= 0 || max_seq_len < 0 ||
      max_seq_len > 131072 || !(softmax_scale == softmax_scale) || split_tokens < 0)
    return PA_ERR_INVALID_ARG;
  if (batch == 0) return PA_OK;
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out || !workspace)
    return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pool) |
       reinterpret_cast<uintptr_t>(v_pool) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return PA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PA_ERR_INVALID_ARG;
  const int full_grid = decode_grid_size();
  if (full_grid <= 0) return PA_ERR_CUDA;
  const int sm_grid = max_ctas > 0 ? std::min(full_grid, static_cast<int>(max_ctas)) : full_grid;
  const DecodePlan plan = decode_plan(batch, max_seq_len, split_tokens, sm_grid);
  const int hkv = dims.num_kv_heads;
  if (workspace_bytes < ws_layout(batch, plan.ws_ranges, hkv).total) return PA_ERR_WORKSPACE_TOO_SMALL;
  const WsLayout w = ws_layout(batch, plan.max_ranges, hkv);

  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    const int smem = static_cast<int>(sizeof(DecodeSmem));
    cudaError_t e = cudaFuncSetAttribute(decode_splitkv_kernel<8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_splitkv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_splitkv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_splitkv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return record_cuda_error(e, "cudaFuncSetAttribute(decode)");
    // the merge kernel uses no shared memory; giving it the split kernel's carveout keeps the
    // SMs from reconfiguring shared memory / L1 between the two launches of every call
    e = cudaFuncSetAttribute(decode_merge_kernel<kMergeWarpsSmall>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_merge_kernel<kMergeWarpsLarge>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_merge_dims_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return record_cuda_error(e, "cudaFuncSetAttribute(decode merge)");
    configured_device = dev;
  }

  DecodeParams p;
  p.hq = dims.num_q_heads;
  p.stage_pages = kHkv / hkv;
  p.q = static_cast<const uint16_t*>(q);
  p.k_pool = static_cast<const uint8_t*>(k_pool);
  p.v_pool = static_cast<const uint8_t*>(v_pool);
  p.num_pages = num_pages;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.max_seq_len = max_seq_len;
  p.split_pages = plan.split_pages;
  p.max_ranges = plan.max_ranges;
  p.scale_log2 = softmax_scale * kLog2e;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.ws_header = reinterpret_cast<int32_t*>(ws + w.header);
  p.ws_prefix = reinterpret_cast<int32_t*>(ws + w.prefix);
  p.ws_lse = reinterpret_cast<float*>(ws + w.lse);
  p.ws_o = reinterpret_cast<float*>(ws + w.o);
  p.status = status;
  p.wait_limit_ns = g_debug_starve ? kDebugWaitLimitNs : kWaitLimitNs;
  p.starve = g_debug_starve ? 1 : 0;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // Short batches in one launch (decode_cluster_kernel; see small_path)
  {
    const SmallPath sp = small_path(hkv, batch, max_seq_len, split_tokens);
    if (sp.C > 0 && (max_ctas <= 0 || static_cast<int64_t>(batch) * (hkv / sp.hpc * sp.C) <= max_ctas)) {
      const int C = sp.C;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(batch) * static_cast<unsigned>(hkv / sp.hpc * C));
      cfg.blockDim = dim3(kSmallThreads);
      cfg.dynamicSmemBytes = sizeof(SmallSmem);  // allowed by small_path's capacity query
      cfg.stream = st;
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(C);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 2;
      cudaError_t e;
      const bool two = sp.hpc == 2;
      switch (hkv) {
        case 8: e = two ? cudaLaunchKernelEx(&cfg, decode_cluster_kernel<8, 2>, p)
                        : cudaLaunchKernelEx(&cfg, decode_cluster_kernel<8, 1>, p); break;
        case 4: e = two ? cudaLaunchKernelEx(&cfg, decode_cluster_kernel<4, 2>, p)
                        : cudaLaunchKernelEx(&cfg, decode_cluster_kernel<4, 1>, p); break;
        case 2: e = two ? cudaLaunchKernelEx(&cfg, decode_cluster_kernel<2, 2>, p)
                        : cudaLaunchKernelEx(&cfg, decode_cluster_kernel<2, 1>, p); break;
        default: e = cudaLaunchKernelEx(&cfg, decode_cluster_kernel<1, 1>, p); break;
      }
      if (e != cudaSuccess) return record_cuda_error(e, "decode_cluster_kernel");
      return PA_OK;
    }
  }
  {
    // a programmatic dependent of the previous work on the stream: it may launch during that
    // work's tail and waits (griddepcontrol.wait) before reading any input
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sizeof(DecodeSmem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    switch (hkv) {
      case 8: e = cudaLaunchKernelEx(&cfg, decode_splitkv_kernel<8>, p); break;
      case 4: e = cudaLaunchKernelEx(&cfg, decode_splitkv_kernel<4>, p); break;
      case 2: e = cudaLaunchKernelEx(&cfg, decode_splitkv_kernel<2>, p); break;
      default: e = cudaLaunchKernelEx(&cfg, decode_splitkv_kernel<1>, p); break;
    }
    if (e != cudaSuccess) return record_cuda_error(e, "decode_splitkv_kernel");
  }
  {
    cudaLaunchConfig_t cfg = {};
    // partials per sequence when the lengths are equal: ceil(ranges / batch), plus one for a
    // cut at each end, times the page slots per range; more than 4 warps take in one round of
    // 4 loads -> 16 warps per head
    const int partials = ((plan.max_ranges + batch - 1) / batch + 1) * p.stage_pages;
    const bool many = partials > kMergeManyPartials;
    const bool small = partials > 4 * kMergeWarpsLarge;
    cfg.gridDim = dim3(batch, dims.num_q_heads, many ? kMergeDimParts : 1);
    cfg.blockDim = dim3((small ? kMergeWarpsSmall : kMergeWarpsLarge) * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = many ? cudaLaunchKernelEx(&cfg, decode_merge_dims_kernel, p)
                  : small ? cudaLaunchKernelEx(&cfg, decode_merge_kernel<kMergeWarpsSmall>, p)
                          : cudaLaunchKernelEx(&cfg, decode_merge_kernel<kMergeWarpsLarge>, p);
    if (e != cudaSuccess) return record_cuda_error(e, "decode_merge_kernel");
  }
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status attn_decode_paged(pa_dims dims, const void* q, const void* k_pool,
                                       const void* v_pool, int64_t num_pages,
                                       const int32_t* block_table, int32_t bt_stride,
                                       const int32_t* seq_lens, int32_t batch,
                                       int32_t max_seq_len, float softmax_scale,
                                       int32_t split_tokens, void* out, float* lse,
                                       void* workspace, size_t workspace_bytes, int32_t* status,
                                       pa_stream_t stream) {
  return pa::decode_call(dims, q, k_pool, v_pool, num_pages, block_table, bt_stride, seq_lens,
                         batch, max_seq_len, softmax_scale, split_tokens, out, lse, workspace,
                         workspace_bytes, status, stream, 0);
}

extern "C" pa_status attn_decode_paged_ex(pa_dims dims, const void* q, const void* k_pool,
                                          const void* v_pool, int64_t num_pages,
                                          const int32_t* block_table, int32_t bt_stride,
                                          const int32_t* seq_lens, int32_t batch,
                                          int32_t max_seq_len, float softmax_scale,
                                          int32_t split_tokens, void* out, float* lse,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t* status, pa_stream_t stream,
                                          const pa_launch_opts* opts) {
  const int32_t cap = opts != nullptr ? opts->max_ctas : 0;
  if (cap < 0) return PA_ERR_INVALID_ARG;
  return pa::decode_call(dims, q, k_pool, v_pool, num_pages, block_table, bt_stride, seq_lens,
                         batch, max_seq_len, softmax_scale, split_tokens, out, lse, workspace,
                         workspace_bytes, status, stream, cap);
}

// ---------------------------------------------------------------------------------------------
// attn_decode_paged_noalloc: the same decode, with its scratch in a fixed device array.
//
// For callers that cannot allocate device memory themselves: an engine that has handed all
// free HBM to its own KV-cache pool up front (a cudaMalloc would fail), a host process that
// embeds this library as a plugin without exposing an allocator, or a latency-critical loop
// where cudaMalloc/cudaFree may synchronize the device. Such a caller still passes q, the
// pools, the tables and the outputs; the split-KV partials go to g_decode_scratch, a
// file-scope array that every GPU which loads this library holds until the process exits.
// ---------------------------------------------------------------------------------------------
namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(9) << 19;  // 4.5 MiB
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[64] = {nullptr};

// Device address of g_decode_scratch on the current device. In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device (with that device
// current) and cached.
pa_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) return record_cuda_error(e, "cudaGetSymbolAddress(g_decode_scratch)");
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status attn_decode_paged_noalloc(pa_dims dims, const void* q, const void* k_pool,
                                               const void* v_pool, int64_t num_pages,
                                               const int32_t* block_table, int32_t bt_stride,
                                               const int32_t* seq_lens, int32_t batch,
                                               int32_t max_seq_len, float softmax_scale,
                                               void* out, float* lse, int32_t* status,
                                               pa_stream_t stream) {
  using namespace pa;
  if (batch < 0) return PA_ERR_INVALID_ARG;
  if (batch > 0) {
    const int grid = decode_grid_size();
    if (grid <= 0) return PA_ERR_CUDA;
    const size_t need = pa_decode_workspace_size(dims, batch, max_seq_len, 0);
    if (need > kStaticScratchBytes) {
      snprintf_error("attn_decode_paged_noalloc: batch %d needs %zu bytes of scratch on this GPU, "
                     "more than the built-in %zu bytes; use attn_decode_paged with a workspace",
                     batch, need, kStaticScratchBytes);
      return PA_ERR_WORKSPACE_TOO_SMALL;
    }
  }
  void* scratch = nullptr;
  const pa_status st = static_scratch(&scratch);
  if (st != PA_OK) return st;
  return attn_decode_paged(dims, q, k_pool, v_pool, num_pages, block_table, bt_stride, seq_lens,
                           batch, max_seq_len, softmax_scale, 0, out, lse, scratch,
                           kStaticScratchBytes, status, stream);
}
