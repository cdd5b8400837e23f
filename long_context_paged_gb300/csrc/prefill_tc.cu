// attn_prefill_chunk on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Source: chunked prefill of long audio prompts, 4096 tokens per scheduling step, each chunk
// attending causally to the KV cache of the earlier chunks plus its own tokens ("Optimizing
// ASR Models to Transcribe 90-Minute Multi-Speaker Audio", "Chunked Prefill for Long Audio";
// "MOSS-Transcribe-Diarize" cookbook, "Inference Pipeline"). QK^T and PV are dense
// contractions here (thousands of queries per KV read), so they run on tcgen05.mma.
//
// Work decomposition. A job is 128 queries of one chunk x both query heads of one KV head
// (GQA 16/8, or 2N/N heads when the KV heads are partitioned across devices): two 128-row M
// tiles that share every K/V tile read. A job's causal key range is
// J tiles of 128 keys; one (job, key tile) pair is a unit. Jobs are ordered sequence, then KV
// head, then query tile. A persistent grid of one CTA per SM first runs whole jobs round-robin
// (CTA c takes jobs c, c + G, ...; all CTAs of a round start at key tile 0 together, so the CTAs
// of a KV head read the same K/V tiles from L2), then splits the units of the remaining jobs
// into equal contiguous ranges, so the work stays balanced to about one tile whatever the
// chunk lengths and offsets. A job cut by range boundaries leaves normalised partial results
// (o, lse) in the workspace; prefill_merge_kernel combines them by log-sum-exp.
//
// Per 128-key tile j of a job:
//   S_t = Q_t K_j^T         tcgen05.mma, A = Q_t (smem), B = K_j (smem), D = S_t (TMEM fp32)
//   P_t = softmax part      4 warps per M tile, one thread per row: tcgen05.ld S_t, mask the
//                           diagonal, exp2 on the MUFU unit, row sum; P_t written back
//                           over S_t as bf16
//   O_t += P_t V_j          tcgen05.mma, A = P_t (TMEM), B = V_j (smem, MN-major), D = O_t
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
// Warp roles: 0-3 softmax of M tile 0, 4-7 softmax of M tile 1, 8 TMA producer of V, 9 MMA
// issuer, 10 TMA producer of Q and K, 11 scheduler: it alone walks the work split and publishes
// each piece (job, key-tile range) in a small shared-memory ring, so the other roles hold only
// the few fields they use instead of the walker's state (registers are what bounds the
// softmax and the issuer).
// K/V tiles arrive by tiled TMA straight from the page pools: one 16-token page x 64 dims per
// copy (a 3-D tensor map over [tokens][kv heads][dims] with 128-byte swizzle), so the block
// table is applied per page without a gather pass. Pages past the sequence are fetched at an
// out-of-range coordinate and arrive as zeros; V rows of the last partial page are zeroed in
// shared memory before use, so unwritten slots can never reach P*V.
// The running row max moves only when a tile exceeds it by more than 8 (log2 units); O is then
// rescaled in TMEM by its owning warps; the previous P*V has completed by then, since the
// commit the warps waited on for this tile's S covers every earlier MMA of the issuer.
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "pa_common.cuh"
#include "tc_common.cuh"

namespace pa {

bool make_map_3d(CUtensorMap* map, const void* base, uint64_t outer, uint64_t heads,
                 uint32_t box_rows);

namespace {

constexpr int kTileM = 128;   // queries per job (per head)
constexpr int kTileN = 128;   // keys per K/V tile
constexpr int kThreads = 384; // 8 softmax warps + producer + MMA + 2 spare (3 warpgroups)
constexpr int kProducerWarp = 8;   // V tiles
constexpr int kMmaWarp = 9;
constexpr int kKProducerWarp = 10; // Q and K tiles
constexpr int kSchedWarp = 11;      // walks the work split and publishes the pieces
constexpr int kPieceRing = 4;       // published pieces in flight
constexpr int kPieceReaders = 11;   // warps that read every piece: 8 softmax, 2 producers, MMA
constexpr uint32_t kBlockBytes = 128 * 128;  // 128 rows x 64 bf16 (one swizzled 64-dim block)
constexpr uint32_t kTileBytes = 2 * kBlockBytes;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kMaxBatch = 128;   // chunks per call (the unit prefix lives in shared memory)
constexpr int kVStages = 3;   // V is needed a whole P*V later than K: one more stage in flight
// Fixed cost of a job beyond its key tiles, in tiles: its epilogue and the restart of the
// softmax -> P -> P*V chain on its first tile (measured ~5.5 us a job, about 3 tiles). In the
// work split each job occupies its key tiles followed by this many cost units, so that a CTA whose
// share holds many short jobs is not overloaded; the cost units hold no key tile.
constexpr int kJobCost = 3;
// Register split: the two softmax warpgroups grow to 208 registers per thread, the
// producer/MMA/scheduler warpgroup shrinks to 88 (measured: 200/104 about 1 % slower, 216/72
// and 192/120 7-9 % slower: the issuer's loop and the softmax both stall when they spill);
// 256 * 208 + 128 * 88 = 64,512 = 384 threads x 168, the budget the CTA is launched with
// (checked on the host before every launch).
constexpr int kSoftmaxRegs = 208;
constexpr int kControlRegs = 88;
constexpr int kLaunchRegs = (256 * kSoftmaxRegs + 128 * kControlRegs) / kThreads;
// A partial result: o [2 heads][32 float4 columns][128 rows] (16-byte units; consecutive rows
// are adjacent, so a warp's 32 rows store and load 512 contiguous bytes), then lse [2][128] fp32.
constexpr size_t kRecordO = 2 * 128 * 128 * sizeof(float);
constexpr size_t kRecordBytes = kRecordO + 2 * 128 * sizeof(float);
constexpr int kMergeRows = 128;  // threads of a merge CTA: one per row of a query tile

// One piece of the walk as the roles use it: key tiles [jb, je) of job (b, g, qt), with the
// chunk's first packed row q0, its length n, the sequence's keys L and the chunk's offset off;
// J = the job's key tiles; valid = 0 ends the walk.
struct PieceDesc {
  int32_t b, g, qt, q0, n, L, off, J, jb, je, valid;
};

struct PrefillTcSmem {  // placed at a 1024-byte aligned address (swizzle atoms)
  uint8_t q[2][2][kBlockBytes];   // [M tile][64-dim block]
  uint8_t k[2][2][kBlockBytes];   // [stage][64-dim block]
  uint8_t v[kVStages][2][kBlockBytes];
  uint64_t q_full, q_empty;
  uint64_t k_full[2], k_empty[2];
  // pv_full[st]: P_0 of the tile in V stage st is in TMEM and that V tile has landed (four
  // softmax-0 warps arrive, the V producer arrives and its copies complete bytes on it);
  // p1_full: P_1 of the current tile is in TMEM
  uint64_t pv_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], p1_full, o_ready[2], o_free[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  PieceDesc piece[kPieceRing];
  uint64_t piece_full[kPieceRing], piece_empty[kPieceRing];
  long long warp_sums[kThreads / 32];
  long long total_units;
  long long unit_prefix[kMaxBatch + 1];  // first unit of each sequence
  int32_t job_prefix[kMaxBatch + 1];     // first job of each sequence
  int32_t total_jobs;
  int32_t plan_rounds;                   // whole-job rounds of the balanced split
  long long plan_u0, plan_u1;            // this CTA's range of the remaining units
};

// The dynamic shared memory of a CTA starts 1024-byte aligned on this GPU (after the 1 KB the
// system reserves per block), which the swizzled operand tiles need; the kernel checks it.
static_assert(sizeof(PrefillTcSmem) <= 232448, "prefill shared memory over the 227 KB limit");

struct PrefillTcParams {
  int32_t hkv, hq;        // KV heads and query heads of the call (hq = 2 hkv)
  const int32_t* cu_q_lens;
  const int32_t* seq_lens;
  const int32_t* block_table;
  int32_t bt_stride;
  int32_t batch;
  int64_t num_pages;
  float scale_log2;
  uint16_t* out;
  float* lse;
  int32_t* status;
  long long* ws_header;   // [0] grid size, [1] total units, [2] first unit after the whole
                          // jobs, [3] jobs done whole in the round-robin phase
  long long* ws_prefix;   // [batch + 1] first unit of each sequence
  int32_t* ws_job_prefix; // [batch + 1] first job of each sequence
  long long* ws_tail;     // [grid + 1] first unit of each CTA's range after the whole jobs
  uint8_t* ws_records;    // [2 * grid][kRecordBytes]
};

// ---------------------------------------------------------------------------------------------
// Job geometry of one sequence (same arithmetic in every role and in the merge kernel).
// ---------------------------------------------------------------------------------------------
struct SeqGeom {
  int q0, n, L, off, nqt;
  long long a, Jlast, T;  // full-tile J is a + qt; the last tile's is Jlast; T = units per head
};

__device__ __forceinline__ SeqGeom seq_geom(const PrefillTcParams& p, int b, bool report) {
  SeqGeom s;
  s.q0 = p.cu_q_lens[b];
  s.n = p.cu_q_lens[b + 1] - s.q0;
  s.L = p.seq_lens[b];
  s.nqt = 0;
  s.off = s.L - s.n;
  s.a = s.Jlast = s.T = 0;
  if (s.n <= 0) return s;
  if (s.n > s.L || s.L > p.bt_stride * kPage) {
    if (report) flag_error(p.status, PA_DEV_ERR_LENGTH);
    return s;
  }
  s.nqt = (s.n + kTileM - 1) / kTileM;
  s.a = (s.off + kTileN - 1) / kTileN + 1;
  s.Jlast = (s.off + s.n - 1) / kTileN + 1;
  const long long full = s.nqt - 1;
  s.T = full * s.a + full * (full - 1) / 2 + s.Jlast + static_cast<long long>(s.nqt) * kJobCost;
  return s;
}

__device__ __forceinline__ long long tiles_of(const SeqGeom& s, int qt) {
  return qt < s.nqt - 1 ? s.a + qt : s.Jlast;
}
// Units of the jobs before q tile qt of one head: their key tiles and their cost units.
__device__ __forceinline__ long long units_before(const SeqGeom& s, int qt) {
  return static_cast<long long>(qt) * (s.a + kJobCost) + static_cast<long long>(qt) * (qt - 1) / 2;
}

// One job piece this CTA owns: key tiles [jb, je) of job (b, g, qt).
struct Piece {
  int b, g, qt;
  SeqGeom s;
  long long u0;  // first unit of the job
  int J, jb, je;
  bool valid;
};

// The pieces one CTA owns, in order: first whole jobs c, c + G, c + 2G, ... (G = grid size) for
// `rounds` rounds, all CTAs starting at key tile 0 together so that the CTAs of one KV head stream
// the same K/V tiles through L2 at about the same time; then a range [U0, U1) of the units of the
// remaining jobs (sized by plan_split so that every CTA ends with the same number of units),
// whose first and last pieces may be parts of jobs shared with neighbouring CTAs.
struct JobWalker {
  const PrefillTcParams* p;
  const long long* prefix;
  const int32_t* jprefix;
  long long U0, U1;
  int rounds, round, G;
  Piece cur;

  __device__ void set(int b, int g, int qt, long long u0, const SeqGeom& s) {
    cur.b = b;
    cur.g = g;
    cur.qt = qt;
    cur.s = s;
    cur.u0 = u0;
    cur.J = static_cast<int>(tiles_of(s, qt));
    cur.jb = static_cast<int>(max(U0, u0) - u0);
    cur.je = static_cast<int>(min(U1, u0 + cur.J) - u0);
    cur.valid = u0 < U1 && cur.jb < cur.je;
  }

  __device__ void set_whole_job(int jo) {
    int lo = 0, hi = p->batch;  // last b with jprefix[b] <= jo < jprefix[b+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (jprefix[mid] <= jo) lo = mid; else hi = mid;
    }
    const SeqGeom s = seq_geom(*p, lo, false);
    const int rem = jo - jprefix[lo];
    const int g = rem / s.nqt, qt = rem - g * s.nqt;
    cur.b = lo;
    cur.g = g;
    cur.qt = qt;
    cur.s = s;
    cur.u0 = prefix[lo] + g * s.T + units_before(s, qt);
    cur.J = static_cast<int>(tiles_of(s, qt));
    cur.jb = 0;
    cur.je = cur.J;
    cur.valid = true;
  }

  __device__ void start_tail() {
    if (U0 >= U1) {
      cur.valid = false;
      return;
    }
    int lo = 0, hi = p->batch;  // last b with prefix[b] <= U0 < prefix[b+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= U0) lo = mid; else hi = mid;
    }
    const SeqGeom s = seq_geom(*p, lo, false);
    const long long rem = U0 - prefix[lo];
    const int g = static_cast<int>(rem / s.T);
    const long long rem2 = rem - g * s.T;
    int qt = 0;
    while (qt + 1 < s.nqt && units_before(s, qt + 1) <= rem2) ++qt;
    set(lo, g, qt, prefix[lo] + g * s.T + units_before(s, qt), s);
    // a range that starts in the cost units after a job's last key tile holds none of its tiles
    if (!cur.valid && cur.u0 + cur.J + kJobCost < U1) advance_tail();
  }

  __device__ void start(const PrefillTcParams& pp, const long long* pre, const int32_t* jpre,
                        int n_rounds, int grid, long long u_begin, long long u_end) {
    p = &pp;
    prefix = pre;
    jprefix = jpre;
    U0 = u_begin;
    U1 = u_end;
    rounds = n_rounds;
    G = grid;
    round = 0;
    if (rounds > 0) set_whole_job(static_cast<int>(blockIdx.x));
    else start_tail();
  }

  __device__ void next() {
    if (round < rounds) {
      if (++round < rounds) set_whole_job(static_cast<int>(blockIdx.x) + round * G);
      else start_tail();
      return;
    }
    advance_tail();
  }

  // the job after cur in unit order (the tail phase walks its range job by job)
  __device__ void advance_tail() {
    long long u0 = cur.u0 + cur.J + kJobCost;
    int b = cur.b, g = cur.g, qt = cur.qt + 1;
    SeqGeom s = cur.s;
    if (qt >= s.nqt) {
      qt = 0;
      if (++g >= p->hkv) {
        g = 0;
        do {
          ++b;
          if (b >= p->batch) {
            cur.valid = false;
            return;
          }
          s = seq_geom(*p, b, false);
        } while (s.nqt == 0);
        u0 = prefix[b];
      }
    }
    set(b, g, qt, u0, s);
  }
};

__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_wait_bounded(bar, parity)) return true;
  flag_error(status, PA_DEV_ERR_TIMEOUT);
  return false;
}

// The next published piece, read by a whole warp: wait for its slot, copy it, release the slot.
// A wait that gives up ends the walk (valid = 0) after flagging PA_DEV_ERR_TIMEOUT.
__device__ __forceinline__ PieceDesc take_piece_warp(PrefillTcSmem& s, uint32_t& k, int lane,
                                                     int32_t* status) {
  const uint32_t slot = k % kPieceRing, ph = (k / kPieceRing) & 1;
  PieceDesc d;
  if (!__all_sync(0xffffffffu, wait_or_flag(&s.piece_full[slot], ph, status))) {
    d.valid = 0;
    return d;
  }
  d = s.piece[slot];
  __syncwarp();
  if (lane == 0) mbar_arrive(&s.piece_empty[slot]);
  ++k;
  return d;
}

__device__ __forceinline__ long long warp_incl_scan64(long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// unit_prefix[b] = first unit of sequence b (8 heads x T_b units each).
__device__ void build_unit_prefix(const PrefillTcParams& p, PrefillTcSmem& s) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (p.batch + kThreads - 1) / kThreads;
  const int b0 = min(p.batch, tid * per), b1 = min(p.batch, b0 + per);
  long long local = 0;
  int local_jobs = 0;
  for (int b = b0; b < b1; ++b) {
    const SeqGeom g = seq_geom(p, b, blockIdx.x == 0);
    local += p.hkv * g.T;
    local_jobs += p.hkv * g.nqt;
  }
  const long long incl = warp_incl_scan64((static_cast<long long>(local_jobs) << 40) | local, lane);
  // (jobs in the top 24 bits, units in the low 40: both sums fit: units < 2^40, jobs < 2^23)
  if (lane == 31) s.warp_sums[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    long long run = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      const long long v = s.warp_sums[w];
      s.warp_sums[w] = run;
      run += v;
    }
    s.total_units = run;
  }
  __syncthreads();
  const long long packed = s.warp_sums[warp] + incl - ((static_cast<long long>(local_jobs) << 40) | local);
  long long run = packed & ((1ll << 40) - 1);
  int jrun = static_cast<int>(packed >> 40);
  for (int b = b0; b < b1; ++b) {
    const SeqGeom g = seq_geom(p, b, false);
    s.unit_prefix[b] = run;
    s.job_prefix[b] = jrun;
    run += p.hkv * g.T;
    jrun += p.hkv * g.nqt;
  }
  __syncthreads();
  if (tid == 0) {
    s.total_jobs = static_cast<int>(s.total_units >> 40);
    s.total_units &= (1ll << 40) - 1;
    s.unit_prefix[p.batch] = s.total_units;
    s.job_prefix[p.batch] = s.total_jobs;
  }
  __syncthreads();
}

// Units of job jo (its key tiles plus kJobCost): jobs are numbered sequence by sequence, then KV
// head, then q tile.
__device__ long long job_units(const PrefillTcParams& p, const PrefillTcSmem& s, int jo) {
  int lo = 0, hi = p.batch;  // last b with job_prefix[b] <= jo (a sequence that has jobs)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.job_prefix[mid] <= jo) lo = mid; else hi = mid;
  }
  const SeqGeom g = seq_geom(p, lo, false);
  return tiles_of(g, (jo - s.job_prefix[lo]) % g.nqt) + kJobCost;
}

// Balanced split of all units over the G CTAs (G <= kThreads, one CTA per thread here). With
// target = ceil(total / G): whole jobs go round-robin (CTA c takes jobs c, c + G, ...) for as many
// rounds as keep every CTA's whole-job units within target; the units of the remaining jobs are
// then cut into consecutive ranges, CTA c's of size target - whole(c), so CTAs whose whole jobs were
// short take more of the rest and all end level even when job lengths differ widely (chunks of
// different lengths and offsets in one call). Every CTA computes the same plan; CTA 0 also
// publishes the range starts for the merge kernel.
__device__ void plan_split(const PrefillTcParams& p, PrefillTcSmem& s, int G, int& rounds,
                           long long& T0, long long& U0, long long& U1) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long total = s.total_units;
  const long long target = (total + G - 1) / G;
  const int rmax = s.total_jobs / G;
  if (tid == 0) s.plan_rounds = rmax;
  __syncthreads();
  if (tid < G) {
    long long acc = 0;
    int r = 0;
    for (; r < rmax; ++r) {
      acc += job_units(p, s, tid + r * G);
      if (acc > target) break;
    }
    if (r < rmax) atomicMin(&s.plan_rounds, r);
  }
  __syncthreads();
  rounds = s.plan_rounds;
  long long tail = 0;
  if (tid < G) {
    long long whole = 0;
    for (int r = 0; r < rounds; ++r) whole += job_units(p, s, tid + r * G);
    tail = target - whole;  // >= 0: every CTA's whole jobs fit in target for this many rounds
  }
  // exclusive scan of the range sizes over the CTAs
  const long long incl = warp_incl_scan64(tail, lane);
  if (lane == 31) s.warp_sums[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    long long run = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      const long long v = s.warp_sums[w];
      s.warp_sums[w] = run;
      run += v;
    }
  }
  __syncthreads();
  const long long excl = s.warp_sums[warp] + incl - tail;
  // first unit after the whole jobs: that of job rounds * G
  const int n_dp = rounds * G;
  T0 = total;
  if (n_dp < s.total_jobs) {
    int lo = 0, hi = p.batch;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s.job_prefix[mid] <= n_dp) lo = mid; else hi = mid;
    }
    const SeqGeom g0 = seq_geom(p, lo, false);
    const int rem = n_dp - s.job_prefix[lo];
    T0 = s.unit_prefix[lo] + (rem / g0.nqt) * g0.T + units_before(g0, rem % g0.nqt);
  }
  if (tid < G) {
    const long long u0 = min(total, T0 + excl), u1 = min(total, T0 + excl + tail);
    if (tid == static_cast<int>(blockIdx.x)) {
      s.plan_u0 = u0;
      s.plan_u1 = u1;
    }
    if (blockIdx.x == 0) p.ws_tail[tid] = u0;
  }
  if (blockIdx.x == 0 && tid == 0) p.ws_tail[G] = total;
  __syncthreads();
  U0 = s.plan_u0;
  U1 = s.plan_u1;
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                  const __grid_constant__ CUtensorMap k_map,
                  const __grid_constant__ CUtensorMap v_map, const PrefillTcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.launch_dependents;");  // the merge kernel waits for completion
  if ((smem_addr(smem_raw) & 1023u) != 0) {
    // not the layout this kernel was built for: do nothing, and make the merge do nothing
    // (it skips every job below ws_header[3])
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      p.ws_header[3] = 0x7fffffffffffffffll;
      flag_error(p.status, PA_DEV_ERR_INTERNAL);
    }
    return;
  }
  PrefillTcSmem& s = *reinterpret_cast<PrefillTcSmem*>(smem_raw);
  build_unit_prefix(p, s);
  const long long total = s.total_units;
  const int G = gridDim.x;
  int rounds;
  long long T0, U0, U1;
  plan_split(p, s, G, rounds, T0, U0, U1);
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) {
      p.ws_header[0] = G;
      p.ws_header[1] = total;
      p.ws_header[2] = T0;
      p.ws_header[3] = static_cast<long long>(rounds) * G;
    }
    for (int b = threadIdx.x; b <= p.batch; b += kThreads) {
      p.ws_prefix[b] = s.unit_prefix[b];
      p.ws_job_prefix[b] = s.job_prefix[b];
    }
  }
  if (rounds == 0 && U0 >= U1) return;  // uniform across the CTA: nothing allocated yet

  if (threadIdx.x == 0) {
    mbar_init(&s.q_full, 1);
    mbar_init(&s.q_empty, 2);       // released by each M tile's softmax (see below)
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 2);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.o_ready[i], 1);
      mbar_init(&s.o_free[i], 4);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&s.pv_full[i], 5);   // 4 softmax-0 warps + the V producer (+ its bytes)
      mbar_init(&s.v_empty[i], 2);
    }
    mbar_init(&s.p1_full, 4);         // one arrive per softmax-1 warp
    mbar_init(&s.mma_done, 1);
    for (int i = 0; i < kPieceRing; ++i) {
      mbar_init(&s.piece_full[i], 1);
      mbar_init(&s.piece_empty[i], kPieceReaders);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tc::tmem_alloc<512>(&s.tmem_base);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s.tmem_base;


  if (warp >= 8) {
    tc::regs_decrease<kControlRegs>();
  if (warp == kProducerWarp || warp == kKProducerWarp) {
    // ------------------------------------------------------------------ TMA producers
    // Warp 10 loads Q and the K tiles, warp 8 the V tiles, each as soon as its own ring has a
    // free stage (K is needed a whole P*V earlier than V).
    const bool is_k = warp == kKProducerWarp;
    const CUtensorMap* map = is_k ? &k_map : &v_map;
    uint8_t(*ring)[2][kBlockBytes] = is_k ? s.k : s.v;
    const uint32_t nst = is_k ? 2u : static_cast<uint32_t>(kVStages);
    uint64_t* full = is_k ? s.k_full : s.pv_full;
    uint64_t* empty = is_k ? s.k_empty : s.v_empty;
    const int oob_token = static_cast<int>(p.num_pages * kPage);  // zero-filled coordinate
    bool ok = true;
    uint32_t it = 0, jc = 0, pk = 0;
    for (PieceDesc pc = take_piece_warp(s, pk, lane, p.status); pc.valid && ok;
         pc = take_piece_warp(s, pk, lane, p.status)) {
      const int32_t* bt_row = p.block_table + static_cast<int64_t>(pc.b) * p.bt_stride;
      auto page_token = [&](int j) {
        int tok = oob_token;
        const int key0 = j * kTileN + kPage * lane;
        if (lane < kTileN / kPage && key0 < pc.L) {
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
      if (is_k) {
        if (lane == 0) {
          ok = wait_or_flag(&s.q_empty, (jc & 1) ^ 1u, p.status);
          if (ok) {
            mbar_arrive_expect_tx(&s.q_full, 4 * kBlockBytes);
            for (int t = 0; t < 2; ++t)
              for (int kb = 0; kb < 2; ++kb)
                tc::tma_load_3d(s.q[t][kb], &q_map, kb * 64, 2 * pc.g + t,
                                pc.q0 + pc.qt * kTileM, &s.q_full);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      int tok = page_token(pc.jb);
      int tok_next = (pc.jb + 1 < pc.je) ? page_token(pc.jb + 1) : oob_token;
      for (int j = pc.jb; j < pc.je && ok; ++j, ++it) {
        const int st = it % nst;
        const uint32_t ph = (it / nst) & 1;
        const int tok_ahead = (j + 2 < pc.je) ? page_token(j + 2) : oob_token;
        if (lane == 0) ok = wait_or_flag(&empty[st], ph ^ 1u, p.status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&full[st], kTileBytes);
        __syncwarp();
        {
          // 16 lanes issue the 16 copies of the tile at once (page pg = lane / 2, 64-dim
          // block lane % 2): one warp-wide instruction instead of 16 single-lane ones
          const int pg = (lane >> 1) & 7, kb = lane & 1;
          const int t = __shfl_sync(0xffffffffu, tok, pg);
          if (lane < 2 * (kTileN / kPage))
            tc::tma_load_3d(ring[st][kb] + pg * 2048, map, kb * 64, pc.g, t, &full[st]);
        }
        tok = tok_next;
        tok_next = tok_ahead;
      }
      ++jc;
    }
    // do not leave while copies into this CTA's shared memory may still be landing
    if (lane == 0 && it > 0) {
      for (uint32_t k = (it >= nst ? it - nst : 0); k < it; ++k)
        wait_or_flag(&full[k % nst], (k / nst) & 1, p.status);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    // The tensor pipe queues only about one instruction ahead of the issuing thread, so the
    // work between two MMA groups shows up directly as idle pipe time. Lane 0 runs the whole
    // loop alone (no per-tile warp collectives); ring stages and barrier parities are
    // counters; descriptors are built once and selected, and a K step is a constant added to
    // the start field (16-byte units; shared memory stays below 256 KB, so it cannot carry out
    // of its 14 bits).
    constexpr uint32_t id_s = tc::idesc_bf16(128, kTileN, 0, 0);    // S = Q K^T
    constexpr uint32_t id_o = tc::idesc_bf16(128, 128, 0, 1);       // O = P V, V MN-major
    static_assert(kVStages == 3, "the V descriptor selection below assumes three stages");
    if (lane == 0) {
      const uint64_t dq0 = tc::smem_desc_sw128(smem_addr(s.q[0][0]), 16, 1024);
      const uint64_t dq1 = tc::smem_desc_sw128(smem_addr(s.q[1][0]), 16, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(s.k[0][0]), 16, 1024);
      const uint64_t dk1 = tc::smem_desc_sw128(smem_addr(s.k[1][0]), 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(s.v[0][0]), kBlockBytes, 1024);
      const uint64_t dv1 = tc::smem_desc_sw128(smem_addr(s.v[1][0]), kBlockBytes, 1024);
      const uint64_t dv2 = tc::smem_desc_sw128(smem_addr(s.v[2][0]), kBlockBytes, 1024);
      auto issue_s = [&](uint32_t d, uint64_t a, uint64_t b) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = ((kk >> 2) * kBlockBytes + (kk & 3) * 32) >> 4;
          if (kk == 0) tc::mma_ss_c<false>(d, a + off, b + off, id_s);
          else tc::mma_ss_c<true>(d, a + off, b + off, id_s);
        }
      };
      auto issue_pv = [&](uint32_t d, uint32_t a, uint64_t b, uint32_t acc) {
        tc::mma_ts(d, a, b, id_o, acc);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk) tc::mma_ts_c<true>(d, a + kk * 8, b + kk * (2048 >> 4), id_o);
      };
      // This thread waits only for P of each M tile (P_0's barrier also takes the V copies'
      // bytes, so it certifies V) and for the next K tile, and commits only S completion per
      // tile and O completion per piece: the K / V / Q stages are released by the softmax
      // warps, which observe S_t(j) done (and through that commit also P_t V(j-1) done).
      uint32_t kst = 0, kph = 0;     // K ring: stage and parity of the next tile to consume
      uint32_t vst = 0, vph = 0;     // V ring: stage and parity of the current tile
      uint32_t tph = 0;              // parity of the current tile's S / P phases
      bool ok = true;
      uint32_t jc = 0;
      uint32_t pk = 0;
      for (;; ++jc) {
        // the next piece: only its tile count and the sequence end are needed here
        const uint32_t pslot = pk % kPieceRing;
        if (!wait_or_flag(&s.piece_full[pslot], (pk / kPieceRing) & 1, p.status)) break;
        const volatile PieceDesc& pv = s.piece[pslot];
        const int pvalid = pv.valid, pjb = pv.jb, pje = pv.je, pL = pv.L;
        mbar_arrive(&s.piece_empty[pslot]);
        ++pk;
        if (!pvalid || !ok) break;
        const int nt = pje - pjb;
        // The piece's last tile runs past the sequence end when L < je * 128. Its page that
        // holds key L - 1 was loaded whole, so the V rows of the pool slots after the last key
        // ([zl, next multiple of 16)) are zeroed, that P = 0 there cannot meet an unwritten
        // (possibly NaN) slot; the pages after it were never loaded (zero fill).
        const int zl = pL - (pje - 1) * kTileN;
        const int zero_i = (zl > 0 && zl < kTileN && (zl & 15) != 0) ? nt - 1 : -1;
        const uint32_t qph = jc & 1, oph = (jc - 1) & 1;
        ok = wait_or_flag(&s.q_full, qph, p.status) && wait_or_flag(&s.k_full[kst], kph, p.status);
        if (!ok) break;
        tc::fence_after_sync();
        uint64_t dk = kst ? dk1 : dk0;
        issue_s(tmem, dq0, dk);
        tc::mma_commit(&s.s_full[0]);
        issue_s(tmem + 128, dq1, dk);
        tc::mma_commit(&s.s_full[1]);
        kph ^= kst;
        kst ^= 1u;
        for (int i = 0; i < nt; ++i) {
          const bool more = i + 1 < nt;
          const uint64_t dv = vst == 0 ? dv0 : (vst == 1 ? dv1 : dv2);
          const uint32_t acc = i > 0 ? 1u : 0u;
          if (!wait_or_flag(&s.pv_full[vst], vph, p.status) ||
              (i == 0 && jc > 0 && !wait_or_flag(&s.o_free[0], oph, p.status))) {
            ok = false;
            break;
          }
          if (i == zero_i) {
            for (int e = zl * 16; e < ((zl + 15) & ~15) * 16; ++e) {
              const int r = e >> 4, c = e & 15;   // row, 16-byte chunk (8 per 64-dim block)
              *reinterpret_cast<uint4*>(s.v[vst][c >> 3] + r * 128 + (c & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            tc::fence_proxy_async_smem();
          }
          tc::fence_after_sync();
          issue_pv(tmem + 256, tmem, dv, acc);
          if (more) {
            if (!wait_or_flag(&s.k_full[kst], kph, p.status)) { ok = false; break; }
            tc::fence_after_sync();
            dk = kst ? dk1 : dk0;
            issue_s(tmem, dq0, dk);
            tc::mma_commit(&s.s_full[0]);
          } else {
            tc::mma_commit(&s.o_ready[0]);
          }
          if (!wait_or_flag(&s.p1_full, tph, p.status) ||
              (i == 0 && jc > 0 && !wait_or_flag(&s.o_free[1], oph, p.status))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          issue_pv(tmem + 384, tmem + 128, dv, acc);
          if (more) {
            issue_s(tmem + 128, dq1, dk);
            tc::mma_commit(&s.s_full[1]);
            kph ^= kst;
            kst ^= 1u;
          } else {
            tc::mma_commit(&s.o_ready[1]);
          }
          vst = vst == 2 ? 0u : vst + 1;
          vph ^= vst == 0 ? 1u : 0u;
          tph ^= 1u;
        }
      }
    }
    __syncwarp();
    // every MMA lane 0 issued must have finished before TMEM is released
    if (lane == 0) {
      tc::mma_commit(&s.mma_done);
      wait_or_flag(&s.mma_done, 0, p.status);
    }
    __syncwarp();
  } else if (warp == kSchedWarp) {
    // ------------------------------------------------------------------ scheduler
    if (lane == 0) {
      JobWalker jw;
      jw.start(p, s.unit_prefix, s.job_prefix, rounds, G, U0, U1);
      for (uint32_t k = 0;; ++k) {
        const uint32_t slot = k % kPieceRing, ph = (k / kPieceRing) & 1;
        if (!wait_or_flag(&s.piece_empty[slot], ph ^ 1u, p.status)) break;
        const Piece& c = jw.cur;
        PieceDesc d;
        d.b = c.b;
        d.g = c.g;
        d.qt = c.qt;
        d.q0 = c.s.q0;
        d.n = c.s.n;
        d.L = c.s.L;
        d.off = c.s.off;
        d.J = c.J;
        d.jb = c.jb;
        d.je = c.je;
        d.valid = c.valid ? 1 : 0;
        s.piece[slot] = d;
        mbar_arrive(&s.piece_full[slot]);  // release: the readers' waits make d visible
        if (!c.valid) break;
        jw.next();
      }
    }
    __syncwarp();
  }
  } else {
    tc::regs_increase<kSoftmaxRegs>();
    // ------------------------------------------------------------------ softmax warps
    const int t = warp >> 2;                       // M tile = query head 2g + t
    const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;             // row of the tile
    const uint32_t lane_bits = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_bits + t * 128;
    const uint32_t t_o = tmem + lane_bits + 256 + t * 128;
    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
    bool ok = true;
    uint32_t it = 0, jcs = 0;
    const bool leader = quarter == 0 && lane == 0;  // releases stages for this M tile
    uint32_t pk = 0;
    for (;; ++jcs) {
      // the next piece; its slot is held until the epilogue, which reads the rest of it
      const uint32_t pslot = pk % kPieceRing;
      if (!__all_sync(0xffffffffu, wait_or_flag(&s.piece_full[pslot], (pk / kPieceRing) & 1, p.status)))
        break;
      const volatile PieceDesc& pv = s.piece[pslot];
      if (!pv.valid || !ok) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.piece_empty[pslot]);
        break;
      }
      const int pjb = pv.jb;
      const int nt = pv.je - pjb;
      const int qrow = pv.qt * kTileM + r;
      const int qpos = pv.off + qrow;              // absolute position of this query
      float m_used = -CUDART_INF_F, l = 0.f;
      for (int i = 0; i < nt; ++i) {
        const uint32_t cur = it + i;
        ok = __all_sync(0xffffffffu, wait_or_flag(&s.s_full[t], cur & 1, p.status));
        if (!ok) break;
        // S_t(cur) is done, and its commit also covers P_t V(cur - 1): this M tile is finished
        // with K stage cur and V stage cur - 1 (the last V stage of a piece is released after
        // the epilogue's wait), and with Q after the piece's last tile
        if (leader) {
          mbar_arrive(&s.k_empty[cur & 1]);
          if (i > 0) mbar_arrive(&s.v_empty[(cur - 1) % kVStages]);
          if (i + 1 == nt) mbar_arrive(&s.q_empty);
        }
        tc::fence_after_sync();
        uint32_t sb[128];  // raw scores (fp32 bits) of this row
        float cm[4];       // the maximum of each 32-column piece, from the TMEM load itself
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tc::tmem_ld32_max(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sb + c * 32), cm[c]);
        tc::tmem_wait_ld();
        const int k0 = (pjb + i) * kTileN;
        float mx = fmax3(cm[0], cm[1], fmaxf(cm[2], cm[3]));
        if (k0 + kTileN - 1 > qpos) {
          // the tile crosses this row's position: mask the keys after the query, then take the
          // row max over what is left (8 independent partial maxima, two new elements per
          // three-input max)
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (k0 + c > qpos) sb[c] = 0xff800000u;  // -inf: key after this query
          float pm[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            pm[k] = fmax3(__uint_as_float(sb[k]), __uint_as_float(sb[k + 8]), __uint_as_float(sb[k + 16]));
#pragma unroll
          for (int c = 24; c < 120; c += 16) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              pm[k] = fmax3(pm[k], __uint_as_float(sb[c + k]), __uint_as_float(sb[c + 8 + k]));
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) pm[k] = fmaxf(pm[k], __uint_as_float(sb[120 + k]));
          mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
        }
        const float mx2 = mx * p.scale_log2;
        const bool grow = mx2 > m_used + kRescaleThreshold;
        if (__any_sync(0xffffffffu, grow)) {
          const float m_new = grow ? mx2 : m_used;
          const float alpha = (m_used == -CUDART_INF_F) ? 0.f : fast_exp2(m_used - m_new);
          if (i > 0) {
            // O_t holds the sum through the previous tile: P_t V(cur - 1) completed before
            // S_t(cur), whose completion this thread has already observed
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t o32[32];
              tc::tmem_ld32(t_o + c * 32, o32);
              tc::tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) o32[k] = __float_as_uint(__uint_as_float(o32[k]) * alpha);
              tc::tmem_st32(t_o + c * 32, o32);
            }
            tc::tmem_wait_st();
          }
          l *= alpha;
          m_used = m_new;
        }
        // probabilities (bf16) over S's first 64 columns. A row that has not met a visible key
        // yet (its piece starts past the row's position) keeps m_used = -inf; a finite offset
        // then gives exp2(-inf) = 0 for its masked scores instead of NaN.
        const float m_eff = (m_used == -CUDART_INF_F) ? 0.f : m_used;
        const float2 nm2 = make_float2(-m_eff, -m_eff);
        float2 ls[4];  // 4 independent paired partial sums
#pragma unroll
        for (int k = 0; k < 4; ++k) ls[k] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float2 x = fma2(make_float2(__uint_as_float(sb[c * 64 + 2 * k]),
                                              __uint_as_float(sb[c * 64 + 2 * k + 1])), sc2, nm2);
            // exp2 on the MUFU unit (moving a share of them to an FMA-pipe polynomial, or
            // fusing the row max into this pass, measured slower on GB300)
            const float2 e = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            ls[k & 3] = add2(ls[k & 3], e);
            pk[k] = pack_bf16x2(e.x, e.y);
          }
          tc::tmem_st32(t_s + c * 32, pk);
        }
        const float2 lsum = add2(add2(ls[0], ls[1]), add2(ls[2], ls[3]));
        l += lsum.x + lsum.y;
        tc::tmem_wait_st();
        tc::fence_before_sync();
        // one elected arrive per warp: 128 arrivals on one barrier word serialise for hundreds
        // of cycles on the path to the next P*V
        __syncwarp();
        if (lane == 0) mbar_arrive(t == 0 ? &s.pv_full[cur % kVStages] : &s.p1_full);
      }
      if (!ok) break;
      // epilogue of the piece: O / l
      ok = __all_sync(0xffffffffu, wait_or_flag(&s.o_ready[t], jcs & 1, p.status));
      if (!ok) break;
      tc::fence_after_sync();
      if (leader) mbar_arrive(&s.v_empty[(it + nt - 1) % kVStages]);
      const int pn = pv.n, pq0 = pv.q0, pJ = pv.J, pg = pv.g;
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.piece_empty[pslot]);
      ++pk;
      const bool live = qrow < pn;
      const float inv = 1.0f / l;
      const bool whole = pjb == 0 && pjb + nt == pJ;
      const int head = 2 * pg + t;
      // all of O's 128 columns loaded at once (the scores' registers are free here), one wait;
      // O's TMEM columns are then released to the next piece's first P*V before the stores
      uint32_t oall[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(t_o + c * 32, oall[c]);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.o_free[t]);
      if (whole) {
        uint16_t* dst = p.out + (static_cast<int64_t>(pq0 + qrow) * p.hq + head) * kHeadDim;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t (&o32)[32] = oall[c];
          if (live) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o32[8 * k + 0]) * inv, __uint_as_float(o32[8 * k + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(o32[8 * k + 2]) * inv, __uint_as_float(o32[8 * k + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(o32[8 * k + 4]) * inv, __uint_as_float(o32[8 * k + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(o32[8 * k + 6]) * inv, __uint_as_float(o32[8 * k + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + c * 32 + 8 * k) = w;
            }
          }
        }
        if (live && p.lse != nullptr)
          p.lse[static_cast<int64_t>(pq0 + qrow) * p.hq + head] = (m_used + log2f(l)) * kLn2;
      } else {
        // a piece of a job shared with neighbouring CTAs: slot 1 if it starts the job, else 0.
        // A row that saw no key in this piece contributes nothing: o = 0, lse = -inf.
        const int slot = pjb == 0 ? 1 : 0;
        const bool empty = m_used == -CUDART_INF_F;
        const float sc_o = empty ? 0.f : inv;
        uint8_t* rec = p.ws_records + (2 * static_cast<size_t>(blockIdx.x) + slot) * kRecordBytes;
        float4* dst = reinterpret_cast<float4*>(rec) + t * 32 * 128 + r;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t (&o32)[32] = oall[c];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[(c * 8 + k) * 128] =
                make_float4(__uint_as_float(o32[4 * k]) * sc_o, __uint_as_float(o32[4 * k + 1]) * sc_o,
                            __uint_as_float(o32[4 * k + 2]) * sc_o, __uint_as_float(o32[4 * k + 3]) * sc_o);
        }
        reinterpret_cast<float*>(rec + kRecordO)[t * 128 + r] =
            empty ? -CUDART_INF_F : (m_used + log2f(l)) * kLn2;
      }
      it += nt;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc<512>(tmem);
  }
}

// Combine the pieces of jobs that were cut by CTA range boundaries. Eight CTAs per job (two
// heads x four 32-dim quarters), one thread per row. The pieces are slot 1 of the first CTA and
// slot 0 of each later CTA.
__global__ void __launch_bounds__(kMergeRows) prefill_merge_kernel(const PrefillTcParams p) {
  // programmatic dependent of prefill_tc_kernel: wait until that grid is complete and visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // CTA (qt, g * 8 + t * 4 + quarter, b), counted from the end of the grid: rows of query tile
  // qt, head 2g + t, dims 32 * quarter .. +31; one thread per row. A job cut into pieces is
  // merged by 8 CTAs, so the few split jobs of a call are spread over many SMs instead of one CTA
  // each. The split jobs are the last ones (the whole-job rounds take the first), so the grid is
  // walked backwards: their CTAs start first and the rest only check and exit.
  const int b = gridDim.z - 1 - blockIdx.z;
  const int y = gridDim.y - 1 - blockIdx.y;
  const int g = y >> 3, t = (y >> 2) & 1, quarter = y & 3;
  const int qt = gridDim.x - 1 - blockIdx.x;
  const SeqGeom s = seq_geom(p, b, false);
  if (qt >= s.nqt) return;
  const int jo = p.ws_job_prefix[b] + g * s.nqt + qt;
  if (jo < p.ws_header[3]) return;  // done whole in the round-robin phase
  const int G = min(static_cast<int>(p.ws_header[0]), kThreads);  // the prefill grid, <= kThreads
  const long long u0 = p.ws_prefix[b] + g * s.T + units_before(s, qt);
  const long long J = tiles_of(s, qt);
  // the split's range starts, staged in shared memory: one round of loads instead of a chain of
  // dependent ones per binary search
  __shared__ long long tail[kThreads + 1];
  for (int i = threadIdx.x; i <= G; i += kMergeRows) tail[i] = p.ws_tail[i];
  __syncthreads();
  // the CTA whose range [tail[c], tail[c + 1]) holds unit u (the last c with a start <= u: a CTA
  // with an empty range shares its start with the next one)
  auto cta_of = [&](long long u) {
    int lo = 0, hi = G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tail[mid] <= u) lo = mid; else hi = mid;
    }
    return lo;
  };
  const int c0 = cta_of(u0), c1 = cta_of(u0 + J - 1);
  if (c0 == c1) return;
  const int r = threadIdx.x;
  const int qrow = qt * kTileM + r;
  if (qrow >= s.n) return;
  // the piece in CTA c0 starts the job (slot 1); later CTAs hold continuations (slot 0); CTAs with
  // an empty range in between hold nothing
  auto rec_of = [&](int c) {
    return p.ws_records + (2 * static_cast<size_t>(c) + (c == c0 ? 1 : 0)) * kRecordBytes;
  };
  auto empty_range = [&](int c) { return tail[c] == tail[c + 1]; };
  float m = -CUDART_INF_F;
  for (int c = c0; c <= c1; ++c)
    if (!empty_range(c)) m = fmaxf(m, reinterpret_cast<const float*>(rec_of(c) + kRecordO)[t * 128 + r]);
  float acc[32];
#pragma unroll
  for (int d = 0; d < 32; ++d) acc[d] = 0.f;
  float sum = 0.f;
#pragma unroll 2
  for (int c = c0; c <= c1; ++c) {
    if (empty_range(c)) continue;
    const uint8_t* rec = rec_of(c);
    const float lp = reinterpret_cast<const float*>(rec + kRecordO)[t * 128 + r];
    if (lp == -CUDART_INF_F) continue;  // the piece held no key visible to this row
    const float w = fast_exp2((lp - m) * kLog2e);
    sum += w;
    const float4* o = reinterpret_cast<const float4*>(rec) + (t * 32 + quarter * 8) * 128 + r;
    float4 v[8];
#pragma unroll
    for (int d = 0; d < 8; ++d) v[d] = o[d * 128];
#pragma unroll
    for (int d = 0; d < 8; ++d) {
      acc[4 * d] += w * v[d].x;
      acc[4 * d + 1] += w * v[d].y;
      acc[4 * d + 2] += w * v[d].z;
      acc[4 * d + 3] += w * v[d].w;
    }
  }
  const float inv = 1.0f / sum;
  const int head = 2 * g + t;
  uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(s.q0 + qrow) * p.hq + head) * kHeadDim +
                                        32 * quarter);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint4 w;
    w.x = pack_bf16x2(acc[8 * k + 0] * inv, acc[8 * k + 1] * inv);
    w.y = pack_bf16x2(acc[8 * k + 2] * inv, acc[8 * k + 3] * inv);
    w.z = pack_bf16x2(acc[8 * k + 4] * inv, acc[8 * k + 5] * inv);
    w.w = pack_bf16x2(acc[8 * k + 6] * inv, acc[8 * k + 7] * inv);
    dst[k] = w;
  }
  if (quarter == 0 && p.lse != nullptr)
    p.lse[static_cast<int64_t>(s.q0 + qrow) * p.hq + head] = m + logf(sum);
}

// ---------------------------------------------------------------------------------------------
// host side: tensor maps (driver entry point looked up once), workspace layout, launch
// ---------------------------------------------------------------------------------------------
size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct PrefillWs {
  size_t header, prefix, job_prefix, tail, records, total;
};

PrefillWs prefill_ws(int batch, int grid) {
  PrefillWs w;
  w.header = 0;
  w.prefix = 256;
  w.job_prefix = align256(w.prefix + sizeof(long long) * (batch + 1));
  w.tail = align256(w.job_prefix + sizeof(int32_t) * (batch + 1));
  w.records = align256(w.tail + sizeof(long long) * (grid + 1));
  w.total = align256(w.records + 2 * static_cast<size_t>(grid) * kRecordBytes);
  return w;
}

// One persistent CTA per SM; plan_split gives each CTA one thread of its CTA, so at most kThreads.
int prefill_grid() { return std::min(sm_count_current_device(), kThreads); }

}  // namespace

size_t prefill_workspace_bytes(int batch) {
  const int grid = prefill_grid();
  if (grid <= 0 || batch < 0) return 0;
  return prefill_ws(batch, grid).total;
}

pa_status launch_prefill_tc(int32_t hkv, const void* q, int32_t total_q, const int32_t* cu_q_lens,
                            const void* k_pool, const void* v_pool, int64_t num_pages,
                            const int32_t* block_table, int32_t bt_stride,
                            const int32_t* seq_lens, int32_t batch, int32_t max_q_len,
                            float softmax_scale, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, int32_t* status, cudaStream_t stream,
                            int32_t max_ctas) {
  if (batch > kMaxBatch) {
    snprintf_error("attn_prefill_chunk: at most %d chunks per call", kMaxBatch);
    return PA_ERR_UNSUPPORTED;
  }
  if (num_pages * kPage >= (int64_t(1) << 31) || total_q >= (1 << 24)) return PA_ERR_UNSUPPORTED;
  const int full_grid = prefill_grid();
  if (full_grid <= 0) return PA_ERR_CUDA;
  // one persistent CTA per SM, or fewer when the caller caps the grid (the plan adapts to it)
  const int grid = max_ctas > 0 ? std::min(full_grid, static_cast<int>(max_ctas)) : full_grid;
  const PrefillWs w = prefill_ws(batch, grid);
  if (workspace == nullptr || workspace_bytes < w.total) return PA_ERR_WORKSPACE_TOO_SMALL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PA_ERR_INVALID_ARG;
  CUtensorMap qm, km, vm;
  const int hq = kGroup * hkv;
  if (!make_map_3d(&qm, q, static_cast<uint64_t>(total_q), hq, kTileM) ||
      !make_map_3d(&km, k_pool, static_cast<uint64_t>(num_pages) * kPage, hkv, kPage) ||
      !make_map_3d(&vm, v_pool, static_cast<uint64_t>(num_pages) * kPage, hkv, kPage)) {
    snprintf_error("cuTensorMapEncodeTiled failed for the prefill operands");
    return PA_ERR_CUDA;
  }
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  const int smem = static_cast<int>(sizeof(PrefillTcSmem));
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return record_cuda_error(e, "cudaFuncSetAttribute(prefill_tc)");
    // same carveout for the shared-memory-free merge kernel: no reconfiguration between them
    e = cudaFuncSetAttribute(prefill_merge_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return record_cuda_error(e, "cudaFuncSetAttribute(prefill merge)");
    // The in-kernel register split needs the full launch budget; a build that launched with
    // fewer registers per thread would make setmaxnreg.inc wait forever, so refuse to launch.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, prefill_tc_kernel);
    if (e != cudaSuccess) return record_cuda_error(e, "cudaFuncGetAttributes(prefill_tc)");
    if (fa.numRegs < kLaunchRegs) {
      snprintf_error("prefill_tc_kernel built with %d registers/thread, needs %d for its split",
                     fa.numRegs, kLaunchRegs);
      return PA_ERR_UNSUPPORTED;
    }
    configured_device = dev;
  }
  PrefillTcParams p;
  p.hkv = hkv;
  p.hq = hq;
  p.cu_q_lens = cu_q_lens;
  p.seq_lens = seq_lens;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.batch = batch;
  p.num_pages = num_pages;
  p.scale_log2 = softmax_scale * kLog2e;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.status = status;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.ws_header = reinterpret_cast<long long*>(ws + w.header);
  p.ws_prefix = reinterpret_cast<long long*>(ws + w.prefix);
  p.ws_job_prefix = reinterpret_cast<int32_t*>(ws + w.job_prefix);
  p.ws_tail = reinterpret_cast<long long*>(ws + w.tail);
  p.ws_records = ws + w.records;
  prefill_tc_kernel<<<grid, kThreads, smem, stream>>>(qm, km, vm, p);
  PA_CHECK_LAUNCH("prefill_tc_kernel");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((max_q_len + kTileM - 1) / kTileM, hkv * 8, batch);
  cfg.blockDim = dim3(kMergeRows);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_merge_kernel, p);
  if (e != cudaSuccess) return record_cuda_error(e, "prefill_merge_kernel");
  return PA_OK;
}

}  // namespace pa
