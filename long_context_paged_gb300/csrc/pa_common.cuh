// Device helpers shared by the kernels: bf16 unpacking, paired fp32 FMA, mbarriers, bulk
// (TMA) copies, bounded waits and the device status word. sm_103a only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

constexpr int kHeadDim = 128;
constexpr int kPage = 16;
constexpr int kHkv = 8;             // KV heads of the decoder (at most this many per call)
constexpr int kHq = 16;
constexpr int kGroup = kHq / kHkv;  // query heads per KV head

// Head counts a call accepts: the decoder's GQA 16/8, or the slice of it that one device holds
// when the KV heads are partitioned across devices (8/N KV heads with their 16/N query heads,
// N = 1, 2, 4, 8); head_dim 128 and 16-token pages.
inline bool gqa_dims_supported(const pa_dims& d) {
  const int h = d.num_kv_heads;
  return (h == 1 || h == 2 || h == 4 || h == 8) && d.num_q_heads == kGroup * h &&
         d.head_dim == kHeadDim && d.page_size == kPage;
}
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------------------------
// Host-side error bookkeeping (defined in api.cu).
// ---------------------------------------------------------------------------------------------
pa_status record_cuda_error(cudaError_t err, const char* where);
// printf-style text for pa_last_error() (calling thread).
void snprintf_error(const char* fmt, ...);
int sm_count_current_device();

#define PA_CHECK_LAUNCH(where)                                        \
  do {                                                                \
    cudaError_t e_ = cudaGetLastError();                              \
    if (e_ != cudaSuccess) return ::pa::record_cuda_error(e_, where); \
  } while (0)

// ---------------------------------------------------------------------------------------------
// Device status word.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void flag_error(int32_t* status, uint32_t bit) {
  if (status != nullptr) atomicOr(reinterpret_cast<unsigned int*>(status), bit);
}

// ---------------------------------------------------------------------------------------------
// bf16 <-> fp32.  A bf16 is the upper 16 bits of the fp32 with the same value, so widening is
// a shift (low half) or a mask (high half) of the packed 32-bit word.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// fp32 -> bf16 round-to-nearest-even of two values, packed (lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Paired fp32 FMA (one instruction for two lanes of a float2): d = a * b + c, each rounded.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------------------------
// Shared-memory addressing, mbarriers and bulk copies (PTX ISA: mbarrier, cp.async.bulk).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase. Gives up after `limit_ns` of wall time (checked every
// 64 polls) and returns false; the caller then flags PA_DEV_ERR_TIMEOUT and unwinds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: kernels here finish in milliseconds

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later); like fmaxf, a NaN
// operand is ignored when another operand is a number.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Bulk global->shared copy completing on an mbarrier (bytes: multiple of 16, both addresses
// 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 16-byte shared-memory load (a plain C++ load, so it stays ordered after the "memory"
// clobber of the mbarrier waits).
__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

}  // namespace pa
