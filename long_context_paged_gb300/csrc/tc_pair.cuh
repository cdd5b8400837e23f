// tcgen05 forms for CTA pairs (.cta_group::2), written from the PTX ISA. The two CTAs of a
// cluster of 2 work as one MMA unit: one M = 256 tcgen05.mma, issued by the even CTA, reads A rows
// 0-127 from the even CTA's shared memory and rows 128-255 from the odd CTA's, B's first N/2 rows
// from the even CTA and the rest from the odd one (each at the same shared-memory offset), and
// writes each CTA's 128 accumulator rows into that CTA's TMEM. TMEM is allocated by one warp of
// each CTA together, at the same column in both. A kernel uses one .cta_group value in all its
// tcgen05 operations: a kernel that uses these forms uses none of the cta_group::1 ones.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "pa_common.cuh"

namespace pa {
namespace tc {

template <int kCols>
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_slot) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(smem_slot)),
               "n"(kCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <int kCols>
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(kCols)
               : "memory");
}
// D[tmem] (+)= A[smem] * B[smem] over the pair (issued by the even CTA only)
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at shared::cluster address `bar` (this CTA's, or the odd CTA's
// from mapa) when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// Tiled TMA load (2-D) into this CTA's shared memory, completing its bytes on the mbarrier at
// shared::cluster address `bar`, which may be the even CTA's of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int c0,
                                                 int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(smem_dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

}  // namespace tc
}  // namespace pa
