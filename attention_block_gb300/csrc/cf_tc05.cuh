// cf_tc05.cuh -- fifth-generation tensor-core (tcgen05) helpers for sm_103a:
// tensor-memory (TMEM) allocation, the shared-memory matrix descriptor of a
// K-major operand written with the 128-byte swizzle, the instruction
// descriptor of kind::f16, the MMA itself, its commit to an mbarrier, and
// TMEM loads.  Inline PTX only.
//
// Conventions used throughout:
//   * one CTA (cta_group::1); the MMA is issued by a single thread;
//   * A is M x K and B is N x K.  A K-major operand lies in slabs of 64
//     16-bit elements (128 bytes) per row, rows of a slab consecutive and
//     8-row groups 1024 bytes apart; an M-major A lies in 64-column boxes of
//     K rows of 128 bytes (the layout a 2D TMA load with the 128-byte swizzle
//     writes).  Inside a 128-byte row r the 16-byte chunk j sits at chunk
//     j ^ (r & 7) (the 128-byte swizzle); slab and box bases are 1024-byte
//     aligned;
//   * the fp32 accumulator D (M = 128) occupies TMEM lanes 0..127 (row m in
//     lane m) and N consecutive columns from the allocation's base column.
#pragma once

#include <stdint.h>

#include "cf_ptx.cuh"

namespace cf {

// Allocate `ncols` TMEM columns (a power of two, 32..512) for this CTA; the
// whole warp executes it and the TMEM address lands in the shared word `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// Free the allocation (the warp that allocated, after every use).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Order tcgen05 operations across a thread barrier.
__device__ __forceinline__ void tc05_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc05_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand with the 128-byte
// swizzle: start address (16-byte units, bits 0-13), leading byte offset
// (bits 16-29; not used by this layout, 16 bytes), stride byte offset between
// 8-row groups (bits 32-45), descriptor version 1 (bits 46-47), base offset 0,
// layout 2 = 128-byte swizzle (bits 61-63).  A k offset inside the 128-byte
// rows is added to the start address (32 bytes per 16-element k step).
__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t saddr, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Shared-memory matrix descriptor of an M- (or N-) major operand with the
// 128-byte swizzle: rows of 64 consecutive M elements (128 bytes) along K,
// one K row every 128 bytes, 8-row K groups `sbo_bytes` apart (1024 when the
// rows are consecutive) and successive 64-element M blocks `lbo_bytes` apart
// (the distance between two 64-column TMA boxes).  A K step of 16 rows
// advances the start address by 16 * 128 bytes.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                       uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), A and B both fp16 (0) or both bf16 (1) (bits 7-9, 10-12), A
// M-major (bit 15 = 1) or K-major (0), B K-major (bit 16 = 0), N >> 3 (bits
// 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_kind_f16(bool bf16, int M, int N,
                                                      bool a_mn = false) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[adesc] . B[bdesc]^T for one K step of 16 elements; issued by
// one thread.  accumulate = false overwrites D.
__device__ __forceinline__ void tc05_mma_f16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive (once) on `bar` when every MMA this thread issued so far completes.
__device__ __forceinline__ void tc05_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 8 consecutive fp32 columns of the 32 TMEM lanes of this warp's quarter
// (warp w % 4 reads lanes 32 (w % 4) .. +31; taddr carries the lane base in
// bits 16-31 and the column in bits 0-15); waits for the load.
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, float (&v)[8]) {
  uint32_t r0, r1, r2, r3, r4, r5, r6, r7;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3), "=r"(r4), "=r"(r5), "=r"(r6), "=r"(r7)
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  v[0] = __uint_as_float(r0);
  v[1] = __uint_as_float(r1);
  v[2] = __uint_as_float(r2);
  v[3] = __uint_as_float(r3);
  v[4] = __uint_as_float(r4);
  v[5] = __uint_as_float(r5);
  v[6] = __uint_as_float(r6);
  v[7] = __uint_as_float(r7);
}

// 16 consecutive fp32 columns of the warp's 32 TMEM lanes, without waiting:
// call tmem_wait_ld() before using v (several loads can share one wait).
__device__ __forceinline__ void tmem_ld_32x32b_x16_nowait(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
// 8 consecutive fp32 columns of the warp's 32 TMEM lanes, without waiting.
__device__ __forceinline__ void tmem_ld_32x32b_x8_nowait(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7])
      : "r"(taddr));
}
// N (8 or 16) consecutive fp32 columns, without waiting.
template <int N>
__device__ __forceinline__ void tmem_ld_32x32b_nowait(uint32_t taddr, uint32_t (&v)[N]) {
  static_assert(N == 8 || N == 16, "8 or 16 columns");
  if constexpr (N == 16)
    tmem_ld_32x32b_x16_nowait(taddr, v);
  else
    tmem_ld_32x32b_x8_nowait(taddr, v);
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// TMEM columns to allocate for `need` columns: a power of two, at least 32.
__host__ __device__ constexpr int tmem_cols_for(int need) {
  return need <= 32 ? 32 : (need <= 64 ? 64 : (need <= 128 ? 128 : (need <= 256 ? 256 : 512)));
}

// Wait for the phase of `bar` with the given parity, at most ~`limit` polls,
// without the early exit on a recorded error that the ring waits take: used
// before freeing TMEM, to let MMAs still in flight finish.  Returns whether
// the phase completed.
__device__ __forceinline__ bool tc05_drain(uint64_t* bar, uint32_t parity, uint32_t limit) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait_cta(a, parity)) return true;
  return false;
}

}  // namespace cf
