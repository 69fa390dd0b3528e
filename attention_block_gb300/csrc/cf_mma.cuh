// cf_mma.cuh -- warp-level tensor-core helpers for the batched projections:
// mma.sync m16n8k16 (fp16 or bf16 inputs, fp32 accumulate) and ldmatrix
// fragment loads from shared memory.
//
// Fragment conventions (one warp, lane = 0..31, gq = lane / 4, tq = lane % 4):
//   A (16x16, row-major)  4 regs: (gq, 2tq..+1), (gq+8, ..), (gq, 2tq+8..), (gq+8, ..)
//   B (16x8, k-major)     2 regs: (k = 2tq..+1, n = gq), (k = 2tq+8..+9, n = gq)
//   C (16x8, fp32)        4 regs: (gq, 2tq), (gq, 2tq+1), (gq+8, 2tq), (gq+8, 2tq+1)
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "cf_ptx.cuh"

namespace cf {

template <typename T>
struct MmaKind;  // PTX type names of the 16-bit input types
template <>
struct MmaKind<__half> {
  // The attention's fp32 operands (scaled query, probabilities) enter as one
  // fp16 value each (11 significant bits; the products still accumulate in
  // fp32): the attention output then carries a mean relative error of about
  // the fp16 unit roundoff (2.6e-4 measured on the 64-row, 2048-hidden MHA
  // layer, against a 1e-3 bound) and the block output about 1e-5.
  static constexpr bool kAttnHiLo = false;
  static constexpr bool kBf16 = false;
  static __device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  // hi = nearest 16-bit value of v, lo = nearest 16-bit value of (v - hi),
  // packed two per word (element e0 in the low half).
  static __device__ __forceinline__ void split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(v0, v1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
  }
};
template <>
struct MmaKind<__nv_bfloat16> {
  // bf16 keeps 8 significant bits: the attention operands enter as hi + lo
  // pairs (about fp32 accuracy).
  static constexpr bool kAttnHiLo = true;
  static constexpr bool kBf16 = true;
  static __device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ void split2(float v0, float v1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
  }
};

// A fragment of a 16x16 block of a row-major 16-bit matrix at `base` (row
// pitch `pitch` bytes, a multiple of 16 that is not a multiple of 128, so the
// eight rows of each 8x8 sub-matrix fall in distinct banks).
__device__ __forceinline__ void ldmatrix_a(uint32_t (&a)[4], const void* base, int pitch,
                                           int lane) {
  const int r = lane & 15, kh = lane >> 4;  // lanes 16..31 address the k+8 half
  const uint32_t addr = smem_u32(base) + r * pitch + kh * 16;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}

// ldmatrix_a for a matrix with only `nrows` stored rows: the lanes of rows
// >= nrows read the 16-byte zero chunk at `zero16` instead (the zero padding
// rows of a 16-row tile need no storage).
__device__ __forceinline__ void ldmatrix_a_rows(uint32_t (&a)[4], const void* base, int pitch,
                                                int nrows, const void* zero16, int lane) {
  const int r = lane & 15, kh = lane >> 4;
  const uint32_t addr = r < nrows ? smem_u32(base) + r * pitch + kh * 16 : smem_u32(zero16);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}

// B fragment (16 k-rows x 8 n-columns) from a TMA box written with the
// 128-byte swizzle: the box holds rows of 64 16-bit elements (128 bytes);
// the 16-byte chunk j of row k sits at chunk position j ^ (k & 7).  `box`
// must be 1024-byte aligned; k0 is a multiple of 16, n0 a multiple of 8.
__device__ __forceinline__ void ldmatrix_b_sw128(uint32_t& b0, uint32_t& b1, const void* box,
                                                 int k0, int n0, int lane) {
  const int k = k0 + (lane & 15);
  const int chunk = (n0 >> 3) ^ (k & 7);
  const uint32_t addr = smem_u32(box) + k * 128 + chunk * 16;
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(b0), "=r"(b1)
               : "r"(addr));
}

// B fragment (16 k-columns x 8 n-rows) whose columns are rows of a TMA box
// written with the 128-byte swizzle: B[k][n] = box[n0 + n][k0 + k] (box rows
// of 64 16-bit elements, base 1024-byte aligned; n0 a multiple of 8, k0 of
// 16 below 64).  Matrix i of the pair holds columns k0 + 8 i .. k0 + 8 i + 7.
__device__ __forceinline__ void ldmatrix_bt_sw128(uint32_t& b0, uint32_t& b1, const void* box,
                                                  int n0, int k0, int lane) {
  const int r = n0 + (lane & 7);
  const int chunk = ((k0 >> 3) + ((lane >> 3) & 1)) ^ (r & 7);
  const uint32_t addr = smem_u32(box) + r * 128 + chunk * 16;
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(b0), "=r"(b1)
               : "r"(addr));
}

// A fragment (16 m-rows x 16 k-columns) of the TRANSPOSE of a TMA box written
// with the 128-byte swizzle: A[m][k] = box[k0 + k][m0 + m], i.e. the 8x8
// blocks (k0..7, m0..7), (k0..7, m8..15), (k8..15, m0..7), (k8..15, m8..15)
// of the box, each transposed.  m0 is a multiple of 16 below 64, k0 of 16.
__device__ __forceinline__ void ldmatrix_at_sw128(uint32_t (&a)[4], const void* box, int k0,
                                                  int m0, int lane) {
  const int i = lane >> 3;  // sub-matrix this lane addresses
  const int k = k0 + ((i >> 1) << 3) + (lane & 7);
  const int chunk = ((m0 >> 3) + (i & 1)) ^ (k & 7);
  const uint32_t addr = smem_u32(box) + k * 128 + chunk * 16;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}

// B fragment (16 k-rows x 8 n-columns) whose columns are the rows of two
// row-major 16-bit matrices: B[k][n] = hi[n][k0 + k] for n < 4 and
// lo[n - 4][k0 + k] for n >= 4 (row pitch `pitch` bytes, a multiple of 16);
// rows >= nrows (<= 4) of either read the 16-byte zero chunk at `zero16`.
// With hi + lo the two halves of a split fp32 operand, one mma gives both
// partial products of four rows in separate accumulator columns.
__device__ __forceinline__ void ldmatrix_b_hilo_rows(uint32_t& b0, uint32_t& b1, const void* hi,
                                                     const void* lo, int pitch, int nrows,
                                                     const void* zero16, int k0, int lane) {
  const int n = lane & 7, kh = (lane >> 3) & 1;  // lanes 0..15 address the two matrices
  const int r = n & 3;
  const void* rowp = n < 4 ? hi : lo;
  const uint32_t addr =
      r < nrows ? smem_u32(rowp) + r * pitch + (k0 + kh * 8) * 2 : smem_u32(zero16);
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(b0), "=r"(b1)
               : "r"(addr));
}

// Four 8x8 16-bit matrices; lane l supplies the row address of matrix l / 8,
// row l % 8.  Register i holds matrix i in the mma fragment layout (thread t:
// row t / 4, elements 2 (t % 4) and 2 (t % 4) + 1); with .trans, matrix i is
// transposed first.
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Transpose of an 8x8 16-bit matrix held in the mma fragment layout (thread
// t: row t / 4, elements 2 (t % 4), 2 (t % 4) + 1): returns the fragment of
// the transposed matrix in the same layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// Byte offset of row r, 16-byte chunk c of a TMA box written with the
// 128-byte swizzle (rows of 128 bytes, box base 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

}  // namespace cf
