// cf_common.cuh -- helpers shared by the decode kernels: 16-bit/fp32
// conversions and vector loads, warp sums, the KV tile split, the RoPE angle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cf_params.h"
#include "cf_ptx.cuh"

namespace cf {

// ------------------------------------------------------------ conversions --
template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
  static __device__ __forceinline__ void words(const uint32_t* w, int nw, float* f) {
    for (int i = 0; i < nw; ++i) f[i] = __uint_as_float(w[i]);
  }
};
template <>
struct Elem<__half> {
  static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
  static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
  static __device__ __forceinline__ void words(const uint32_t* w, int nw, float* f) {
    for (int i = 0; i < nw; ++i) {
      float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
};
template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
  static __device__ __forceinline__ void words(const uint32_t* w, int nw, float* f) {
    for (int i = 0; i < nw; ++i) {
      float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
};

// Load NE contiguous elements (NE*sizeof(T) in {4, 8, 16} bytes, naturally
// aligned) and widen them to fp32.
template <typename T, int NE>
__device__ __forceinline__ void load_cvt(const T* p, float* f) {
  constexpr int B = NE * (int)sizeof(T);
  static_assert(B == 4 || B == 8 || B == 16, "vector width");
  if constexpr (B == 16) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
    Elem<T>::words(w, 4, f);
  } else if constexpr (B == 8) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    uint32_t w[2] = {u.x, u.y};
    Elem<T>::words(w, 2, f);
  } else {
    uint32_t w[1] = {*reinterpret_cast<const uint32_t*>(p)};
    Elem<T>::words(w, 1, f);
  }
}

// Store 4 consecutive elements from fp32 (round to nearest even).
template <typename T>
__device__ __forceinline__ void store4(T* p, const float* f) {
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  } else {
    T t[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) t[e] = Elem<T>::from_f(f[e]);
    *reinterpret_cast<uint2*>(p) = *reinterpret_cast<const uint2*>(t);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Position in a ring of n mbarrier-guarded slots: the slot of use `it` and
// the parity of its pass (the k-th fill of a slot completes the barrier's
// phase k), advanced by counting: a division by a runtime divisor is a long
// dependent instruction chain, paid per stage otherwise.
struct RingPos {
  int slot;
  uint32_t phase;
  __device__ __forceinline__ RingPos(int it, int n)
      : slot(it % n), phase((uint32_t)(it / n) & 1u) {}
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Position tiles [t0, t1) of the cached keys 0..pos-1 handled by block `rank`
// (balanced split of ceil(pos/Rt) tiles over N blocks).  pos < 0 marks an
// invalid row; pos == 0 has no cached key (only the new token).  Rt and N are
// powers of two (the plans make them so), so the split takes shifts and a
// 64-bit product, not divisions.
__device__ __forceinline__ void kv_tile_range(int pos, int Rt, int rank, int N, int& t0,
                                              int& t1) {
  if (pos <= 0) {
    t0 = t1 = 0;
    return;
  }
  const int lr = __ffs(Rt) - 1, ln = __ffs(N) - 1;
  const unsigned nt = ((unsigned)pos + (unsigned)(Rt - 1)) >> lr;
  t0 = (int)(((unsigned long long)rank * nt) >> ln);
  t1 = (int)(((unsigned long long)(rank + 1) * nt) >> ln);
}

// cos and sin of the RoPE angle pos * theta^(-2i/d) [LNA §三] without FP64
// (GB300's double-precision path is slow and this sits between two cluster
// exchanges).  The angle is reduced to a fraction of a turn exactly: the turn
// rate c = theta^(-2i/d) / (2 pi) comes from the host (computed in float64)
// as an unevaluated pair hi + lo of floats; pos < 2^24 is exact in fp32;
// pos*hi is split into its rounded value and exact error with one FMA
// (Dekker's two-product); subtracting the nearest integer is exact
// (Sterbenz).  The remaining fraction t, |t| <= 1/2 + 2^-20, goes to
// sincospif(2t) = (sin, cos)(2 pi t); the angle error stays below 1e-7 rad
// for every pos < 2^24.
__device__ __forceinline__ void rope_cos_sin(int pos, float hi, float lo, float& c, float& s) {
  const float pf = (float)pos;
  const float ph = pf * hi;
  const float pe = fmaf(pf, hi, -ph);
  const float fr = ph - rintf(ph);
  const float t = fr + fmaf(pf, lo, pe);
  sincospif(2.0f * t, &s, &c);
}

constexpr int kBarConsumers = 1;  // named barrier id of the 256 consumer threads

}  // namespace cf
