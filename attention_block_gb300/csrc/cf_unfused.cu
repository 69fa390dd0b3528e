// cf_unfused.cu -- the same decode step as three separate kernels with their
// intermediates in HBM, the unfused layout the fused kernel is measured
// against ([CF §1.1] the three-kernel baseline, page "ClusterFusion框架深度解析"
// (devpress.csdn.net); the operations of [LNA §三], page "大模型推理中的算子融合优化：
// LayerNorm + Attention" (asdsk.com)):
//
//   1. uf_proj_kernel:  y = (x ∘ g) · W_qkv                  (fp32 [B, C] to HBM)
//   2. uf_attn_kernel:  r = rsqrt(mean x² + eps); q, k, v = r·y; RoPE; KV append;
//                       split-KV online softmax; the last split of each
//                       (row, KV head) combines the partials -> o (fp32 [B, nq·d])
//   3. uf_proj_kernel:  acc += o · W_o (split over the reduction, fp32 atomics);
//                       the last block of each output tile writes out = x + acc
//
// Plain CUDA-core code: each projection block streams a 64-column band of the
// weight (16-byte loads, eight batch rows per block), the attention is a
// warp-per-position flash-decoding loop.  It computes what the fused kernel
// computes and is checked against the same float64 oracle.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "cf.h"
#include "cf_common.cuh"
#include "cf_params.h"
#include "cf_unfused.h"

namespace cf {

namespace {

constexpr int kUfThreads = 256;
constexpr int kUfKC = 512;  // reduction rows staged per step
constexpr int kUfU = 8;     // weight rows in flight per lane group

// One BAND-column band of out[b0..b0+BT, :] += in[b0.., kbeg..kend] · W[kbeg..kend,
// band] (grid [ncol/BAND, nbt, KS]).  Lane l reads the 16-byte chunk
// (l % (BAND/EV)) of row (l / (BAND/EV)) of each group of rows, several groups
// in flight; the first band of the QKV projection also writes the rows' RMSNorm
// scales; the in
// rows (x ∘ g for the QKV projection, o for the output projection) are staged
// in fp32.  The KS reduction splits add into fp32 y (mode 0, zeroed again by
// its reader) or acc (mode 1, whose last block per output tile adds the
// residual and writes out).
template <typename T, int MODE, int BT, int BAND>
__global__ void __launch_bounds__(kUfThreads, 2) uf_proj_kernel(const UfParams p) {
  constexpr int U = BT == 1 ? kUfU : kUfU / 2;  // weight rows in flight per lane group
  __shared__ float xs[BT][kUfKC];
  __shared__ float red[kUfThreads / 32][BT][BAND];
  __shared__ int last;
  constexpr int EV = 16 / (int)sizeof(T);  // columns per 16-byte chunk
  constexpr int CPR = BAND / EV;           // chunks per band row
  constexpr int RG = 32 / CPR;             // rows per warp step
  constexpr int NWP = kUfThreads / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cc = lane % CPR, ro = lane / CPR;
  const int c0 = blockIdx.x * BAND, b0 = blockIdx.y * BT;
  const int K = MODE == 0 ? p.H : p.nq * p.D;
  const int ncol = MODE == 0 ? (p.nq + 2 * p.nkv) * p.D : p.H;
  const int kper = K / gridDim.z, kbeg = blockIdx.z * kper, kend = kbeg + kper;
  const T* W = reinterpret_cast<const T*>(MODE == 0 ? p.w_qkv : p.w_o);
  const T* x = reinterpret_cast<const T*>(p.hidden);
  const T* g = reinterpret_cast<const T*>(p.ln_w);
  float acc[BT][EV];
#pragma unroll
  for (int b = 0; b < BT; ++b)
#pragma unroll
    for (int e = 0; e < EV; ++e) acc[b][e] = 0.f;
  for (int kc = kbeg; kc < kend; kc += kUfKC) {
    const int kn = min(kUfKC, kend - kc);
    __syncthreads();
    for (int i = tid; i < BT * kUfKC; i += kUfThreads) {
      const int b = i / kUfKC, k = i % kUfKC;
      float v = 0.f;
      if (b0 + b < p.B && k < kn) {
        if (MODE == 0)
          v = Elem<T>::to_f(x[(size_t)(b0 + b) * p.H + kc + k]) * Elem<T>::to_f(g[kc + k]);
        else
          v = p.o32[(size_t)(b0 + b) * K + kc + k];
      }
      xs[b][k] = v;
    }
    __syncthreads();
    const T* wb = W + (size_t)kc * ncol + c0 + cc * EV;
    for (int k = warp * RG + ro; k < kn; k += NWP * RG * U) {
      float wv[U][EV];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int kk = k + u * NWP * RG;
        if (kk < kn) load_cvt<T, EV>(wb + (size_t)kk * ncol, wv[u]);
        else
#pragma unroll
          for (int e = 0; e < EV; ++e) wv[u][e] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int kk = min(k + u * NWP * RG, kUfKC - 1);
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          const float xv = xs[b][kk];
#pragma unroll
          for (int e = 0; e < EV; ++e) acc[b][e] = fmaf(xv, wv[u][e], acc[b][e]);
        }
      }
    }
  }
  // sum the lanes that share a chunk (rows of the group), then the warps
#pragma unroll
  for (int off = CPR; off < 32; off <<= 1)
#pragma unroll
    for (int b = 0; b < BT; ++b)
#pragma unroll
      for (int e = 0; e < EV; ++e) acc[b][e] += __shfl_xor_sync(0xffffffffu, acc[b][e], off);
  if (ro == 0)
#pragma unroll
    for (int b = 0; b < BT; ++b)
#pragma unroll
      for (int e = 0; e < EV; ++e) red[warp][b][cc * EV + e] = acc[b][e];
  __syncthreads();
  // RMSNorm scales of the rows, once (QKV projection, first band and split)
  if (MODE == 0 && blockIdx.x == 0 && blockIdx.z == 0) {
    for (int b = warp; b < BT; b += NWP) {
      float ss = 0.f;
      if (b0 + b < p.B)
        for (int i = lane; i < p.H; i += 32) {
          const float v = Elem<T>::to_f(x[(size_t)(b0 + b) * p.H + i]);
          ss = fmaf(v, v, ss);
        }
      ss = warp_sum(ss);
      if (lane == 0 && b0 + b < p.B) p.rinv[b0 + b] = 1.0f / sqrtf(ss / (float)p.H + p.eps);
    }
  }
  for (int i = tid; i < BT * BAND; i += kUfThreads) {
    const int b = i / BAND, c = i % BAND;
    if (b0 + b >= p.B) continue;
    float v = 0.f;
    for (int w = 0; w < NWP; ++w) v += red[w][b][c];
    if (MODE == 0) atomicAdd(p.y + (size_t)(b0 + b) * ncol + c0 + c, v);
    else atomicAdd(p.acc + (size_t)(b0 + b) * p.H + c0 + c, v);
  }
  if (MODE == 1) {
    __threadfence();
    __syncthreads();
    int* cnt = p.cnt_out + blockIdx.y * gridDim.x + blockIdx.x;
    if (tid == 0) {
      const int t = atomicAdd(cnt, 1);
      last = (t == (int)gridDim.z - 1);
      if (last) __threadfence();
    }
    __syncthreads();
    if (last) {
      T* out = reinterpret_cast<T*>(p.out);
      for (int i = tid; i < BT * BAND; i += kUfThreads) {
        const int b = i / BAND, c = i % BAND;
        if (b0 + b >= p.B) continue;
        const size_t off = (size_t)(b0 + b) * p.H + c0 + c;
        const float v = __ldcg(p.acc + off);
        __stcg(p.acc + off, 0.f);
        out[off] = Elem<T>::from_f(Elem<T>::to_f(x[off]) + v);
      }
      if (tid == 0) *cnt = 0;
    }
  }
}

// Split-KV attention of batch row b, KV head g, position split s (grid
// [NS, nkv, B]).  Each warp takes every 8th cached position of the split;
// lane l owns head dims [l*D/32, (l+1)*D/32) of the G query heads.
template <typename T, int D, int G>
__global__ void __launch_bounds__(kUfThreads, 2) uf_attn_kernel(const UfParams p) {
  constexpr int NW = kUfThreads / 32;
  __shared__ float q[G][D], kn[D], vn[D];
  __shared__ float ws[NW][G][D + 2];
  __shared__ float s_r;
  __shared__ int last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z, NS = gridDim.x;
  const int C = (p.nq + 2 * p.nkv) * D;
  const T* x = reinterpret_cast<const T*>(p.hidden) + (size_t)b * p.H;
  int pos = p.positions[b];
  if (pos < 0 || pos >= p.S) {
    if (s == 0 && g == 0 && tid == 0) atomicOr(p.errflag, kDevErrPosRange);
    pos = -1;
  }
  if (tid == 0) s_r = p.rinv[b];  // RMSNorm scale (from the QKV projection)
  __syncthreads();
  // q, k, v of the head group: scale, RoPE (rotate-half), append
  const float* y = p.y + (size_t)b * C;
  for (int i = tid; i < (G + 2) * (D / 2); i += kUfThreads) {
    const int sg = i / (D / 2), j = i % (D / 2);
    const int col = sg < G ? (g * G + sg) * D : (sg == G ? (p.nq + g) * D : (p.nq + p.nkv + g) * D);
    float a = y[col + j] * s_r, bv = y[col + j + D / 2] * s_r;
    if (sg <= G && pos >= 0) {
      float c, sn;
      rope_cos_sin(pos, p.turn_hi[j], p.turn_lo[j], c, sn);
      const float ra = a * c - bv * sn, rb = bv * c + a * sn;
      a = ra;
      bv = rb;
    }
    float* dst = sg < G ? q[sg] : (sg == G ? kn : vn);
    dst[j] = a;
    dst[j + D / 2] = bv;
    if (sg >= G && s == 0 && pos >= 0) {
      T* cache = reinterpret_cast<T*>(sg == G ? p.k_cache : p.v_cache);
      const size_t base = (((size_t)b * p.S + pos) * p.nkv + g) * D;
      cache[base + j] = Elem<T>::from_f(a);
      cache[base + j + D / 2] = Elem<T>::from_f(bv);
    }
  }
  __syncthreads();
  // this split's positions of the cached keys 0..pos-1: LPP lanes per
  // position (8, or 16 for grouped heads), each lane D/LPP dims of the G heads
  constexpr int LPP = G >= 4 ? 16 : 8, NGRP = 32 / LPP, DPL = D / LPP;
  constexpr int EP = 16 / (int)sizeof(T) < DPL ? 16 / (int)sizeof(T) : DPL;  // elements per load
  const int grp = lane / LPP, kl = lane % LPP;
  float qr[G][DPL], o[G][DPL], m[G], l[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      qr[h][e] = q[h][kl * DPL + e] * p.qk_scale_log2;
      o[h][e] = 0.f;
    }
  }
  auto update = [&](const float (&sc)[G], const float* vf, bool ok) {
    if (!ok) return;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mn = fmaxf(m[h], sc[h]);
      const float al = exp2f(m[h] - mn), pe = exp2f(sc[h] - mn);
      l[h] = fmaf(l[h], al, pe);
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(o[h][e], al, pe * vf[e]);
      m[h] = mn;
    }
  };
  auto scores = [&](const float* kf, float (&sc)[G]) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; e += 2) {
        a0 = fmaf(qr[h][e], kf[e], a0);
        a1 = fmaf(qr[h][e + 1], kf[e + 1], a1);
      }
      sc[h] = a0 + a1;
    }
  };
  if (pos > 0) {
    const int ch = (pos + NS - 1) / NS;
    const int t0 = s * ch, t1 = min(pos, t0 + ch);
    const T* kc = reinterpret_cast<const T*>(p.k_cache);
    const T* vc = reinterpret_cast<const T*>(p.v_cache);
    constexpr int UP = 2;  // positions per lane group per step
    for (int tb = t0 + warp * NGRP * UP; tb < t1; tb += NW * NGRP * UP) {
      float kf[UP][DPL], vf[UP][DPL], sc[UP][G];
      bool ok[UP];
#pragma unroll
      for (int u = 0; u < UP; ++u) {
        const int t = tb + u * NGRP + grp;
        ok[u] = t < t1;
        const size_t base = (((size_t)b * p.S + (ok[u] ? t : t0)) * p.nkv + g) * D + kl * DPL;
#pragma unroll
        for (int c = 0; c < DPL / EP; ++c) {
          load_cvt<T, EP>(kc + base + c * EP, kf[u] + c * EP);
          load_cvt<T, EP>(vc + base + c * EP, vf[u] + c * EP);
        }
        scores(kf[u], sc[u]);
      }
#pragma unroll
      for (int off = LPP / 2; off >= 1; off >>= 1)
#pragma unroll
        for (int u = 0; u < UP; ++u)
#pragma unroll
          for (int h = 0; h < G; ++h) sc[u][h] += __shfl_xor_sync(0xffffffffu, sc[u][h], off);
#pragma unroll
      for (int u = 0; u < UP; ++u) update(sc[u], vf[u], ok[u]);
    }
  }
  if (s == NS - 1 && warp == 0 && pos >= 0) {  // the new token, by lane group 0
    float kf[DPL], vf[DPL], sc[G];
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      kf[e] = kn[kl * DPL + e];
      vf[e] = vn[kl * DPL + e];
    }
    scores(kf, sc);
#pragma unroll
    for (int off = LPP / 2; off >= 1; off >>= 1)
#pragma unroll
      for (int h = 0; h < G; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], off);
    update(sc, vf, grp == 0);
  }
  // merge the lane groups of the warp
#pragma unroll
  for (int off = LPP; off < 32; off <<= 1)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
      const float lo = __shfl_xor_sync(0xffffffffu, l[h], off);
      const float mn = fmaxf(m[h], mo);
      const float a = mn == -INFINITY ? 0.f : exp2f(m[h] - mn);
      const float bsc = mn == -INFINITY ? 0.f : exp2f(mo - mn);
      l[h] = l[h] * a + lo * bsc;
#pragma unroll
      for (int e = 0; e < DPL; ++e) {
        const float oo = __shfl_xor_sync(0xffffffffu, o[h][e], off);
        o[h][e] = o[h][e] * a + oo * bsc;
      }
      m[h] = mn;
    }
  // merge the warps, write this split's partial (o, m, l)
  if (grp == 0)
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int e = 0; e < DPL; ++e) ws[warp][h][kl * DPL + e] = o[h][e];
      if (kl == 0) {
        ws[warp][h][D] = m[h];
        ws[warp][h][D + 1] = l[h];
      }
    }
  __syncthreads();
  const int PW = D + 4;
  float* part = p.part + (((size_t)b * p.nkv + g) * NS + s) * G * PW;
  for (int i = tid; i < G * D; i += kUfThreads) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, ws[w][h][D]);
    float O = 0.f, L = 0.f;
    if (M != -INFINITY)
      for (int w = 0; w < NW; ++w) {
        const float f = exp2f(ws[w][h][D] - M);
        O = fmaf(f, ws[w][h][d], O);
        L = fmaf(f, ws[w][h][D + 1], L);
      }
    part[h * PW + d] = O;
    if (d == 0) {
      part[h * PW + D] = M;
      part[h * PW + D + 1] = L;
    }
  }
  // the last split of (b, g) combines the NS partials into o
  __threadfence();
  __syncthreads();
  int* cnt = p.cnt_attn + b * p.nkv + g;
  if (tid == 0) {
    const int t = atomicAdd(cnt, 1);
    last = (t == NS - 1);
    if (last) __threadfence();
  }
  __syncthreads();
  if (!last) return;
  const float* pb = p.part + ((size_t)b * p.nkv + g) * NS * G * PW;
  for (int i = tid; i < G * D; i += kUfThreads) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
    for (int s2 = 0; s2 < NS; ++s2) M = fmaxf(M, __ldcg(pb + (s2 * G + h) * PW + D));
    float O = 0.f, L = 0.f;
    if (M != -INFINITY)
      for (int s2 = 0; s2 < NS; ++s2) {
        const float* pp = pb + (s2 * G + h) * PW;
        const float f = exp2f(__ldcg(pp + D) - M);
        O = fmaf(f, __ldcg(pp + d), O);
        L = fmaf(f, __ldcg(pp + D + 1), L);
      }
    p.o32[((size_t)b * p.nq + g * G + h) * D + d] = (L > 0.f) ? O / L : 0.f;
  }
  // the projection rows of this group are consumed: clear them for the
  // next step's accumulating projection
  for (int i = tid; i < (G + 2) * D; i += kUfThreads) {
    const int sg = i / D, j = i % D;
    const int col = sg < G ? (g * G + sg) * D : (sg == G ? (p.nq + g) * D : (p.nq + p.nkv + g) * D);
    p.y[(size_t)b * C + col + j] = 0.f;
  }
  if (tid == 0) *cnt = 0;
}

// 128-column bands (256-byte row segments) where the column count allows,
// else 64
template <typename T, int BT>
void launch_proj(const UfParams& p, int mode, int ks, cudaStream_t st) {
  const int ncol = mode == 0 ? (p.nq + 2 * p.nkv) * p.D : p.H;
  const dim3 g64(ncol / 64, (p.B + BT - 1) / BT, ks), g128(ncol / 128, (p.B + BT - 1) / BT, ks);
  const bool wide = ncol % 128 == 0;
  if (mode == 0) {
    if (wide) uf_proj_kernel<T, 0, BT, 128><<<g128, kUfThreads, 0, st>>>(p);
    else uf_proj_kernel<T, 0, BT, 64><<<g64, kUfThreads, 0, st>>>(p);
  } else {
    if (wide) uf_proj_kernel<T, 1, BT, 128><<<g128, kUfThreads, 0, st>>>(p);
    else uf_proj_kernel<T, 1, BT, 64><<<g64, kUfThreads, 0, st>>>(p);
  }
}

template <typename T>
int launch_all(const UfParams& p, int G, cudaStream_t st) {
  const bool one = p.B == 1;
  if (one) launch_proj<T, 1>(p, 0, p.KS1, st);
  else launch_proj<T, 8>(p, 0, p.KS1, st);
  const dim3 ga(p.NS, p.nkv, p.B);
  if (p.D == 128 && G == 1) uf_attn_kernel<T, 128, 1><<<ga, kUfThreads, 0, st>>>(p);
  else if (p.D == 128 && G == 4) uf_attn_kernel<T, 128, 4><<<ga, kUfThreads, 0, st>>>(p);
  else if (p.D == 64 && G == 1) uf_attn_kernel<T, 64, 1><<<ga, kUfThreads, 0, st>>>(p);
  else if (p.D == 64 && G == 4) uf_attn_kernel<T, 64, 4><<<ga, kUfThreads, 0, st>>>(p);
  else return CF_ERR_UNSUPPORTED;
  if (one) launch_proj<T, 1>(p, 1, p.KS, st);
  else launch_proj<T, 8>(p, 1, p.KS, st);
  return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}

}  // namespace

int unfused_launch(const UfParams& p, int dtype, int G, cudaStream_t st) {
  if (dtype == CF_F32) return launch_all<float>(p, G, st);
  if (dtype == CF_F16) return launch_all<__half>(p, G, st);
  return launch_all<__nv_bfloat16>(p, G, st);
}

}  // namespace cf
