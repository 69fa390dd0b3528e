// cf_attention.cuh -- one batch row's split-KV online-softmax attention
// inside a block ([CF §3.2] 在线softmax, page "ClusterFusion框架深度解析"
// (devpress.csdn.net); GQA grouping of "大模型推理中的算子融合优化：LayerNorm +
// Attention" (asdsk.com) §三).
//
// The block's 8 consumer warps take the row's K/V position tiles from the
// TMA ring in order (the producer issues exactly the tiles of
// kv_tile_range(pos, Rt, seq_rank, seq_n)); LPP lanes share one position and
// each lane owns D/LPP head dimensions of the G query heads of the KV head.
// Scores are kept in log2 units (q pre-scaled by log2(e)/sqrt(d), exp2f).
// Each lane group keeps a running (m, l, o); the groups are merged with warp
// shuffles, the warps through shared memory, into `rec` = [G][D+4] holding
// the unnormalized o, then m at D and l at D+1.
#pragma once

#include "cf_common.cuh"
#include "cf_params.h"
#include "cf_ptx.cuh"

namespace cf {

template <typename T, int D, int G>
struct AttnShape {
  static constexpr int LPP = (4 * G < 8) ? 8 : ((4 * G > 32) ? 32 : 4 * G);  // lanes/position
  static constexpr int NGRP = 32 / LPP;
  static constexpr int DPL = D / LPP;  // dims per lane
  static constexpr int PB = (DPL * (int)sizeof(T) < 16) ? DPL * (int)sizeof(T) : 16;
  static constexpr int EP = PB / (int)sizeof(T);  // elements per load piece
  static constexpr int NPC = DPL / EP;            // pieces per lane
  static_assert(DPL % EP == 0 && NPC >= 1 && DPL % 2 == 0, "lane split");
};

// q: the row's G query heads [G][D] (fp32, post-RoPE); kn, vn: the new token's
// key and value [D] (fp32), folded in when `fold_new`; tl: this block's
// timeline row (stamps when non-null).  `it` is the consumer's ring counter.
template <typename T, int D, int G>
__device__ void attend_row(const KParams& p, const float* q_in, const float* kn, const float* vn,
                           int pos, int seq_rank, int seq_n, bool fold_new,
                           uint8_t* ring, uint64_t* full, uint64_t* empty, int& it, float* wst,
                           float* rec, unsigned long long* tl) {
  using S = AttnShape<T, D, G>;
  constexpr int LPP = S::LPP, NGRP = S::NGRP, DPL = S::DPL, EP = S::EP, NPC = S::NPC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane / LPP, kl = lane % LPP;
  float q[G][DPL], o[G][DPL], m[G], l[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int i = 0; i < NPC; ++i)
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        const int dim = (kl + i * LPP) * EP + e;
        q[h][i * EP + e] = q_in[h * D + dim] * p.qk_scale_log2;
        o[h][i * EP + e] = 0.f;
      }
  }
  // Two positions' contribution to this lane group's running state: the two
  // dot products, reductions and exponentials are independent
  // (instruction-level parallelism); the state is rescaled once.
  auto score = [&](const T* krow, float (&sc)[G]) {
    float kf[DPL];
#pragma unroll
    for (int i = 0; i < NPC; ++i) load_cvt<T, EP>(krow + (kl + i * LPP) * EP, kf + i * EP);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; e += 2) {
        s0 = fmaf(q[h][e], kf[e], s0);
        s1 = fmaf(q[h][e + 1], kf[e + 1], s1);
      }
      sc[h] = s0 + s1;
    }
  };
  auto consume2 = [&](const T* kA, const T* vA, bool okA, const T* kB, const T* vB, bool okB) {
    float sa[G], sb[G];
    score(kA, sa);
    score(kB, sb);
#pragma unroll
    for (int off = LPP / 2; off >= 1; off >>= 1)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        sa[h] += __shfl_xor_sync(0xffffffffu, sa[h], off);
        sb[h] += __shfl_xor_sync(0xffffffffu, sb[h], off);
      }
    if (okA || okB) {
      float va[DPL], vb[DPL];
#pragma unroll
      for (int i = 0; i < NPC; ++i) {
        load_cvt<T, EP>(vA + (kl + i * LPP) * EP, va + i * EP);
        load_cvt<T, EP>(vB + (kl + i * LPP) * EP, vb + i * EP);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mn = m[h];
        if (okA) mn = fmaxf(mn, sa[h]);
        if (okB) mn = fmaxf(mn, sb[h]);
        const float alpha = exp2f(m[h] - mn);
        const float pa = okA ? exp2f(sa[h] - mn) : 0.f;
        const float pb2 = okB ? exp2f(sb[h] - mn) : 0.f;
        l[h] = fmaf(l[h], alpha, pa + pb2);
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(o[h][e], alpha, fmaf(pa, va[e], pb2 * vb[e]));
        m[h] = mn;
      }
    }
  };
  auto stamp = [&](int slot) {
    if (tl != nullptr && tid == 0) tl[slot] = globaltimer_ns();
  };
  int t0, t1;
  kv_tile_range(pos, p.Rt, seq_rank, seq_n, t0, t1);
  constexpr int kStep = kConsumerWarps * NGRP;  // positions per warp-wide pass
  RingPos rp(it, p.stages);
  for (int t = t0; t < t1; ++t, ++it, rp.next(p.stages)) {
    const int s = rp.slot;
    mbar_wait(&full[s], rp.phase, p.errflag);
    if (t == t0) stamp(kTlAttnFirst);
    const T* Kt = reinterpret_cast<const T*>(ring + (size_t)s * p.stage_bytes);
    const T* Vt = Kt + (size_t)p.Rt * D;
    const int lim = min(p.Rt, pos - t * p.Rt);  // cached positions < pos only
    for (int pb = warp * NGRP; pb < lim; pb += 2 * kStep) {
      const int pa = pb + grp, pbb = pb + kStep + grp;
      const bool okA = pa < lim, okB = pbb < lim;
      const int ra = okA ? pa : pb, rb = okB ? pbb : pb;
      consume2(Kt + (size_t)ra * D, Vt + (size_t)ra * D, okA, Kt + (size_t)rb * D,
               Vt + (size_t)rb * D, okB);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  // The new token (position pos) comes from shared memory, not the cache.
  if (fold_new && warp == 0 && pos >= 0) {
    float kf[DPL], vf[DPL];
#pragma unroll
    for (int i = 0; i < NPC; ++i)
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        kf[i * EP + e] = kn[(kl + i * LPP) * EP + e];
        vf[i * EP + e] = vn[(kl + i * LPP) * EP + e];
      }
    float sc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) s = fmaf(q[h][e], kf[e], s);
      sc[h] = s;
    }
#pragma unroll
    for (int off = LPP / 2; off >= 1; off >>= 1)
#pragma unroll
      for (int h = 0; h < G; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], off);
    if (grp == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mn = fmaxf(m[h], sc[h]);
        const float alpha = exp2f(m[h] - mn);
        const float pe = exp2f(sc[h] - mn);
        l[h] = fmaf(l[h], alpha, pe);
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(o[h][e], alpha, pe * vf[e]);
        m[h] = mn;
      }
    }
  }
  stamp(kTlAttnLoop);
  // Merge the lane groups of the warp.
#pragma unroll
  for (int off = LPP; off < 32; off <<= 1)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
      const float lo = __shfl_xor_sync(0xffffffffu, l[h], off);
      const float mn = fmaxf(m[h], mo);
      const float a = (mn == -INFINITY) ? 0.f : exp2f(m[h] - mn);
      const float bsc = (mn == -INFINITY) ? 0.f : exp2f(mo - mn);
      l[h] = l[h] * a + lo * bsc;
#pragma unroll
      for (int e = 0; e < DPL; ++e) {
        const float oo = __shfl_xor_sync(0xffffffffu, o[h][e], off);
        o[h][e] = o[h][e] * a + oo * bsc;
      }
      m[h] = mn;
    }
  if (grp == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float* st = wst + (warp * G + h) * (D + 4);
#pragma unroll
      for (int i = 0; i < NPC; ++i)
#pragma unroll
        for (int e = 0; e < EP; ++e) st[(kl + i * LPP) * EP + e] = o[h][i * EP + e];
      if (kl == 0) {
        st[D] = m[h];
        st[D + 1] = l[h];
      }
    }
  }
  named_sync(kBarConsumers, kConsumers);
  stamp(kTlAttnWarps);
  // Merge the 8 warps into this block's (o, m, l) record of the row.
  for (int idx = tid; idx < G * D; idx += kConsumers) {
    const int h = idx / D, dim = idx % D;
    float M = -INFINITY;
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wst[(w * G + h) * (D + 4) + D]);
    float O = 0.f, L = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float* st = wst + (w * G + h) * (D + 4);
        const float f = exp2f(st[D] - M);
        O = fmaf(f, st[dim], O);
        L = fmaf(f, st[D + 1], L);
      }
    }
    float* dst = rec + h * (D + 4);
    dst[dim] = O;
    if (dim == 0) {
      dst[D] = M;
      dst[D + 1] = L;
    }
  }
  named_sync(kBarConsumers, kConsumers);
}

}  // namespace cf
