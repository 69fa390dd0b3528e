// cf_attention_tc.cuh -- one batch row's attention over its whole KV sequence
// on the tensor cores, for the batched decode kernel ([CF §3.2] 在线softmax,
// page "ClusterFusion框架深度解析" (devpress.csdn.net); GQA grouping of
// "大模型推理中的算子融合优化：LayerNorm + Attention" (asdsk.com) §三).
//
// Positions are the M dimension of mma.sync m16n8k16 and the G query heads
// that share KV head g its N dimension (8 columns, G used):
//   S^T [positions x heads] = K [positions x d] . Q^T [d x heads]
//   O^T [d x heads]        += V^T [d x positions] . P^T [positions x heads]
// K and V^T come straight from the stage with ldmatrix (V^T through the
// transposing form); the probabilities P leave the S^T accumulators as packed
// 16-bit pairs and become the B operand of the second product through
// movmatrix.trans.  Q (fp32) and P (fp32, in [0, 1]) enter as 16-bit hi + lo
// pairs for bf16 storage, so both products keep about fp32 accuracy, and as
// single fp16 values for fp16 storage (MmaKind::kAttnHiLo); K and V are exact
// in their storage type.
//
// K/V tiles arrive as boxes of 64 columns (128 bytes) written with the
// 128-byte swizzle: stage = K [D/64][Rt][64] then V [D/64][Rt][64].  A warp
// takes 32 positions of a tile at a time; the Rt/32 chunks of a tile go to
// Rt/32 warps (at most 8), and when that is fewer than 8 the warps form groups
// that take alternate tiles, so several tiles are in work at once (every warp
// still waits for and releases every tile in order).  Each warp
// keeps its own running (m, l, o); the warps are merged through shared memory
// (for G > 1 in two halves of 4 warps) at the end into `rec` = [G][D+4]: unnormalized o,
// then m at D and l at D+1 (log2 units).
#pragma once

#include "cf_common.cuh"
#include "cf_mma.cuh"
#include "cf_params.h"
#include "cf_ptx.cuh"

namespace cf {

// Warp-state slots of the final merge (the `wst` scratch holds
// attn_tc_slots(G) * G * (D + 4) floats).
__host__ __device__ constexpr int attn_tc_slots(int G) { return G > 1 ? 4 : 8; }

// q_in: [G][D] fp32 post-RoPE queries; kn, vn: the new token's key and value
// [D] fp32 (folded in by warp 0 when `fold_new`); pos: the new token's
// position (cached keys 0..pos-1 come from the ring), < 0 for an invalid row;
// wst: [attn_tc_slots(G)][G][D+4] floats of scratch; qf: [D/16][32] uint4 of scratch for
// the Q fragments (shared by the 8 warps); `it` is the consumer's ring
// counter.  Called by the 256 consumer threads together; Rt is a power of two
// >= 32.
template <typename T, int D, int G>
__device__ void attend_row_tc(const KParams& p, const float* q_in, const float* kn,
                              const float* vn, int pos, bool fold_new, uint8_t* ring,
                              uint64_t* full, uint64_t* empty, int& it, float* wst, uint4* qf,
                              float* rec, unsigned long long* tl) {
  static_assert(G <= 8, "query heads per KV head must fit the 8 columns of the B operand");
  static_assert(D % 64 == 0, "head_dim in 64-column boxes");
  using MK = MmaKind<T>;
  constexpr int KS = D / 16;  // k steps of S^T = K Q^T
  constexpr int MD = D / 16;  // 16-row tiles of O^T
  constexpr int NB = D / 64;  // swizzled boxes per K (or V) tile
  constexpr int NA = MK::kAttnHiLo ? 2 : 4;  // S^T accumulators per 16-row tile (per product)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int h0 = 2 * tq;  // this lane's two head columns h0, h0 + 1

  // Q^T as B fragments (hi + lo), column gq = head gq: warp w builds k steps
  // w, w + 8, ...; lane l's part of step ks is qf[ks][l] = {hi b0, hi b1,
  // lo b0, lo b1}.
  for (int ks = warp; ks < KS; ks += kConsumerWarps) {
    float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
    if (gq < G) {
      const float* qr = q_in + gq * D + ks * 16 + 2 * tq;
      v0 = qr[0] * p.qk_scale_log2;
      v1 = qr[1] * p.qk_scale_log2;
      v2 = qr[8] * p.qk_scale_log2;
      v3 = qr[9] * p.qk_scale_log2;
    }
    uint4 f;
    MK::split2(v0, v1, f.x, f.z);
    MK::split2(v2, v3, f.y, f.w);
    qf[ks * 32 + lane] = f;
  }
  named_sync(kBarConsumers, kConsumers);

  // O^T accumulators: tile md, registers (dim md*16+gq, head h0), (.., h0+1),
  // (dim md*16+gq+8, h0), (.., h0+1).
  float o[MD][4];
#pragma unroll
  for (int md = 0; md < MD; ++md)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[md][e] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const bool hv0 = h0 < G, hv1 = h0 + 1 < G;

  auto stamp = [&](int slot) {
    if (tl != nullptr && tid == 0) tl[slot] = globaltimer_ns();
  };
  const int CH = p.Rt / 32;                                   // 32-position chunks per tile
  const int WPT = CH < kConsumerWarps ? CH : kConsumerWarps;  // warps per tile
  const int GROUPS = kConsumerWarps / WPT;                    // groups taking alternate tiles
  const int my_group = warp / WPT, my_slot = warp % WPT;
  const uint32_t box_bytes = (uint32_t)(p.Rt * 128);
  // ldmatrix row/chunk pattern shared by K (A of S^T) and V (A of O^T,
  // transposing form): lanes 0-7 rows 0-7 chunk 0, 8-15 rows 8-15 chunk 0,
  // 16-23 rows 0-7 chunk 1, 24-31 rows 8-15 chunk 1.
  const int lrow = (lane & 7) + (((lane >> 3) & 1) << 3);
  const int lch = lane >> 4;
  int t0, t1;
  kv_tile_range(pos, p.Rt, 0, 1, t0, t1);
  // ring slot of tile t and the group that owns it, advanced by counting
  RingPos rp(it, p.stages);
  int gsel = 0;
  auto next = [&]() {
    ++it;
    rp.next(p.stages);
    if (++gsel == GROUPS) gsel = 0;
  };
  for (int t = t0; t < t1; ++t, next()) {
    // Every warp waits for every tile, in ring order, and arrives once on its
    // release: a warp never waits on a stage whose earlier phase is still
    // pending (its parity would read as complete).  Only the owning group
    // computes on the tile.
    const int s = rp.slot;
    mbar_wait(&full[s], rp.phase, p.errflag);
    if (t == t0) stamp(kTlAttnFirst);
    if (gsel != my_group) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      continue;
    }
    uint8_t* st = ring + (size_t)s * p.stage_bytes;
    const uint32_t kbase = smem_u32(st);
    const uint32_t vbase = kbase + NB * box_bytes;
    const int lim = min(p.Rt, pos - t * p.Rt);  // valid positions of this tile
    bool wrote = false;
    for (int c = my_slot; c < CH; c += WPT) {
      const int cb = c * 32;
      if (cb >= lim) break;
      if (cb + 32 > lim) {
        // Positions past the row's end may hold anything (even NaN); zero
        // their V rows so that 0 * V stays 0 in the P V product.
        for (int r = lim + (lane >> 3); r < cb + 32; r += 4)
#pragma unroll
          for (int b = 0; b < NB; ++b)
            *reinterpret_cast<uint4*>(st + (NB + b) * box_bytes + r * 128 + (lane & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        wrote = true;
        __syncwarp();
      }
      // ---- S^T for positions cb..cb+31 (two 16-row tiles).  A dependent
      // mma.sync waits for the full latency of the one before it, so the k
      // steps rotate over NA accumulators per tile and the hi and lo products
      // go to separate ones: consecutive MMAs are independent.
      float sa[2][NA][4], sb[2][NA][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j = 0; j < NA; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) sa[mt][j][e] = sb[mt][j][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint4 f = qf[ks * 32 + lane];
        const int ch = ks * 2 + lch;
        uint32_t a[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
          ldsm_x4(a[mt][0], a[mt][1], a[mt][2], a[mt][3],
                  kbase + (ch >> 3) * box_bytes + sw128(cb + mt * 16 + lrow, ch & 7));
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          MK::mma(sa[mt][ks % NA], a[mt], f.x, f.y);
          if constexpr (MK::kAttnHiLo) MK::mma(sb[mt][ks % NA], a[mt], f.z, f.w);
        }
      }
      // ---- online softmax per head column (positions are spread over gq)
      float sc[2][4];
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pp = cb + mt * 16 + gq + ((e >> 1) << 3);
          float v = 0.f;
#pragma unroll
          for (int j = 0; j < NA; ++j) v += MK::kAttnHiLo ? sa[mt][j][e] + sb[mt][j][e] : sa[mt][j][e];
          sc[mt][e] = (pp < lim) ? v : -INFINITY;
        }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        mx0 = fmaxf(mx0, fmaxf(sc[mt][0], sc[mt][2]));
        mx1 = fmaxf(mx1, fmaxf(sc[mt][1], sc[mt][3]));
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      // finite: position cb is valid
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      const float al0 = exp2f(m[0] - mn0), al1 = exp2f(m[1] - mn1);
      m[0] = mn0;
      m[1] = mn1;
      float pr[2][4];
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        pr[mt][0] = hv0 ? exp2f(sc[mt][0] - mn0) : 0.f;
        pr[mt][2] = hv0 ? exp2f(sc[mt][2] - mn0) : 0.f;
        pr[mt][1] = hv1 ? exp2f(sc[mt][1] - mn1) : 0.f;
        pr[mt][3] = hv1 ? exp2f(sc[mt][3] - mn1) : 0.f;
        ps0 += pr[mt][0] + pr[mt][2];
        ps1 += pr[mt][1] + pr[mt][3];
      }
      l[0] = fmaf(l[0], al0, ps0);
      l[1] = fmaf(l[1], al1, ps1);
      // ---- P^T as B fragments: (positions 2tq.., head gq) per 8-position
      // half, from the S^T layout (position gq, heads 2tq..) by transposing
      uint32_t bh[2][2], bl[2][2];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        uint32_t h01, l01, h23, l23;
        MK::split2(pr[mt][0], pr[mt][1], h01, l01);
        MK::split2(pr[mt][2], pr[mt][3], h23, l23);
        bh[mt][0] = movmatrix_trans(h01);
        bh[mt][1] = movmatrix_trans(h23);
        if constexpr (MK::kAttnHiLo) {
          bl[mt][0] = movmatrix_trans(l01);
          bl[mt][1] = movmatrix_trans(l23);
        }
      }
      // ---- O^T += V^T P^T: k = 32 positions in two steps, into fresh
      // accumulators, the dimension tiles interleaved so that consecutive
      // MMAs are independent (the lo products in a second pass over V^T);
      // the running O^T is rescaled and the chunk added once
      float pa[MD][4];
#pragma unroll
      for (int md = 0; md < MD; ++md)
#pragma unroll
        for (int e = 0; e < 4; ++e) pa[md][e] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hl = 0; hl < (MK::kAttnHiLo ? 2 : 1); ++hl)
#pragma unroll
          for (int md = 0; md < MD; ++md) {
            const int ch = md * 2 + lch;
            uint32_t a[4];
            ldsm_x4_trans(a[0], a[2], a[1], a[3],
                          vbase + (ch >> 3) * box_bytes + sw128(cb + mt * 16 + lrow, ch & 7));
            if (hl == 0) MK::mma(pa[md], a, bh[mt][0], bh[mt][1]);
            else MK::mma(pa[md], a, bl[mt][0], bl[mt][1]);
          }
#pragma unroll
      for (int md = 0; md < MD; ++md) {
        o[md][0] = fmaf(o[md][0], al0, pa[md][0]);
        o[md][1] = fmaf(o[md][1], al1, pa[md][1]);
        o[md][2] = fmaf(o[md][2], al0, pa[md][2]);
        o[md][3] = fmaf(o[md][3], al1, pa[md][3]);
      }
    }
    // Generic-proxy writes into the stage must be ordered before the TMA
    // write that refills it.
    if (wrote) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  // The new token (position pos) comes from shared memory, not the cache.
  if (fold_new && warp == 0 && pos >= 0) {
    float sn0 = 0.f, sn1 = 0.f;
    if (hv0)
      for (int d = 0; d < D; ++d) sn0 = fmaf(q_in[h0 * D + d] * p.qk_scale_log2, kn[d], sn0);
    if (hv1)
      for (int d = 0; d < D; ++d) sn1 = fmaf(q_in[(h0 + 1) * D + d] * p.qk_scale_log2, kn[d], sn1);
    const float mn0 = hv0 ? fmaxf(m[0], sn0) : m[0], mn1 = hv1 ? fmaxf(m[1], sn1) : m[1];
    const float al0 = hv0 ? exp2f(m[0] - mn0) : 1.f, al1 = hv1 ? exp2f(m[1] - mn1) : 1.f;
    const float pe0 = hv0 ? exp2f(sn0 - mn0) : 0.f, pe1 = hv1 ? exp2f(sn1 - mn1) : 0.f;
    // the lanes' partial sums are summed over gq later: count the new token
    // once (gq == 0)
    l[0] = fmaf(l[0], al0, gq == 0 ? pe0 : 0.f);
    l[1] = fmaf(l[1], al1, gq == 0 ? pe1 : 0.f);
    m[0] = mn0;
    m[1] = mn1;
#pragma unroll
    for (int md = 0; md < MD; ++md) {
      const float va = vn[md * 16 + gq], vb = vn[md * 16 + gq + 8];
      o[md][0] = fmaf(o[md][0], al0, pe0 * va);
      o[md][1] = fmaf(o[md][1], al1, pe1 * va);
      o[md][2] = fmaf(o[md][2], al0, pe0 * vb);
      o[md][3] = fmaf(o[md][3], al1, pe1 * vb);
    }
  }
  stamp(kTlAttnLoop);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
    l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
  }
  // Merge the 8 warps' states into the row's (o, m, l) record through
  // attn_tc_slots<G>() warp slots of shared memory: for G > 1 in two halves
  // (warps 0-3, then 4-7), for one head (small states) in one pass.
  constexpr int HS = attn_tc_slots(G);                            // slots
  constexpr int NH = kConsumerWarps / HS;                         // passes
  constexpr int PER = (G * D + kConsumers - 1) / kConsumers;      // elements per thread
  float PM[PER], PO[PER], PL[PER];
#pragma unroll
  for (int half = 0; half < NH; ++half) {
    if (warp / HS == half) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (h0 + j >= G) continue;
        float* stw = wst + ((warp % HS) * G + h0 + j) * (D + 4);
#pragma unroll
        for (int md = 0; md < MD; ++md) {
          stw[md * 16 + gq] = o[md][j];
          stw[md * 16 + gq + 8] = o[md][2 + j];
        }
        if (gq == 0) {
          stw[D] = m[j];
          stw[D + 1] = l[j];
        }
      }
    }
    named_sync(kBarConsumers, kConsumers);
    if (half == 0) stamp(kTlAttnWarps);
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int idx = tid + u * kConsumers;
      if (idx >= G * D) continue;
      const int h = idx / D, dim = idx % D;
      float M = half ? PM[u] : -INFINITY;
      for (int w = 0; w < HS; ++w) M = fmaxf(M, wst[(w * G + h) * (D + 4) + D]);
      float O = 0.f, L = 0.f;
      if (M != -INFINITY) {
        if (half && PM[u] != -INFINITY) {
          const float f = exp2f(PM[u] - M);
          O = PO[u] * f;
          L = PL[u] * f;
        }
        for (int w = 0; w < HS; ++w) {
          const float* sw = wst + (w * G + h) * (D + 4);
          const float f = exp2f(sw[D] - M);
          O = fmaf(f, sw[dim], O);
          L = fmaf(f, sw[D + 1], L);
        }
      }
      PM[u] = M;
      PO[u] = O;
      PL[u] = L;
    }
    named_sync(kBarConsumers, kConsumers);
  }
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int idx = tid + u * kConsumers;
    if (idx >= G * D) continue;
    const int h = idx / D, dim = idx % D;
    float* dst = rec + h * (D + 4);
    dst[dim] = PO[u];
    if (dim == 0) {
      dst[D] = PM[u];
      dst[D + 1] = PL[u];
    }
  }
  named_sync(kBarConsumers, kConsumers);
}

}  // namespace cf
