// cf_kernel.cuh -- the fused single-token decode attention block for sm_103a.
//
// Pages cited by title and section:
//   [CF]  "ClusterFusion框架深度解析：LLM推理优化的集群级通信革命" (devpress.csdn.net)
//   [LNA] "大模型推理中的算子融合优化：LayerNorm + Attention 的 CUDA Kernel 手写与验证"
//         (asdsk.com)
//
// One launch computes, for every batch row, RMSNorm -> merged QKV projection
// -> RoPE -> KV-cache append -> split-KV online-softmax attention -> output
// projection + residual ([CF §3.2] fused_qkv_attention_out, [LNA §一]).
//
// Mapping [CF §3.2 空间映射策略]: one thread-block cluster per (KV head g,
// batch tile of BT rows); for GQA the cluster serves the G = nq/nkv query
// heads of its KV head, so each K/V byte is read once.  The N blocks of a
// cluster split
//   * the hidden (reduction) dimension of the QKV projection: block c owns
//     rows [c*H/N, (c+1)*H/N) of W_qkv's head columns; the partial q/k/v are
//     combined by ClusterReduce (reduce-scatter form), which leaves block c
//     owning head-dim slice c (the RoPE pairs (i, i+d/2) with i in
//     [c*P, (c+1)*P), P = d/(2N)); block c rotates and appends its slice, and
//     ClusterGather then gives every block the full q', k', v [CF §3.1.2,
//     "QKV向量共享"];
//   * the KV sequence of the attention: block c takes its share of the
//     position tiles and produces online-softmax partials (m, l, o); these
//     are combined with ClusterReduce(max) and a rescaled ClusterReduce(sum)
//     [CF §3.2 在线softmax, §3.1.1];
//   * the output columns of the O projection: block c multiplies o by its
//     column band of W_o and adds into an fp32 accumulator with atomics
//     [CF §3.2 原子写合并]; the last block to finish a (batch tile, band)
//     adds the residual, rounds to the storage type and writes `out`.
//
// Data movement: one producer warp streams every byte the block needs
// (W_qkv tiles, then K/V tiles, then W_o tiles) through a ring of
// shared-memory stages with TMA tensor copies (evict-first in L2), running
// ahead of the 8 consumer warps across phase boundaries, so HBM stays busy
// while the consumers are in a cluster exchange ([CF §4.2] "通信-计算重叠",
// done with TMA instead of cuda::memcpy_async).  Intermediates never touch
// HBM: normed hidden, q/k/v, softmax statistics and partial outputs live in
// shared memory and move between blocks over DSMEM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cf_attention.cuh"
#include "cf_cluster.cuh"
#include "cf_common.cuh"
#include "cf_params.h"
#include "cf_ptx.cuh"

namespace cf {


// MINB: blocks per SM the register allocation must allow (2 for the
// small-state instances, so two 288-thread blocks fit in 64K registers).
template <typename T, int D, int G, int BT, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) cf_decode_kernel(const __grid_constant__ KParams p) {
  constexpr int NSEG = G + 2;          // q heads of the group, k, v
  constexpr int CPL = D / 32;          // projection columns per lane per segment
  static_assert(D == 64 || D == 128, "head_dim");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int N = p.N;
  const int rank = (int)cluster_ctarank();
  const int cid = blockIdx.x / N;
  const int g = cid / p.nbt;  // KV head
  const int bt = cid % p.nbt; // batch tile
  const int b0 = bt * BT;
  const int P = D / (2 * N);            // RoPE pairs per head-dim slice
  // P is a power of two: index splits by shift and mask (a division by a
  // runtime divisor is a long dependent chain on the exchange path)
  const int lP = 31 - __clz(P);
  const int SE = BT * NSEG * 2 * P;     // floats per slice
  const int Hc = p.H / N;               // K band rows == O-proj column band
  const int k0 = rank * Hc;
  const int nrounds = __ffs(N) - 1;
  const int SMP = BT * G * (D + 4);

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + p.L.bars);
  uint64_t* full = bars + BarIdx::full;
  uint64_t* empty = bars + BarIdx::empty;
  uint8_t* ring = sm + p.L.ring;
  float* xn = reinterpret_cast<float*>(sm + p.L.xn);
  float* red = reinterpret_cast<float*>(sm + p.L.red);
  float* scratch = reinterpret_cast<float*>(sm + p.L.scratch);
  float* qkv = reinterpret_cast<float*>(sm + p.L.qkv);
  float* smx = reinterpret_cast<float*>(sm + p.L.sm);
  float* mscale = reinterpret_cast<float*>(sm + p.L.scale);
  float* rope = reinterpret_cast<float*>(sm + p.L.rope);
  int* s_pos = reinterpret_cast<int*>(sm + p.L.misc);
  int* s_flag = s_pos + BT;
  float* s_rinv = reinterpret_cast<float*>(s_flag + 4);

  // ---------------------------------------------------------------- setup --
  // Programmatic dependent launch: let the next kernel in the stream start
  // its own set-up as our blocks retire; it waits (griddepcontrol.wait
  // below) for this grid to finish before it reads global memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int r = 0; r < nrounds; ++r) {
      mbar_init(&bars[BarIdx::rs + r], 1);
      mbar_init(&bars[BarIdx::ga + r], 1);
      mbar_init(&bars[BarIdx::sm + r], 1);
    }
    fence_mbar_init_cluster();
    for (int r = 0; r < nrounds; ++r) {
      mbar_arrive_expect_tx(&bars[BarIdx::rs + r], reduce_scatter_round_bytes(N, r, SE));
      mbar_arrive_expect_tx(&bars[BarIdx::ga + r], gather_round_bytes(r, SE));
      mbar_arrive_expect_tx(&bars[BarIdx::sm + r], allreduce_round_bytes(SMP));
    }
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tensormap(&p.tm_wqkv);
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
    prefetch_tensormap(&p.tm_wo);
  }
  __syncthreads();
  cluster_sync_all();  // peers' barriers are initialized before any DSMEM traffic
  // Prologue fill: the weights are read-only, so the first ring-full of
  // W_qkv tiles is requested before waiting for the preceding kernel (with
  // programmatic dependent launch this overlaps its tail).  These stages are
  // fresh, so no empty-barrier wait is needed; the producer loop below
  // continues after them.
  const int nkt_all = (p.H / N) / p.Rw;
  const int fill = min(p.stages, nkt_all);
  const uint32_t seg_bytes = (uint32_t)(p.Rw * D * sizeof(T));
  if (warp == kConsumerWarps && lane == 0) {
    const uint64_t pol = policy_evict_first();
    for (int kt = 0; kt < fill; ++kt) {
      uint64_t* bar = &full[kt];
      uint8_t* dst = ring + (size_t)kt * p.stage_bytes;
      mbar_arrive_expect_tx(bar, NSEG * seg_bytes);
      const int y = k0 + kt * p.Rw;
      for (int j = 0; j < G; ++j)
        tma_load_2d(dst + j * seg_bytes, &p.tm_wqkv, (g * G + j) * D, y, bar, pol);
      tma_load_2d(dst + G * seg_bytes, &p.tm_wqkv, (p.nq + g) * D, y, bar, pol);
      tma_load_2d(dst + (G + 1) * seg_bytes, &p.tm_wqkv, (p.nq + p.nkv + g) * D, y, bar, pol);
    }
  }
  // From here on global memory may hold a preceding kernel's results (the
  // previous layer's out, the K/V slot the previous step appended).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid < BT) {
    const int b = b0 + tid;
    int pos = -1;
    if (b < p.B) {
      pos = p.positions[b];
      if (pos < 0 || pos >= p.S) {
        if (rank == 0 && g == 0) atomicOr(p.errflag, kDevErrPosRange);
        pos = -1;
      }
    }
    s_pos[tid] = pos;
  }
  __syncthreads();
  // Optional phase timeline (tuning aid): thread 0 stamps consumer phases,
  // the producer lane its own milestones.
  auto stamp = [&](int slot) {
    if (p.timeline != nullptr && tid == 0)
      p.timeline[blockIdx.x * kTimelineSlots + slot] = globaltimer_ns();
  };
  auto stamp_last_warp = [&](int slot) {  // latest over the consumer warps
    if (p.timeline != nullptr && lane == 0)
      atomicMax(&p.timeline[blockIdx.x * kTimelineSlots + slot], globaltimer_ns());
  };
  stamp(kTlStart);
  if (p.timeline != nullptr && tid == 0)
    p.timeline[blockIdx.x * kTimelineSlots + kTlSmid] = sm_id();

  const int nkt = Hc / p.Rw;
  const int ncb = Hc / p.Co;
  const int nrt = G * D / p.Ro;

  if (warp == kConsumerWarps) {
    // ============================================== TMA producer warp ====
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      RingPos rp(fill, p.stages);  // the prologue filled uses 0 .. fill-1
      auto slot = [&](uint32_t bytes, uint64_t*& bar) -> uint8_t* {
        const int s = rp.slot;
        if (it >= p.stages) mbar_wait(&empty[s], rp.phase ^ 1u, p.errflag);
        rp.next(p.stages);
        bar = &full[s];
        mbar_arrive_expect_tx(bar, bytes);
        return ring + (size_t)s * p.stage_bytes;
      };
      // Phase 1: W_qkv row tiles of this block's K band, G+2 head slices each
      // (the first `fill` were requested before the dependency wait).
      for (int kt = 0; kt < nkt; ++kt, ++it) {
        if (kt < fill) continue;
        uint64_t* bar;
        uint8_t* dst = slot(NSEG * seg_bytes, bar);
        const int y = k0 + kt * p.Rw;
        for (int j = 0; j < G; ++j)
          tma_load_2d(dst + j * seg_bytes, &p.tm_wqkv, (g * G + j) * D, y, bar, pol);
        tma_load_2d(dst + G * seg_bytes, &p.tm_wqkv, (p.nq + g) * D, y, bar, pol);
        tma_load_2d(dst + (G + 1) * seg_bytes, &p.tm_wqkv, (p.nq + p.nkv + g) * D, y, bar, pol);
      }
      if (p.timeline) p.timeline[blockIdx.x * kTimelineSlots + kTlProdW] = globaltimer_ns();
      // Phase 2: K and V tiles of this block's share of each row's positions.
      const uint32_t kv_bytes = (uint32_t)(p.Rt * D * sizeof(T));
      for (int bb = 0; bb < BT; ++bb) {
        int t0, t1;
        kv_tile_range(s_pos[bb], p.Rt, rank, N, t0, t1);
        for (int t = t0; t < t1; ++t, ++it) {
          uint64_t* bar;
          uint8_t* dst = slot(2 * kv_bytes, bar);
          tma_load_4d(dst, &p.tm_k, 0, g, t * p.Rt, b0 + bb, bar, pol);
          tma_load_4d(dst + kv_bytes, &p.tm_v, 0, g, t * p.Rt, b0 + bb, bar, pol);
        }
      }
      if (p.timeline) p.timeline[blockIdx.x * kTimelineSlots + kTlProdKV] = globaltimer_ns();
      // Phase 3: W_o tiles: rows of the group's heads x this block's column band.
      const uint32_t wo_bytes = (uint32_t)(p.Ro * p.Co * sizeof(T));
      for (int cb = 0; cb < ncb; ++cb)
        for (int rt = 0; rt < nrt; ++rt, ++it) {
          uint64_t* bar;
          uint8_t* dst = slot(wo_bytes, bar);
          tma_load_2d(dst, &p.tm_wo, k0 + cb * p.Co, g * G * D + rt * p.Ro, bar, pol);
        }
      if (p.timeline) p.timeline[blockIdx.x * kTimelineSlots + kTlProdAll] = globaltimer_ns();
    }
    __syncwarp();
  } else {
    // ============================================== consumer warps =======
    const T* __restrict__ hidden = reinterpret_cast<const T*>(p.hidden);
    const T* __restrict__ lnw = reinterpret_cast<const T*>(p.ln_w);
    int it = 0;

    // ---- Phase 0: x * ln_weight over the own K band [LNA §三 stage 1] ----
    // RMSNorm is n = x * g * r with one scalar r = 1/sqrt(mean(x^2) + eps)
    // per row; r commutes with the projection, so it is applied to the
    // partial sums after the W_qkv loop and the full-row reduction stays off
    // the path to the first weight tile.
    for (int i = tid; i < N * SE; i += kConsumers) red[i] = 0.f;
    for (int i = tid; i < SMP; i += kConsumers) smx[i] = 0.f;
    // One pass over each row: the sum of squares of the whole row (for r)
    // and x*g for the 16-byte chunks inside the own K band.
    float* wred = s_rinv + BT;  // [8 warps][BT] partial sums of squares
    {
      constexpr int EV = 16 / (int)sizeof(T);
#pragma unroll
      for (int bb = 0; bb < BT; ++bb) {
        float ss = 0.f;
        if (b0 + bb < p.B) {
          const T* x = hidden + (size_t)(b0 + bb) * p.H;
          for (int i = tid * EV; i < p.H; i += kConsumers * EV) {
            float f[EV];
            load_cvt<T, EV>(x + i, f);
#pragma unroll
            for (int e = 0; e < EV; ++e) ss = fmaf(f[e], f[e], ss);
            if (i >= k0 && i < k0 + Hc) {
              float gw[EV];
              load_cvt<T, EV>(lnw + i, gw);
#pragma unroll
              for (int e = 0; e < EV; ++e) xn[bb * Hc + (i - k0) + e] = f[e] * gw[e];
            }
          }
        } else {
          for (int i = tid; i < Hc; i += kConsumers) xn[bb * Hc + i] = 0.f;
        }
        ss = warp_sum(ss);
        if (lane == 0) wred[warp * BT + bb] = ss;
      }
      // cos/sin of this block's own RoPE pairs
      for (int idx = tid; idx < BT * P; idx += kConsumers) {
        const int bb = idx >> lP, j = idx & (P - 1);
        const int pos = s_pos[bb];
        float c = 1.f, sn = 0.f;
        if (pos >= 0) rope_cos_sin(pos, p.turn_hi[rank * P + j], p.turn_lo[rank * P + j], c, sn);
        rope[2 * idx] = c;
        rope[2 * idx + 1] = sn;
      }
    }
    named_sync(kBarConsumers, kConsumers);
    stamp(kTlNorm);
    // ---- Phase 1: merged QKV projection over this block's K band --------
    {
      float acc[BT][NSEG][CPL];
#pragma unroll
      for (int bb = 0; bb < BT; ++bb)
#pragma unroll
        for (int sg = 0; sg < NSEG; ++sg)
#pragma unroll
          for (int e = 0; e < CPL; ++e) acc[bb][sg][e] = 0.f;
      RingPos rp(it, p.stages);
      for (int kt = 0; kt < nkt; ++kt, ++it, rp.next(p.stages)) {
        const int s = rp.slot;
        mbar_wait(&full[s], rp.phase, p.errflag);
        const T* tile = reinterpret_cast<const T*>(ring + (size_t)s * p.stage_bytes);
        for (int r = warp; r < p.Rw; r += kConsumerWarps) {
          float nv[BT];
#pragma unroll
          for (int bb = 0; bb < BT; ++bb) nv[bb] = xn[bb * Hc + kt * p.Rw + r];
#pragma unroll
          for (int sg = 0; sg < NSEG; ++sg) {
            float w[CPL];
            load_cvt<T, CPL>(tile + ((size_t)sg * p.Rw + r) * D + lane * CPL, w);
#pragma unroll
            for (int bb = 0; bb < BT; ++bb)
#pragma unroll
              for (int e = 0; e < CPL; ++e) acc[bb][sg][e] = fmaf(nv[bb], w[e], acc[bb][sg][e]);
          }
        }
        __syncwarp();
        // The last tile's stage is kept from the producer: it becomes the
        // buffer of the cross-warp reduction below and is released after it.
        if (lane == 0 && kt < nkt - 1) mbar_arrive(&empty[s]);
      }
      stamp(kTlProjLoop);
      stamp_last_warp(kTlProjLoopLast);
      // RMSNorm scale r = 1/sqrt(mean(x^2) + eps) of each row from the warp
      // partials of phase 0 (warp shuffles, then one cross-warp step [LNA §五]).
      if (tid < BT) {
        float tot = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) tot += wred[w * BT + tid];
        s_rinv[tid] = (b0 + tid < p.B) ? 1.0f / sqrtf(tot / (float)p.H + p.eps) : 0.f;
      }
      // Sum of the 8 warps' partials through the held stage, [warp][value]
      // [lane] so every access is conflict-free; no atomics, and the
      // summation order is fixed.  When all 8 warps' partials fit the stage
      // they are written at once and every thread sums the 8 copies of its
      // values (one barrier); otherwise a tree (8 -> 4 -> 2 -> 1).
      {
        const int s_last = (it - 1) % p.stages;
        float* tb = reinterpret_cast<float*>(ring + (size_t)s_last * p.stage_bytes);
        constexpr int PW = BT * NSEG * CPL;
        constexpr int NV = PW * 32;  // values per warp
        named_sync(kBarConsumers, kConsumers);  // every warp is done reading the tile
        if (kConsumerWarps * NV * 4 <= p.stage_bytes) {
          float* dst = tb + warp * NV + lane;
#pragma unroll
          for (int bb = 0; bb < BT; ++bb)
#pragma unroll
            for (int sg = 0; sg < NSEG; ++sg)
#pragma unroll
              for (int e = 0; e < CPL; ++e) dst[((bb * NSEG + sg) * CPL + e) * 32] = acc[bb][sg][e];
          named_sync(kBarConsumers, kConsumers);
          // value o = ((bb * NSEG + sg) * CPL + e) * 32 + lane: column lane * CPL + e of
          // segment sg of row bb, stored scaled by r and slice-ordered as below
          for (int o = tid; o < NV; o += kConsumers) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) sum += tb[w * NV + o];
            const int v = o >> 5, e = v % CPL, bs = v / CPL, sg = bs % NSEG, bb = bs / NSEG;
            const int col = (o & 31) * CPL + e;
            const int hi = col / (D / 2), il = col % (D / 2);
            const int c = il >> lP, j = il & (P - 1);
            red[c * SE + ((bb * NSEG + sg) * 2 + hi) * P + j] = sum * s_rinv[bb];
          }
          fence_proxy_async_smem();  // our reads of the stage precede the next TMA write
          named_sync(kBarConsumers, kConsumers);
          if (lane == 0) mbar_arrive(&empty[s_last]);  // hand the stage back
        } else {
          const bool disjoint = 7 * PW * 32 * 4 <= p.stage_bytes;  // one region per step
          int base = 0;
          for (int half = kConsumerWarps / 2; half >= 1; half >>= 1) {
            if (warp >= half && warp < 2 * half) {
              float* dst = tb + (base + warp - half) * PW * 32 + lane;
#pragma unroll
              for (int bb = 0; bb < BT; ++bb)
#pragma unroll
                for (int sg = 0; sg < NSEG; ++sg)
#pragma unroll
                  for (int e = 0; e < CPL; ++e)
                    dst[((bb * NSEG + sg) * CPL + e) * 32] = acc[bb][sg][e];
            }
            named_sync(kBarConsumers, kConsumers);
            if (warp < half) {
              const float* src = tb + (base + warp) * PW * 32 + lane;
#pragma unroll
              for (int bb = 0; bb < BT; ++bb)
#pragma unroll
                for (int sg = 0; sg < NSEG; ++sg)
#pragma unroll
                  for (int e = 0; e < CPL; ++e)
                    acc[bb][sg][e] += src[((bb * NSEG + sg) * CPL + e) * 32];
            }
            if (disjoint) base += half;
            else named_sync(kBarConsumers, kConsumers);
          }
          // Warp 0 holds the block's partial sums: scale by r and store them
          // slice-ordered -- column i of a segment belongs to slice
          // c = (i mod d/2) / P, so each RoPE pair (i, i + d/2) stays in one slice.
          if (warp == 0) {
#pragma unroll
            for (int sg = 0; sg < NSEG; ++sg)
#pragma unroll
              for (int e = 0; e < CPL; ++e) {
                const int col = lane * CPL + e;
                const int hi = col / (D / 2), il = col % (D / 2);
                const int c = il >> lP, j = il & (P - 1);
#pragma unroll
                for (int bb = 0; bb < BT; ++bb)
                  red[c * SE + ((bb * NSEG + sg) * 2 + hi) * P + j] = acc[bb][sg][e] * s_rinv[bb];
              }
          }
          fence_proxy_async_smem();  // our stores into the stage precede the next TMA write
          named_sync(kBarConsumers, kConsumers);
          if (lane == 0) mbar_arrive(&empty[s_last]);  // hand the stage back
        }
      }
      stamp(kTlRinv);
    }

    stamp(kTlProj);
    // ---- ClusterReduce (reduce-scatter): block `rank` owns slice `rank` --
    cluster_reduce_scatter<kConsumers, kBarConsumers>(red, SE, scratch, &bars[BarIdx::rs], rank,
                                                      N, tid, p.errflag);

    stamp(kTlReduceScatter);
    // ---- RoPE on the own slice, then append K/V [LNA §三 stage 3] -------
    {
      float* my = red + rank * SE;
      T* kc = reinterpret_cast<T*>(p.k_cache);
      T* vc = reinterpret_cast<T*>(p.v_cache);
      for (int idx = tid; idx < BT * NSEG * P; idx += kConsumers) {
        const int q = idx >> lP, j = idx & (P - 1);
        const int bb = q / NSEG, sg = q % NSEG;
        const int pos = s_pos[bb];
        if (pos < 0) continue;
        float* lo = my + ((bb * NSEG + sg) * 2) * P + j;
        float* hi = lo + P;
        float a = *lo, bv = *hi;
        if (sg <= G) {  // query heads and the key: rotate-half
          const float c = rope[2 * (bb * P + j)], sn = rope[2 * (bb * P + j) + 1];
          const float ra = a * c - bv * sn;
          const float rb = bv * c + a * sn;
          a = ra;
          bv = rb;
        }
        if (sg >= G) {  // key and value: append (rounded to storage); the
                        // attention below keeps using the fp32 on-chip values
          const T ta = Elem<T>::from_f(a), tb = Elem<T>::from_f(bv);
          T* cache = (sg == G) ? kc : vc;
          const size_t base = (((size_t)(b0 + bb) * p.S + pos) * p.nkv + g) * D;
          cache[base + rank * P + j] = ta;
          cache[base + D / 2 + rank * P + j] = tb;
        }
        *lo = a;
        *hi = bv;
      }
      named_sync(kBarConsumers, kConsumers);
    }

    // ---- ClusterGather of the q'/k'/v slices [CF §3.1.2] -----------------
    cluster_gather<kConsumers, kBarConsumers>(red, SE, &bars[BarIdx::ga], rank, N, tid, p.errflag);
    for (int idx = tid; idx < BT * NSEG * D; idx += kConsumers) {
      const int bb = idx / (NSEG * D), rem = idx % (NSEG * D);
      const int sg = rem / D, dim = rem % D;
      const int hi = dim / (D / 2), il = dim % (D / 2);
      const int c = il >> lP, j = il & (P - 1);
      qkv[idx] = red[c * SE + ((bb * NSEG + sg) * 2 + hi) * P + j];
    }
    named_sync(kBarConsumers, kConsumers);
    if (p.dbg != nullptr && rank == 0) {
      float* dq = p.dbg;
      float* dk = dq + (size_t)p.B * p.nq * D;
      float* dv = dk + (size_t)p.B * p.nkv * D;
      for (int idx = tid; idx < BT * NSEG * D; idx += kConsumers) {
        const int bb = idx / (NSEG * D), rem = idx % (NSEG * D);
        const int sg = rem / D, dim = rem % D;
        const int b = b0 + bb;
        if (b >= p.B || s_pos[bb] < 0) continue;
        if (sg < G) dq[((size_t)b * p.nq + g * G + sg) * D + dim] = qkv[idx];
        else if (sg == G) dk[((size_t)b * p.nkv + g) * D + dim] = qkv[idx];
        else dv[((size_t)b * p.nkv + g) * D + dim] = qkv[idx];
      }
    }

    stamp(kTlGather);
    // ---- Phase 2: split-KV online-softmax attention [CF §3.2] ------------
    // Block `rank` takes its share of each row's position tiles; the last
    // block of the cluster also folds in the new token.
    for (int bb = 0; bb < BT; ++bb) {
      const float* qb = qkv + bb * NSEG * D;
      attend_row<T, D, G>(p, qb, qb + G * D, qb + (G + 1) * D, s_pos[bb], rank, N, rank == N - 1,
                          ring, full, empty, it, scratch, smx + bb * G * (D + 4),
                          (p.timeline != nullptr && bb == 0)
                              ? p.timeline + blockIdx.x * kTimelineSlots
                              : nullptr);
    }

    stamp(kTlAttn);
    // ---- ClusterReduce of the softmax partials [CF §3.1.1, §3.2]: max of
    // the statistics and the rescaled sum of (o, l) in one butterfly ---------
    cluster_allreduce_softmax<kConsumers, kBarConsumers>(smx, BT * G, D, smx + SMP,
                                                         &bars[BarIdx::sm], mscale, rank, N, tid,
                                                         p.errflag);
    stamp(kTlMax);
    // Final attention output o = (sum o_c e^{m_c-m}) / (sum l_c e^{m_c-m}),
    // written over the (no longer needed) q' of the same head.
    for (int idx = tid; idx < BT * G * D; idx += kConsumers) {
      const int bb = idx / (G * D), rem = idx % (G * D);
      const int h = rem / D, dim = rem % D;
      const float* src = smx + (bb * G + h) * (D + 4);
      const float L = src[D + 1];
      qkv[(bb * NSEG + h) * D + dim] = (L > 0.f) ? src[dim] / L : 0.f;
    }
    named_sync(kBarConsumers, kConsumers);
    if (p.dbg != nullptr && rank == 0) {
      float* dob = p.dbg + (size_t)p.B * (p.nq + 2 * p.nkv) * D;
      for (int idx = tid; idx < BT * G * D; idx += kConsumers) {
        const int bb = idx / (G * D), rem = idx % (G * D);
        const int h = rem / D, dim = rem % D;
        const int b = b0 + bb;
        if (b >= p.B || s_pos[bb] < 0) continue;
        dob[((size_t)b * p.nq + g * G + h) * D + dim] = qkv[(bb * NSEG + h) * D + dim];
      }
    }

    stamp(kTlSum);
    // ---- Phase 3: O projection of this block's column band [CF §3.2] -----
    {
      // Each thread owns one 16-byte column chunk (CW columns) of a tile row
      // and every RG-th row; a warp reads whole rows with 16-byte loads.
      constexpr int CW = 16 / (int)sizeof(T);
      const int CC = p.Co / CW;  // chunks per tile row
      const int RG = kConsumers / CC;
      const int cc = tid % CC, rg = tid / CC;
      const int CQ = p.Co / 4;
      RingPos rp(it, p.stages);
      for (int cb = 0; cb < ncb; ++cb) {
        float a[BT][CW];
#pragma unroll
        for (int bb = 0; bb < BT; ++bb)
#pragma unroll
          for (int e = 0; e < CW; ++e) a[bb][e] = 0.f;
        int s_last = 0;  // the box's last tile stage
        for (int rt = 0; rt < nrt; ++rt, ++it, rp.next(p.stages)) {
          const int s = rp.slot;
          s_last = s;
          mbar_wait(&full[s], rp.phase, p.errflag);
          if (cb == 0 && rt == 0) stamp(kTlOprojFirst);
          else if (cb * nrt + rt < 4) stamp(kTlOprojTile1 - 1 + cb * nrt + rt);
          const T* W = reinterpret_cast<const T*>(ring + (size_t)s * p.stage_bytes);
          if (rg < RG) {
            for (int r = rg; r < p.Ro; r += RG) {
              float w[CW];
              load_cvt<T, CW>(W + (size_t)r * p.Co + cc * CW, w);
              const int row = rt * p.Ro + r;
              const int h = row / D, dim = row % D;
#pragma unroll
              for (int bb = 0; bb < BT; ++bb) {
                const float ov = qkv[(bb * NSEG + h) * D + dim];
#pragma unroll
                for (int e = 0; e < CW; ++e) a[bb][e] = fmaf(ov, w[e], a[bb][e]);
              }
            }
          }
          __syncwarp();
          // the box's last tile stage is held for the row-group reduction
          if (lane == 0 && rt < nrt - 1) mbar_arrive(&empty[s]);
        }
        if (cb == ncb - 1) stamp(kTlOprojLoop);
        // Row-group partials [RG][BT][Co] into the held stage, then each
        // float4 of the box summed over the groups in a fixed order and added
        // to the accumulator with one vector atomic.
        float* pb = reinterpret_cast<float*>(ring + (size_t)s_last * p.stage_bytes);
        named_sync(kBarConsumers, kConsumers);  // every warp is done reading the tile
        if (rg < RG)
#pragma unroll
          for (int bb = 0; bb < BT; ++bb)
#pragma unroll
            for (int e4 = 0; e4 < CW; e4 += 4)
              *reinterpret_cast<float4*>(pb + ((size_t)rg * BT + bb) * p.Co + cc * CW + e4) =
                  make_float4(a[bb][e4], a[bb][e4 + 1], a[bb][e4 + 2], a[bb][e4 + 3]);
        named_sync(kBarConsumers, kConsumers);
        for (int bb = 0; bb < BT; ++bb) {
          const int b = b0 + bb;
          for (int cq = tid; cq < CQ; cq += kConsumers) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int gq = 0; gq < RG; ++gq) {
              const float4 u =
                  *reinterpret_cast<const float4*>(pb + ((size_t)gq * BT + bb) * p.Co + cq * 4);
              v.x += u.x;
              v.y += u.y;
              v.z += u.z;
              v.w += u.w;
            }
            if (b < p.B && s_pos[bb] >= 0)
              atomicAdd(
                  reinterpret_cast<float4*>(p.acc + (size_t)b * p.H + k0 + cb * p.Co + cq * 4), v);
          }
        }
        fence_proxy_async_smem();  // our stores into the stage precede the next TMA write
        named_sync(kBarConsumers, kConsumers);
        if (lane == 0) mbar_arrive(&empty[s_last]);
      }
    }

    stamp(kTlOproj);
    // ---- Residual + finalize by the last block of each (tile, band) ------
    __threadfence();
    named_sync(kBarConsumers, kConsumers);
    if (tid == 0) {
      const int ticket = atomicAdd(&p.counters[bt * N + rank], 1);
      const int last = (ticket == p.nkv - 1);
      if (last) __threadfence();
      s_flag[0] = last;
    }
    named_sync(kBarConsumers, kConsumers);
    stamp(kTlTicket);
    if (s_flag[0]) {
      T* out = reinterpret_cast<T*>(p.out);
      float* dproj = p.dbg ? p.dbg + (size_t)p.B * (2 * p.nq + 2 * p.nkv) * D : nullptr;
      const int C4 = Hc / 4;
      for (int bb = 0; bb < BT; ++bb) {
        const int b = b0 + bb;
        if (b >= p.B) continue;
        for (int c4 = tid; c4 < C4; c4 += kConsumers) {
          const size_t off = (size_t)b * p.H + k0 + c4 * 4;
          const float4 v = __ldcg(reinterpret_cast<const float4*>(p.acc + off));
          __stcg(reinterpret_cast<float4*>(p.acc + off), make_float4(0.f, 0.f, 0.f, 0.f));
          float xf[4];
          load_cvt<T, 4>(hidden + off, xf);
          const float r[4] = {xf[0] + v.x, xf[1] + v.y, xf[2] + v.z, xf[3] + v.w};
          store4<T>(out + off, r);
          if (dproj) {
            dproj[off + 0] = v.x;
            dproj[off + 1] = v.y;
            dproj[off + 2] = v.z;
            dproj[off + 3] = v.w;
          }
        }
      }
      if (tid == 0) p.counters[bt * N + rank] = 0;
    }
  }

  stamp(kTlFinal);
  // No block leaves while a peer may still write into its shared memory.
  __syncwarp();
  cluster_sync_exit();
  stamp(kTlEnd);
}

}  // namespace cf
