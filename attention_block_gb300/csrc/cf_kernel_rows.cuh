// cf_kernel_rows.cuh -- the fused decode attention block for batched decode
// (4 to 64 rows per cluster) on sm_103a.
//
// Pages cited by title and section:
//   [CF]  "ClusterFusion框架深度解析：LLM推理优化的集群级通信革命" (devpress.csdn.net)
//   [LNA] "大模型推理中的算子融合优化：LayerNorm + Attention 的 CUDA Kernel 手写与验证"
//         (asdsk.com)
//
// Same computation as cf_kernel.cuh ([CF §3.2] fused_qkv_attention_out,
// [LNA §一]); the mapping changes with the batch.  One thread-block cluster
// serves one KV head g and a tile of BT batch rows, so every weight byte of
// the head group is read once per tile (tiles of one head run together and
// share the weights through L2); its N = BT / RPC blocks
//   * split the hidden (reduction) dimension of the QKV projection, a
//     [BT x H] x [H x (G+2)d] contraction on the tensor cores with fp32
//     accumulation; the fp32 activations enter as a pair of 16-bit values
//     hi + lo, so the product keeps ~fp32 accuracy.  Tiles of 16 or more rows
//     use the fifth-generation tensor cores (tcgen05, accumulators in tensor
//     memory), smaller tiles mma.sync m16n8k16;
//   * combine the partial products with ClusterReduce in reduce-scatter form
//     over BATCH ROWS [CF §3.1.1]: block c ends up owning rows
//     [c*RPC, (c+1)*RPC) of the tile, fully summed, together with their
//     sums of squares (each block adds x^2 over its hidden band while it
//     stages x, so RMSNorm [LNA §三 stage 1] needs no separate pass over x);
//     it applies the norm scale, RoPE and the KV append to its rows and runs
//     their attention over the whole sequence on the tensor cores
//     (cf_attention_tc.cuh), so no cross-block softmax merge is needed;
//   * exchange the attention outputs with ClusterGather [CF §3.1.2] so that
//     every block holds o for all BT rows, then split the output projection
//     by columns (tensor cores again) and merge heads with fp32 atomics
//     [CF §3.2 原子写合并]; the last block per (tile, column band) adds the
//     residual and writes `out`.
// Both cluster exchanges PULL: a block signals its peers (remote mbarrier
// arrivals with cluster-scope release) when its data is complete and the
// peers read it with ld.shared::cluster, so no receive buffers take shared
// memory away from the TMA ring.  Weight and K/V tiles arrive through TMA
// with the 128-byte swizzle, so the ldmatrix fragment loads are free of bank
// conflicts; the batch rows of x arrive with each weight tile.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cf_attention_tc.cuh"
#include "cf_cluster.cuh"
#include "cf_common.cuh"
#include "cf_mma.cuh"
#include "cf_params.h"
#include "cf_ptx.cuh"
#include "cf_tc05.cuh"

namespace cf {

// Floats of one reduce-scatter slice: RPC rows of NC projection partials,
// then the RPC rows' sums of squares (padded to 4).
__host__ __device__ constexpr int rows_slice_floats(int RPC, int NC) {
  return RPC * NC + (RPC + 3) / 4 * 4;
}
// Bytes per row of the O-projection A operand: o as 16-bit hi (G*d values),
// then lo, then 16 bytes of padding (an odd multiple of 16 bytes, so the
// ldmatrix rows fall in distinct banks).
__host__ __device__ constexpr int rows_aop_pitch(int GD) { return 4 * GD + 16; }

template <typename T, int D, int G, int BT, int RPC>
__global__ void __launch_bounds__(kThreads, 1) cf_rows_kernel(const __grid_constant__ KParams p) {
  constexpr int NSEG = G + 2;        // q heads of the group, k, v
  constexpr int NC = NSEG * D;       // projection columns of the group
  constexpr int MR = BT < 16 ? 16 : BT;  // MMA rows (rows >= BT read a zero chunk)
  constexpr int MT = MR / 16;        // MMA row tiles
  constexpr int NTW = NC / 8 / kConsumerWarps;  // projection n-tiles per warp
  constexpr int CB = rows_wqkv_boxes(NC);        // 64-column boxes per W_qkv stage
  constexpr int NCG = NC / 64 / CB;              // W_qkv stages per K slice
  // Tiles of at most four rows run both projections transposed (out^T =
  // W^T x^T): 16 weight columns form the mma's M side and the N side holds
  // the rows' hi and lo halves (4 + 4 columns), so one mma does the work of
  // eight of the row-major form (M = 16 rows, 12 of them zero, and hi and lo
  // in separate mmas).
  constexpr bool TP = BT <= 4 && CB % 2 == 0;
  constexpr int MPW = CB / 2;                    // m-tiles per warp per W_qkv stage (TP)
  constexpr int GD = G * D;          // O-projection reduction size
  constexpr int SE = rows_slice_floats(RPC, NC);
  constexpr int OP = rows_aop_pitch(GD);
  constexpr int NRW = (BT + kConsumerWarps - 1) / kConsumerWarps;  // rows per warp (sumsq)
  // Tiles of 16 or more rows run both projections transposed on tcgen05:
  // M = 128 weight (or output) columns, read straight from the swizzled TMA
  // boxes as an M-major operand; N = 2*BT, the tile's rows as hi halves then
  // lo halves (a K-major operand the consumers stage); K = 16 per MMA.  One
  // thread issues the MMAs and commits them to the ring's empty barriers; the
  // fp32 accumulators live in tensor memory (lane = column, column = row
  // half) and each consumer warp reads one lane quarter, adding hi and lo.
  constexpr bool TC5 = BT >= 16;
  constexpr int N5 = 2 * BT;                     // MMA N
  constexpr int NT5 = (CB + 1) / 2;              // 128-column tiles per W_qkv stage
  constexpr int TCOLS = tmem_cols_for(NCG * NT5 * N5 > 4 * N5 ? NCG * NT5 * N5 : 4 * N5);
  static_assert(!TC5 || (CB >= 2 && NCG * NT5 * N5 <= 512 && 4 * N5 <= 512 && GD % 64 == 0 &&
                         BT % 16 == 0),
                "tensor-memory plan");
  static_assert(BT % RPC == 0 && MR % 16 == 0, "batch tile");
  static_assert(NC % (8 * kConsumerWarps) == 0, "projection columns per warp");
  static_assert(D % 64 == 0, "head_dim in 64-column swizzle boxes");
  static_assert(NCG * CB * 64 == NC && CB * 8 % kConsumerWarps == 0 && NTW == NCG * CB,
                "W_qkv column groups");
  using MK = MmaKind<T>;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int N = p.N;  // == BT / RPC
  const int rank = (int)cluster_ctarank();
  const int cid = blockIdx.x / N;
  const int g = cid / p.nbt;
  const int bt = cid % p.nbt;
  const int b0 = bt * BT;
  const int Hc = p.H / N;  // K band rows == O-proj column band
  const int k0 = rank * Hc;
  const int r0 = rank * RPC;  // first owned row of the tile

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + p.L.bars);
  uint64_t* full = bars + BarIdx::full;
  uint64_t* empty = bars + BarIdx::empty;
  uint64_t* rs_bar = bars + BarIdx::rs;  // peers' partial sums complete
  uint64_t* ga_bar = bars + BarIdx::ga;  // peers' attention outputs complete
  uint8_t* ring = sm + p.L.ring;
  float* red = reinterpret_cast<float*>(sm + p.L.red);       // [N][SE] partials
  uint8_t* un = sm + p.L.scratch;                            // abuf | warp states | A of O-proj
  float* wst = reinterpret_cast<float*>(un);
  uint8_t* aop = un;                                         // [BT][OP] bytes
  float* ofin = reinterpret_cast<float*>(sm + p.L.qkv);      // [RPC][GD] own rows' o
  float* rec = reinterpret_cast<float*>(sm + p.L.sm);        // [G][D+4] attention record
  uint4* qfr = reinterpret_cast<uint4*>(sm + p.L.xn);        // [D/16][32] Q fragments
  float* rope = reinterpret_cast<float*>(sm + p.L.rope);     // [RPC][D/2][2]
  const uint32_t* zero16 = reinterpret_cast<const uint32_t*>(sm + p.L.misc);  // 16 zero bytes
  int* s_pos = reinterpret_cast<int*>(sm + p.L.misc + 16);   // [BT]
  int* s_flag = s_pos + BT;
  float* s_rinv = reinterpret_cast<float*>(s_flag + 4);       // [RPC]
  // tcgen05 completions: [0], [1] x buffers free again, [2], [3] O-projection
  // accumulator buffers ready
  uint64_t* tc_bar = bars + BarIdx::sm;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_flag + 1);  // tensor-memory base

  // ---------------------------------------------------------------- setup --
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    if (N > 1) {
      mbar_init(rs_bar, N - 1);
      mbar_init(ga_bar, N - 1);
    }
    if constexpr (TC5)
      for (int i = 0; i < 4; ++i) mbar_init(&tc_bar[i], 1);
    fence_mbar_init_cluster();
  }
  if (tid < 4) reinterpret_cast<uint32_t*>(sm + p.L.misc)[tid] = 0u;
  if constexpr (TC5) {
    if (warp == 0) {
      tmem_alloc(s_tmem, TCOLS);
      tmem_relinquish();
    }
    tc05_fence_before();
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tensormap(&p.tm_wqkv);
    prefetch_tensormap(&p.tm_x);
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
    prefetch_tensormap(&p.tm_wo);
  }
  __syncthreads();
  if constexpr (TC5) tc05_fence_after();
  cluster_sync_all();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = tid; i < BT; i += kThreads) {
    const int b = b0 + i;
    int pos = -1;
    if (b < p.B) {
      pos = p.positions[b];
      if (pos < 0 || pos >= p.S) {
        if (rank == 0 && g == 0) atomicOr(p.errflag, kDevErrPosRange);
        pos = -1;
      }
    }
    s_pos[i] = pos;
  }
  __syncthreads();
  auto stamp = [&](int slot) {
    if (p.timeline != nullptr && tid == 0)
      p.timeline[blockIdx.x * kTimelineSlots + slot] = globaltimer_ns();
  };
  stamp(kTlStart);

  const int nkt = Hc / p.Rw;
  const int ncb = Hc / p.Co;
  const int nrt = GD / p.Ro;
  const uint32_t wbox_bytes = (uint32_t)(p.Rw * 128);
  const uint32_t x_bytes = (uint32_t)(BT * p.Rw * (int)sizeof(T));
  const int obox = p.Co / 64;                        // 64-column boxes per W_o tile
  const uint32_t obox_bytes = (uint32_t)(p.Ro * 128);

  if (warp == kConsumerWarps) {
    // ============================================== TMA producer warp ====
    if (lane == 0) {
      // Weights: evict-first when this tile is the only reader, otherwise
      // kept at normal priority for the head's other batch tiles.
      const uint64_t pol_w = p.nbt > 1 ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_kv = policy_evict_first();
      int it = 0;
      RingPos rp(0, p.stages);
      auto slot = [&](uint32_t bytes, uint64_t*& bar) -> uint8_t* {
        const int s = rp.slot;
        if (it >= p.stages) mbar_wait(&empty[s], rp.phase ^ 1u, p.errflag);
        rp.next(p.stages);
        bar = &full[s];
        mbar_arrive_expect_tx(bar, bytes);
        return ring + (size_t)s * p.stage_bytes;
      };
      // Phase 1: W_qkv tiles of the K band.  Each slice of Rw rows comes as
      // NCG stages of CB 64-column swizzled boxes (the G+2 head slices' NC
      // columns in order); the first stage of a slice also carries the
      // matching [BT x Rw] slice of x.
      for (int kt = 0; kt < nkt; ++kt) {
        const int y = k0 + kt * p.Rw;
        for (int cg = 0; cg < NCG; ++cg, ++it) {
          uint64_t* bar;
          uint8_t* dst = slot(CB * wbox_bytes + (cg == 0 ? x_bytes : 0u), bar);
          for (int bx = 0; bx < CB; ++bx) {
            const int col = (cg * CB + bx) * 64;  // column inside the group's NC columns
            const int sg = col / D, cin = col % D;
            const int gx = (sg < G) ? ((g * G + sg) * D + cin)
                                    : ((sg == G ? p.nq + g : p.nq + p.nkv + g) * D + cin);
            tma_load_2d(dst + bx * wbox_bytes, &p.tm_wqkv, gx, y, bar, pol_w);
          }
          if (cg == 0) tma_load_2d(dst + CB * wbox_bytes, &p.tm_x, y, b0, bar, pol_w);
        }
      }
      if (p.timeline) p.timeline[blockIdx.x * kTimelineSlots + kTlProdW] = globaltimer_ns();
      // Phase 2: K/V tiles of the owned rows, whole sequence each, as
      // 64-column swizzled boxes: K [D/64][Rt][64] then V.
      const uint32_t kv_box = (uint32_t)(p.Rt * 128);
      constexpr int NB = D / 64;
      for (int r = 0; r < RPC; ++r) {
        int t0, t1;
        kv_tile_range(s_pos[r0 + r], p.Rt, 0, 1, t0, t1);
        for (int t = t0; t < t1; ++t, ++it) {
          uint64_t* bar;
          uint8_t* dst = slot(2 * NB * kv_box, bar);
#pragma unroll
          for (int bx = 0; bx < NB; ++bx) {
            tma_load_4d(dst + bx * kv_box, &p.tm_k, bx * 64, g, t * p.Rt, b0 + r0 + r, bar,
                        pol_kv);
            tma_load_4d(dst + (NB + bx) * kv_box, &p.tm_v, bx * 64, g, t * p.Rt, b0 + r0 + r,
                        bar, pol_kv);
          }
        }
      }
      if (p.timeline) p.timeline[blockIdx.x * kTimelineSlots + kTlProdKV] = globaltimer_ns();
      // Phase 3: W_o tiles (swizzled 64-column boxes) of the column band.
      for (int cb = 0; cb < ncb; ++cb)
        for (int rt = 0; rt < nrt; ++rt, ++it) {
          uint64_t* bar;
          uint8_t* dst = slot(obox * obox_bytes, bar);
          for (int bx = 0; bx < obox; ++bx)
            tma_load_2d(dst + bx * obox_bytes, &p.tm_wo, k0 + cb * p.Co + bx * 64,
                        g * GD + rt * p.Ro, bar, pol_w);
        }
      if (p.timeline) p.timeline[blockIdx.x * kTimelineSlots + kTlProdAll] = globaltimer_ns();
    }
    __syncwarp();
  } else {
    // ============================================== consumer warps =======
    const T* __restrict__ hidden = reinterpret_cast<const T*>(p.hidden);
    const T* __restrict__ lnw = reinterpret_cast<const T*>(p.ln_w);
    int it = 0;
    const int apitch = (p.Rw + 8) * 2;  // bytes per staged A row (odd multiple of 16)
    const int abytes = BT * apitch;

    // ---- Phase 0: the owned rows' RoPE factors ------------------------------
    for (int idx = tid; idx < RPC * (D / 2); idx += kConsumers) {
      const int r = idx / (D / 2), j = idx % (D / 2);
      const int pos = s_pos[r0 + r];
      float c = 1.f, sn = 0.f;
      if (pos >= 0) rope_cos_sin(pos, p.turn_hi[j], p.turn_lo[j], c, sn);
      rope[2 * idx] = c;
      rope[2 * idx + 1] = sn;
    }
    named_sync(kBarConsumers, kConsumers);
    stamp(kTlNorm);

    // ---- Phase 1: [BT x Hc] x [Hc x NC] on the tensor cores, with the
    // rows' sums of squares over the band [LNA §三 stage 1] -----------------
    const uint32_t tmem = TC5 ? *s_tmem : 0u;
    if constexpr (TC5) {
      // x * g of each K slice as the B operand: ceil(Rw/64) K-major swizzled
      // slabs of N5 rows (hi rows 0..BT-1, lo rows BT..2BT-1), double-buffered
      const int xslab = N5 * 128;
      const uint32_t xbuf = (uint32_t)(((p.Rw + 63) / 64) * xslab);
      const uint32_t idesc = idesc_kind_f16(MK::kBf16, 128, N5, true);
      float ss[NRW];
#pragma unroll
      for (int i = 0; i < NRW; ++i) ss[i] = 0.f;
      RingPos rp(it, p.stages);
      for (int kt = 0; kt < nkt; ++kt) {
        uint8_t* xs = un + (size_t)(kt & 1) * xbuf;
        for (int cg = 0; cg < NCG; ++cg, ++it, rp.next(p.stages)) {
          const int s = rp.slot;
          uint8_t* st = ring + (size_t)s * p.stage_bytes;
          if (cg == 0) {
            mbar_wait(&full[s], rp.phase, p.errflag);
            // the MMAs of slice kt - 2 read this buffer
            if (kt >= 2) mbar_wait(&tc_bar[kt & 1], ((kt - 2) >> 1) & 1, p.errflag);
            const T* xt = reinterpret_cast<const T*>(st + CB * wbox_bytes);  // [BT][Rw]
#pragma unroll
            for (int i = 0; i < NRW; ++i) {
              const int row = warp + i * kConsumerWarps;
              if (row < BT) {
                for (int k = 2 * lane; k < p.Rw; k += 64) {
                  float f[2];
                  load_cvt<T, 2>(xt + row * p.Rw + k, f);
                  ss[i] = fmaf(f[0], f[0], fmaf(f[1], f[1], ss[i]));
                  float gw[2];
                  load_cvt<T, 2>(lnw + k0 + kt * p.Rw + k, gw);
                  uint32_t hi, lo;
                  MK::split2(f[0] * gw[0], f[1] * gw[1], hi, lo);
                  uint8_t* sl = xs + (k >> 6) * xslab;
                  const int j = (k & 63) >> 3, e2 = (k & 7) * 2, rl = BT + row;
                  *reinterpret_cast<uint32_t*>(sl + row * 128 + ((j ^ (row & 7)) << 4) + e2) = hi;
                  *reinterpret_cast<uint32_t*>(sl + rl * 128 + ((j ^ (rl & 7)) << 4) + e2) = lo;
                }
              }
            }
            fence_proxy_async_smem();
            named_sync(kBarConsumers, kConsumers);
          }
          if (tid == 0) {
            if (cg != 0) mbar_wait(&full[s], rp.phase, p.errflag);
            tc05_fence_after();
#pragma unroll
            for (int t = 0; t < NT5; ++t) {
              // 128 columns from box c0 / 64 (the last tile of a 3-box stage
              // overlaps the previous one; its duplicate half is not stored)
              const int c0 = (128 * t < CB * 64 - 128) ? 128 * t : CB * 64 - 128;
              const uint32_t a0 = smem_u32(st + (c0 / 64) * wbox_bytes);
              const uint32_t d = tmem + (uint32_t)((cg * NT5 + t) * N5);
              for (int ks = 0; ks < p.Rw / 16; ++ks) {
                const uint64_t ad = smem_desc_mn_sw128(a0 + (uint32_t)ks * 2048u, wbox_bytes, 1024);
                const uint64_t bd =
                    smem_desc_k_sw128(smem_u32(xs + (ks >> 2) * xslab) + (uint32_t)(ks & 3) * 32u,
                                      1024);
                tc05_mma_f16(d, ad, bd, idesc, kt > 0 || ks > 0);
              }
            }
            // the other warps' shares of the stage release, then the MMAs'
            mbar_arrive_cnt(&empty[s], kConsumerWarps - 1);
            tc05_commit(&empty[s]);
            if (cg == NCG - 1) tc05_commit(&tc_bar[kt & 1]);
          }
          __syncwarp();
        }
      }
      // the last slice's commit covers every earlier MMA
      mbar_wait(&tc_bar[(nkt - 1) & 1], ((nkt - 1) >> 1) & 1, p.errflag);
      tc05_fence_after();
      stamp(kTlProjLoop);
      // Partial sums -> red, slice-major (row r to slice r / RPC).  Warp w
      // reads lane quarter w % 4 (32 columns) for rows [h*BT/2, (h+1)*BT/2),
      // h = w / 4: lanes store consecutive columns of one row.
      const int qd = warp & 3, hrow = (warp >> 2) * (BT / 2);
#pragma unroll
      for (int cg = 0; cg < NCG; ++cg)
#pragma unroll
        for (int t = 0; t < NT5; ++t) {
          const int c0 = (128 * t < CB * 64 - 128) ? 128 * t : CB * 64 - 128;
          const int cin = c0 + 32 * qd + lane;
          const bool keep = cin >= 128 * t;
          const int n = cg * CB * 64 + cin;
          const uint32_t d =
              tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)((cg * NT5 + t) * N5 + hrow);
#pragma unroll
          for (int r8 = 0; r8 < BT / 2; r8 += 8) {
            float vh[8], vl[8];
            tmem_ld_32x32b_x8(d + (uint32_t)r8, vh);
            tmem_ld_32x32b_x8(d + (uint32_t)(BT + r8), vl);
            if (keep) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int row = hrow + r8 + i;
                red[(row / RPC) * SE + (row % RPC) * NC + n] = vh[i] + vl[i];
              }
            }
          }
        }
      tc05_fence_before();
#pragma unroll
      for (int i = 0; i < NRW; ++i) {
        const int row = warp + i * kConsumerWarps;
        const float v = warp_sum(ss[i]);
        if (row < BT && lane == 0) red[(row / RPC) * SE + RPC * NC + row % RPC] = v;
      }
      named_sync(kBarConsumers, kConsumers);
    } else {
      float acc[MT][NTW][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mt][j][e] = 0.f;
      float acct[TP ? NCG * MPW : 1][4];  // transposed form: [m-tile][c-fragment]
#pragma unroll
      for (int j = 0; j < (TP ? NCG * MPW : 1); ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acct[j][e] = 0.f;
      float ss[NRW];
#pragma unroll
      for (int i = 0; i < NRW; ++i) ss[i] = 0.f;
      RingPos rp(it, p.stages);
      for (int kt = 0; kt < nkt; ++kt) {
        // x * g of this K slice as hi + lo 16-bit pairs (double-buffered)
        uint8_t* ahi = un + (size_t)(kt & 1) * 2 * abytes;
        uint8_t* alo = ahi + abytes;
#pragma unroll
        for (int cg = 0; cg < NCG; ++cg, ++it, rp.next(p.stages)) {
          const int s = rp.slot;
          mbar_wait(&full[s], rp.phase, p.errflag);
          uint8_t* st = ring + (size_t)s * p.stage_bytes;
          if (cg == 0) {
            // stage the slice's x * g; warp w stages rows w, w+8, ...
            const T* xt = reinterpret_cast<const T*>(st + CB * wbox_bytes);  // [BT][Rw]
#pragma unroll
            for (int i = 0; i < NRW; ++i) {
              const int row = warp + i * kConsumerWarps;
              if (row < BT) {
                for (int k = 2 * lane; k < p.Rw; k += 64) {
                  float f[2];
                  load_cvt<T, 2>(xt + row * p.Rw + k, f);
                  ss[i] = fmaf(f[0], f[0], fmaf(f[1], f[1], ss[i]));
                  float gw[2];
                  load_cvt<T, 2>(lnw + k0 + kt * p.Rw + k, gw);
                  const float v0 = f[0] * gw[0], v1 = f[1] * gw[1];
                  uint32_t hi, lo;
                  MK::split2(v0, v1, hi, lo);
                  *reinterpret_cast<uint32_t*>(ahi + row * apitch + k * 2) = hi;
                  *reinterpret_cast<uint32_t*>(alo + row * apitch + k * 2) = lo;
                }
              }
            }
            named_sync(kBarConsumers, kConsumers);
          }
          if constexpr (TP) {
            for (int ks = 0; ks < p.Rw / 16; ++ks) {
              uint32_t b0x, b1x;
              ldmatrix_b_hilo_rows(b0x, b1x, ahi, alo, apitch, BT, zero16, ks * 16, lane);
#pragma unroll
              for (int jj = 0; jj < MPW; ++jj) {
                const int m0 = (warp * MPW + jj) * 16;  // column inside the stage's CB*64
                uint32_t a[4];
                ldmatrix_at_sw128(a, st + (m0 / 64) * wbox_bytes, ks * 16, m0 % 64, lane);
                MK::mma(acct[cg * MPW + jj], a, b0x, b1x);
              }
            }
          } else {
            for (int ks = 0; ks < p.Rw / 16; ++ks) {
              uint32_t ah[MT][4], al[MT][4];
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                ldmatrix_a_rows(ah[mt], ahi + mt * 16 * apitch + ks * 32, apitch, BT - mt * 16,
                                zero16, lane);
                ldmatrix_a_rows(al[mt], alo + mt * 16 * apitch + ks * 32, apitch, BT - mt * 16,
                                zero16, lane);
              }
#pragma unroll
              for (int jj = 0; jj < CB; ++jj) {
                const int n = (warp * CB + jj) * 8;  // column inside the stage's CB*64
                uint32_t b0r, b1r;
                ldmatrix_b_sw128(b0r, b1r, st + (n / 64) * wbox_bytes, ks * 16, n % 64, lane);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                  MK::mma(acc[mt][cg * CB + jj], ah[mt], b0r, b1r);
                  MK::mma(acc[mt][cg * CB + jj], al[mt], b0r, b1r);
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
      }
      stamp(kTlProjLoop);
      // Partial sums -> red, slice-major: row r goes to slice r / RPC, so the
      // rows block c owns form its contiguous slice c.
      const int gq = lane >> 2, tq = lane & 3;
      if constexpr (TP) {
        // acct j holds columns (gq, gq + 8) of m-tile warp*MPW + j%MPW of
        // column group j/MPW; its c-fragment columns 2tq, 2tq+1 are rows
        // 2tq, 2tq+1 (hi) for tq < 2 and the lo halves of rows 2tq-4, 2tq-3
        // for tq >= 2: lane tq adds the lo part from lane tq + 2.
#pragma unroll
        for (int j = 0; j < NCG * MPW; ++j) {
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = acct[j][e] + __shfl_xor_sync(0xffffffffu, acct[j][e], 2);
          const int col = (j / MPW) * CB * 64 + (warp * MPW + j % MPW) * 16 + gq;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int row = 2 * tq + h;
            if (tq < 2 && row < BT) {
              float* dst = red + (row / RPC) * SE + (row % RPC) * NC + col;
              dst[0] = v[h];
              dst[8] = v[2 + h];
            }
          }
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int j = 0; j < NTW; ++j) {
            // acc j covers n-tile warp*CB + j%CB of column group j/CB
            const int n = (j / CB) * CB * 64 + (warp * CB + j % CB) * 8 + 2 * tq;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int row = mt * 16 + gq + 8 * h;
              if (row < BT)
                *reinterpret_cast<float2*>(red + (row / RPC) * SE + (row % RPC) * NC + n) =
                    make_float2(acc[mt][j][2 * h], acc[mt][j][2 * h + 1]);
            }
          }
      }
#pragma unroll
      for (int i = 0; i < NRW; ++i) {
        const int row = warp + i * kConsumerWarps;
        const float v = warp_sum(ss[i]);
        if (row < BT && lane == 0) red[(row / RPC) * SE + RPC * NC + row % RPC] = v;
      }
      named_sync(kBarConsumers, kConsumers);
    }
    stamp(kTlProj);

    // ---- ClusterReduce (reduce-scatter over rows, pulled): block `rank`
    // owns rows [rank*RPC, (rank+1)*RPC) of the tile, fully summed ---------
    if (N > 1) {
      if (tid == 0) cluster_signal_peers(rs_bar, rank, N);
      cluster_pull_reduce_slice<kConsumers>(red, SE, rs_bar, rank, N, tid, p.errflag);
      named_sync(kBarConsumers, kConsumers);
    }
    float* own = red + rank * SE;  // [RPC][NSEG][D], then [RPC] sums of squares
    if (tid < RPC) {
      s_rinv[tid] = (b0 + r0 + tid < p.B) ? 1.0f / sqrtf(own[RPC * NC + tid] / (float)p.H + p.eps)
                                          : 0.f;
    }
    named_sync(kBarConsumers, kConsumers);
    stamp(kTlReduceScatter);

    // ---- RMSNorm scale, RoPE, KV append of the owned rows [LNA §三] -------
    {
      T* kc = reinterpret_cast<T*>(p.k_cache);
      T* vc = reinterpret_cast<T*>(p.v_cache);
      for (int idx = tid; idx < RPC * NSEG * (D / 2); idx += kConsumers) {
        const int r = idx / (NSEG * (D / 2)), rem = idx % (NSEG * (D / 2));
        const int sg = rem / (D / 2), i = rem % (D / 2);
        const int pos = s_pos[r0 + r];
        float* u = own + (r * NSEG + sg) * D;
        float a = u[i] * s_rinv[r], bv = u[i + D / 2] * s_rinv[r];
        if (sg <= G && pos >= 0) {
          const float c = rope[2 * (r * (D / 2) + i)], sn = rope[2 * (r * (D / 2) + i) + 1];
          const float ra = a * c - bv * sn;
          const float rb = bv * c + a * sn;
          a = ra;
          bv = rb;
        }
        if (sg >= G && pos >= 0) {
          T* cache = (sg == G) ? kc : vc;
          const size_t base = (((size_t)(b0 + r0 + r) * p.S + pos) * p.nkv + g) * D;
          cache[base + i] = Elem<T>::from_f(a);
          cache[base + D / 2 + i] = Elem<T>::from_f(bv);
        }
        u[i] = a;
        u[i + D / 2] = bv;
      }
      named_sync(kBarConsumers, kConsumers);
      if (p.dbg != nullptr) {
        float* dq = p.dbg;
        float* dk = dq + (size_t)p.B * p.nq * D;
        float* dv = dk + (size_t)p.B * p.nkv * D;
        for (int idx = tid; idx < RPC * NC; idx += kConsumers) {
          const int r = idx / NC, rem = idx % NC, sg = rem / D, dim = rem % D;
          const int b = b0 + r0 + r;
          if (b >= p.B || s_pos[r0 + r] < 0) continue;
          if (sg < G) dq[((size_t)b * p.nq + g * G + sg) * D + dim] = own[idx];
          else if (sg == G) dk[((size_t)b * p.nkv + g) * D + dim] = own[idx];
          else dv[((size_t)b * p.nkv + g) * D + dim] = own[idx];
        }
      }
    }
    stamp(kTlGather);

    // ---- Attention of the owned rows over their whole sequence ------------
    for (int r = 0; r < RPC; ++r) {
      const float* qr = own + r * NC;
      attend_row_tc<T, D, G>(p, qr, qr + G * D, qr + (G + 1) * D, s_pos[r0 + r], true, ring, full,
                             empty, it, wst, qfr, rec,
                             (p.timeline != nullptr && r == 0)
                                 ? p.timeline + blockIdx.x * kTimelineSlots
                                 : nullptr);
      for (int idx = tid; idx < GD; idx += kConsumers) {
        const int h = idx / D, dim = idx % D;
        const float L = rec[h * (D + 4) + D + 1];
        ofin[r * GD + idx] = (L > 0.f) ? rec[h * (D + 4) + dim] / L : 0.f;
      }
      named_sync(kBarConsumers, kConsumers);
    }
    stamp(kTlAttn);
    if (p.dbg != nullptr) {
      float* dob = p.dbg + (size_t)p.B * (p.nq + 2 * p.nkv) * D;
      for (int idx = tid; idx < RPC * GD; idx += kConsumers) {
        const int r = idx / GD, rem = idx % GD;
        const int b = b0 + r0 + r;
        if (b >= p.B || s_pos[r0 + r] < 0) continue;
        dob[((size_t)b * p.nq + g * G) * D + rem] = ofin[idx];
      }
    }
    // Own rows of the O-projection operand (o as hi + lo 16-bit values); the
    // warp states that shared this memory are no longer needed.  For tcgen05
    // it is K-major swizzled: GD/64 slabs of N5 rows (hi rows, then lo rows).
    for (int i2 = tid; i2 < RPC * GD / 2; i2 += kConsumers) {
      const int r = (2 * i2) / GD, k = (2 * i2) % GD;
      uint32_t hi, lo;
      MK::split2(ofin[r * GD + k], ofin[r * GD + k + 1], hi, lo);
      if constexpr (TC5) {
        uint8_t* sl = aop + (k >> 6) * (N5 * 128);
        const int j = (k & 63) >> 3, e2 = (k & 7) * 2, rh = r0 + r, rl = BT + r0 + r;
        *reinterpret_cast<uint32_t*>(sl + rh * 128 + ((j ^ (rh & 7)) << 4) + e2) = hi;
        *reinterpret_cast<uint32_t*>(sl + rl * 128 + ((j ^ (rl & 7)) << 4) + e2) = lo;
      } else {
        uint8_t* row = aop + (r0 + r) * OP;
        *reinterpret_cast<uint32_t*>(row + k * 2) = hi;
        *reinterpret_cast<uint32_t*>(row + 2 * GD + k * 2) = lo;
      }
    }
    if constexpr (TC5) fence_proxy_async_smem();
    named_sync(kBarConsumers, kConsumers);
    stamp(kTlMax);

    // ---- ClusterGather of o [CF §3.1.2], pulled: every block gets all BT
    // rows of the A operand ---------------------------------------------------
    if (N > 1) {
      if (tid == 0) cluster_signal_peers(ga_bar, rank, N);
      if constexpr (TC5) {
        // block q's rows: RPC rows of 128 bytes in the hi and the lo half of
        // every slab, i.e. 2 * GD / 64 pieces BT * 128 bytes apart
        cluster_pull_gather<kConsumers>(aop, RPC * 128, RPC * 128, 2 * (GD / 64), BT * 128, ga_bar,
                                        rank, N, tid, p.errflag);
        fence_proxy_async_smem();
      } else {
        cluster_pull_gather<kConsumers>(aop, RPC * OP, RPC * OP, 1, 0, ga_bar, rank, N, tid,
                                        p.errflag);
      }
      named_sync(kBarConsumers, kConsumers);
    }
    stamp(kTlSum);

    // ---- Phase 3: [BT x GD] x [GD x Co] per column box on the tensor cores,
    // fp32 atomics into the accumulator [CF §3.2] ----------------------------
    if constexpr (TC5) {
      // Transposed on tcgen05: per column band, Co/128 tiles of 128 output
      // columns (M) x N5 (the rows' hi and lo halves), K = the band's GD rows
      // of W_o in Ro-row stages.  Bands alternate between two accumulator
      // buffers, so the MMAs of band cb run while the warps drain band cb - 1.
      const int ntl = p.Co / 128;
      const uint32_t idesc = idesc_kind_f16(MK::kBf16, 128, N5, true);
      const int it0 = it;
      const int qd = warp & 3, hrow = (warp >> 2) * (BT / 2);
      RingPos rp(it0, p.stages);  // advanced by the issuing thread only
      for (int cb = 0; cb <= ncb; ++cb) {
        if (cb < ncb && tid == 0) {
          tc05_fence_after();
          const uint32_t dbuf = tmem + (uint32_t)((cb & 1) * 2 * N5);
          for (int rt = 0; rt < nrt; ++rt, rp.next(p.stages)) {
            const int s = rp.slot;
            mbar_wait(&full[s], rp.phase, p.errflag);
            if (cb == 0 && rt == 0) stamp(kTlOprojFirst);
            uint8_t* st = ring + (size_t)s * p.stage_bytes;
            for (int tt = 0; tt < ntl; ++tt) {
              const uint32_t a0 = smem_u32(st + 2 * tt * obox_bytes);
              for (int ks = 0; ks < p.Ro / 16; ++ks) {
                const int kg = rt * p.Ro + ks * 16;
                const uint64_t ad = smem_desc_mn_sw128(a0 + (uint32_t)ks * 2048u, obox_bytes, 1024);
                const uint64_t bd = smem_desc_k_sw128(
                    smem_u32(aop + (kg >> 6) * (N5 * 128)) + (uint32_t)((kg & 63) >> 4) * 32u, 1024);
                tc05_mma_f16(dbuf + (uint32_t)(tt * N5), ad, bd, idesc, rt > 0 || ks > 0);
              }
            }
            mbar_arrive_cnt(&empty[s], kConsumerWarps - 1);
            tc05_commit(&empty[s]);
          }
          tc05_commit(&tc_bar[2 + (cb & 1)]);
        }
        __syncwarp();
        if (cb >= 1) {
          const int pc = cb - 1;
          mbar_wait(&tc_bar[2 + (pc & 1)], (pc >> 1) & 1, p.errflag);
          tc05_fence_after();
          // lane = output column: each atomic instruction of the warp adds
          // 32 consecutive floats of one row (float4 atomics after a lane
          // transpose measured slower: the L2 cost follows the bytes)
          for (int tt = 0; tt < ntl; ++tt) {
            const int col = k0 + pc * p.Co + 128 * tt + 32 * qd + lane;
            const uint32_t d = tmem + ((uint32_t)(32 * qd) << 16) +
                               (uint32_t)((pc & 1) * 2 * N5 + tt * N5 + hrow);
#pragma unroll
            for (int r8 = 0; r8 < BT / 2; r8 += 8) {
              float vh[8], vl[8];
              tmem_ld_32x32b_x8(d + (uint32_t)r8, vh);
              tmem_ld_32x32b_x8(d + (uint32_t)(BT + r8), vl);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int row = hrow + r8 + i;
                if (b0 + row < p.B && s_pos[row] >= 0)
                  atomicAdd(p.acc + (size_t)(b0 + row) * p.H + col, vh[i] + vl[i]);
              }
            }
          }
          tc05_fence_before();
        }
        named_sync(kBarConsumers, kConsumers);
      }
      it = it0 + ncb * nrt;
      // Every MMA has completed (the last band's commit was waited for); make
      // sure of it even after an expired wait before the memory is freed.
      if (tid == 0) {
        tc05_commit(&tc_bar[0]);
        tc05_drain(&tc_bar[0], (uint32_t)(((nkt + 1) / 2) & 1), 1u << 22);
      }
    } else if constexpr (BT <= 4) {
      // Transposed (out^T = W_o^T o^T, see the projection): per column band,
      // warp w takes m-tiles w, w + 8 (16 columns each) of the Co columns.
      const int mtiles = p.Co / 16;
      const int gq = lane >> 2, tq = lane & 3;
      const bool even = (gq & 1) == 0;
      RingPos rp(it, p.stages);
      for (int cb = 0; cb < ncb; ++cb) {
        float acc[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
        for (int rt = 0; rt < nrt; ++rt, ++it, rp.next(p.stages)) {
          const int s = rp.slot;
          mbar_wait(&full[s], rp.phase, p.errflag);
          if (cb == 0 && rt == 0) stamp(kTlOprojFirst);
          uint8_t* st = ring + (size_t)s * p.stage_bytes;
          for (int ks = 0; ks < p.Ro / 16; ++ks) {
            const int kglob = rt * p.Ro + ks * 16;
            uint32_t b0x, b1x;
            ldmatrix_b_hilo_rows(b0x, b1x, aop, aop + 2 * GD, OP, BT, zero16, kglob, lane);
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int mt = warp + j * kConsumerWarps;
              if (mt < mtiles) {
                const int m0 = mt * 16;
                uint32_t a[4];
                ldmatrix_at_sw128(a, st + (m0 / 64) * obox_bytes, ks * 16, m0 % 64, lane);
                MK::mma(acc[j], a, b0x, b1x);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        // c-fragment: columns (gq, gq + 8) x rows (2tq, 2tq + 1), lo halves in
        // lanes tq + 2.  After adding them, even-gq lanes take row 2tq of
        // columns (gq, gq + 1) and (gq + 8, gq + 9) and odd-gq lanes row
        // 2tq + 1 of (gq - 1, gq) and (gq + 7, gq + 8), so each atomic adds two
        // adjacent columns.
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int mt = warp + j * kConsumerWarps;
          if (mt >= mtiles) continue;  // warp-uniform
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = acc[j][e] + __shfl_xor_sync(0xffffffffu, acc[j][e], 2);
          const float x = __shfl_xor_sync(0xffffffffu, even ? v[1] : v[0], 4);
          const float y = __shfl_xor_sync(0xffffffffu, even ? v[3] : v[2], 4);
          const int row = 2 * tq + (even ? 0 : 1);
          const int col = k0 + cb * p.Co + mt * 16 + (even ? gq : gq - 1);
          if (tq < 2 && row < BT && b0 + row < p.B && s_pos[row] >= 0) {
            float* dst = p.acc + (size_t)(b0 + row) * p.H + col;
            atomicAdd(reinterpret_cast<float2*>(dst), even ? make_float2(v[0], x) : make_float2(x, v[1]));
            atomicAdd(reinterpret_cast<float2*>(dst + 8),
                      even ? make_float2(v[2], y) : make_float2(y, v[3]));
          }
        }
      }
    } else {
      const int ntiles = p.Co / 8;
      const int gq = lane >> 2, tq = lane & 3;
      RingPos rp(it, p.stages);
      for (int cb = 0; cb < ncb; ++cb) {
        float acc[MT][4][4];  // up to 4 n-tiles per warp per box (Co <= 256)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][j][e] = 0.f;
        for (int rt = 0; rt < nrt; ++rt, ++it, rp.next(p.stages)) {
          const int s = rp.slot;
          mbar_wait(&full[s], rp.phase, p.errflag);
          if (cb == 0 && rt == 0) stamp(kTlOprojFirst);
          uint8_t* st = ring + (size_t)s * p.stage_bytes;
          for (int ks = 0; ks < p.Ro / 16; ++ks) {
            const int kglob = rt * p.Ro + ks * 16;
            uint32_t ah[MT][4], al[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              ldmatrix_a_rows(ah[mt], aop + mt * 16 * OP + kglob * 2, OP, BT - mt * 16, zero16,
                              lane);
              ldmatrix_a_rows(al[mt], aop + mt * 16 * OP + 2 * GD + kglob * 2, OP, BT - mt * 16,
                              zero16, lane);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int nt = warp + j * kConsumerWarps;
              if (nt < ntiles) {
                const int n = nt * 8;
                uint32_t b0r, b1r;
                ldmatrix_b_sw128(b0r, b1r, st + (n / 64) * obox_bytes, ks * 16, n % 64, lane);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                  MK::mma(acc[mt][j], ah[mt], b0r, b1r);
                  MK::mma(acc[mt][j], al[mt], b0r, b1r);
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int nt = warp + j * kConsumerWarps;
          if (nt >= ntiles) continue;
          const int col = k0 + cb * p.Co + nt * 8 + 2 * tq;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int row = mt * 16 + gq + 8 * h;
              if (row < BT && b0 + row < p.B && s_pos[row] >= 0)
                atomicAdd(reinterpret_cast<float2*>(p.acc + (size_t)(b0 + row) * p.H + col),
                          make_float2(acc[mt][j][2 * h], acc[mt][j][2 * h + 1]));
            }
        }
      }
    }
    stamp(kTlOproj);

    // ---- Residual + finalize by the last block of each (tile, band) ------
    __threadfence();
    named_sync(kBarConsumers, kConsumers);
    if constexpr (TC5) {
      if (warp == 0) {
        tc05_fence_after();
        tmem_dealloc(tmem, TCOLS);
      }
    }
    // The last F blocks to arrive for a (tile, band) split its rows; all but
    // the very last wait (bounded) until every KV head has arrived.  The host
    // asks for F > 1 only when the whole grid is resident at once.  The same
    // counter then counts finished shares; the last share resets it.
    const int F = p.fin_split > 1 ? p.fin_split : 1;
    int* ctr = &p.counters[bt * N + rank];
    if (tid == 0) {
      const int ticket = atomicAdd(ctr, 1);
      int share = -1;
      if (ticket >= p.nkv - F) {
        share = ticket - (p.nkv - F);
        if (ticket != p.nkv - 1) wait_count_at_least(ctr, p.nkv, p.errflag);
        __threadfence();
      }
      s_flag[0] = share;
    }
    named_sync(kBarConsumers, kConsumers);
    stamp(kTlTicket);
    if (s_flag[0] >= 0) {
      const int share = s_flag[0];
      const int rbeg = share * BT / F, rend = (share + 1) * BT / F;
      T* out = reinterpret_cast<T*>(p.out);
      float* dproj = p.dbg ? p.dbg + (size_t)p.B * (2 * p.nq + 2 * p.nkv) * D : nullptr;
      // UNR rows' worth of loads in flight per thread before any store (one
      // block finalizes the whole band, so its memory parallelism sets the
      // launch's tail).
      constexpr int UNR = BT >= 32 ? 8 : 4;
      const int C4 = Hc / 4, total = (rend - rbeg) * C4;
      for (int base = tid; base < total; base += kConsumers * UNR) {
        float4 v[UNR];
        float xf[UNR][4];
        size_t off[UNR];
        bool ok[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int i4 = base + u * kConsumers;
          const int bb = rbeg + i4 / C4, c4 = i4 % C4;
          ok[u] = i4 < total && b0 + bb < p.B;
          off[u] = (size_t)(b0 + bb) * p.H + k0 + c4 * 4;
          if (ok[u]) {
            v[u] = __ldcg(reinterpret_cast<const float4*>(p.acc + off[u]));
            load_cvt<T, 4>(hidden + off[u], xf[u]);
          }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          if (!ok[u]) continue;
          __stcg(reinterpret_cast<float4*>(p.acc + off[u]), make_float4(0.f, 0.f, 0.f, 0.f));
          const float r4[4] = {xf[u][0] + v[u].x, xf[u][1] + v[u].y, xf[u][2] + v[u].z,
                               xf[u][3] + v[u].w};
          store4<T>(out + off[u], r4);
          if (dproj) {
            dproj[off[u] + 0] = v[u].x;
            dproj[off[u] + 1] = v[u].y;
            dproj[off[u] + 2] = v[u].z;
            dproj[off[u] + 3] = v[u].w;
          }
        }
      }
      if (F == 1) {
        if (tid == 0) *ctr = 0;
      } else {
        __threadfence();
        named_sync(kBarConsumers, kConsumers);
        if (tid == 0 && atomicAdd(ctr, 1) == p.nkv + F - 1) *ctr = 0;
      }
    }
  }
  stamp(kTlFinal);
  __syncwarp();
  // Peers may still read this block's shared memory (reduce-scatter slices,
  // the A operand rows) until they pass this barrier.
  cluster_sync_exit();
  stamp(kTlEnd);
}

}  // namespace cf
