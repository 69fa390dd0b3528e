// cf_mla.cu -- the DeepSeek multi-head latent attention (MLA) variant of the
// fused decode attention block on sm_103a, and its C ABI (include/cf_mla.h).
//
// Page cited by title and section:
//   [CF] "ClusterFusion框架深度解析：LLM推理优化的集群级通信革命"
//        (devpress.csdn.net), §5.2 DeepSeek-MLA特殊处理 (the latent key/value
//        cache partitioned across clusters; ClusterReduce in a sparse form),
//        §3.1.1 (ClusterReduce), §3.2 (online softmax, atomic merge).
//   [LNA] "大模型推理中的算子融合优化：LayerNorm + Attention 的 CUDA Kernel
//         手写与验证" (asdsk.com), §三 stage 1 (RMSNorm), §一 (residual).
//
// One persistent launch per decode step: a grid of 4-block clusters, one
// block per SM, every block resident at once (the host sizes the grid from
// the resident-cluster count).  Phases, separated by grid-wide barriers whose
// waits are bounded:
//   A  y = n . [w_q | w_dkv] with n = x * ln_weight; the RMSNorm scale of each
//      row is applied when partial sums are flushed.  The merged weight is cut
//      into 192-column groups (one per query head, then the latent columns)
//      of 64-row tiles; block k takes a contiguous run of tiles and adds its
//      partial sums into the fp32 workspace y with atomics.
//   B  q_lat[h, i] = sum_j w_ukv[i, k part of h, j] q_nope[h, j] (the
//      absorption of w_uk into the query), the RoPE of every query's position
//      part, and the latent row: c' = RMSNorm(c), RoPE(kr), the cache append.
//   C  attention.  The cached positions of a row are split across the
//      clusters assigned to that row and, inside a cluster, across its 4
//      blocks [CF §5.2 潜在键值缓存分区到不同集群].  Warp w keeps online-softmax
//      states (m, l, o_lat[512]) of heads w, w + 8, ...; lane l owns latent
//      dims 16l..16l+15 and position dims 2l, 2l+1 of each cached row.  The
//      sparse ClusterReduce [CF §5.2 修改ClusterReduce支持稀疏归约]: head h's
//      states go only to cluster block (h % 8) % 4 (one st.async push each, no
//      all-reduce), which merges the 4 states and writes one partial per
//      (cluster, head).
//   D  one cluster per head: the merge of the clusters' partials (max, then
//      rescaled sums), o_h = o_lat_h . w_uv_h split over the cluster's blocks
//      by latent rows and summed by ClusterReduce (all-reduce), then the w_o
//      product of each block's column band, fp32 atomics into the
//      accumulator, and the residual by the last head to finish a band.
// A producer warp streams every tile the block reads, in the consumers'
// order, through a ring of shared-memory stages (TMA tensor loads for the
// weights, bulk copies of contiguous latent rows for the cache), running
// ahead across the barriers.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "cf.h"
#include "cf_cluster.cuh"
#include "cf_common.cuh"
#include "cf_mma.cuh"
#include "cf_mla.h"
#include "cf_params.h"
#include "cf_ptx.cuh"
#include "cf_test.h"
#include "cf_tmap.h"

namespace cf {
namespace mla {

constexpr int DN = 128, DR = 64, DV = 128, DC = 512;
constexpr int DQ = DN + DR;     // query / key dims per head
constexpr int DL = DC + DR;     // latent row
// Blocks per cluster: 4.  With one block per SM, 36 clusters of 4 are
// resident on GB300 (144 SMs) but only 15 of 8, too few for one cluster per
// head in phase D.
constexpr int NCLU = 4;
constexpr int WPO = kConsumerWarps / NCLU;  // consumer warps whose heads a block owns
constexpr int DCB = DC / NCLU;              // latent rows of a block in phase D
constexpr int BMAX = 4;         // rows per call
constexpr int KT = 64;          // rows per projection tile
constexpr int GW = DQ;          // columns per projection group (192)
constexpr int RT = 32;          // latent rows per cache tile
constexpr int REC = DC + 4;     // state record: o_lat[512], m, l, 2 pad
constexpr int MAX_STAGES = 8;
constexpr int kMaxClusters = 64;  // resident clusters the phase-D merge handles
constexpr int STAGE_BYTES = RT * DL * 2;  // 36,864: the largest item (a cache tile)
static_assert(STAGE_BYTES == (DL / 64) * RT * 128 && RT % 16 == 0 && RT <= 32, "cache tile = nine swizzled boxes");
static_assert(KT * GW * 2 <= STAGE_BYTES && DC % KT == 0 && DCB * DV * 2 <= STAGE_BYTES &&
                  DV * 128 * 2 <= STAGE_BYTES && DCB % kConsumerWarps == 0, "stage plan");

struct Params {  // 128-byte aligned through its CUtensorMap members
  CUtensorMap tm_wq;    // [H, nh*DQ],  box {192, 64}
  CUtensorMap tm_wdkv;  // [H, DL],     box {192, 64}
  CUtensorMap tm_wukv;  // [DC, nh*(DN+DV)], box {128, 64}   (phase B: k parts)
  CUtensorMap tm_wuv;   // [DC, nh*(DN+DV)], box {128, DCB}  (phase D: v parts)
  CUtensorMap tm_wo;    // [nh*DV, H],  box {wob, DV}
  CUtensorMap tm_cache; // [B*S, DL] latent cache, box {64, RT}, 128-byte swizzle
  const void* hidden;   // [B, H]
  const void* ln_w;     // [H]
  const void* g_kv;     // [DC]
  void* cache;          // [B, S, DL]
  const int* positions; // [B]
  void* out;            // [B, H]
  float* y;             // [B][C1]   zero between launches
  float* qf;            // [B][nh][DL]: q_lat (512), rotated q rope part (64)
  float* lat;           // [B][DL]   the new latent row (fp32)
  float* part;          // [B][ncr_max][nh][REC] cluster partial states
  float* acc;           // [B][H]    zero between launches
  int* bar;             // [0] arrivals, [1] generation of the grid barrier
  int* tickets;         // [NCLU] per column band, zero between launches
  int* errflag;
  unsigned long long* timeline;  // optional [grid][kMlaTlSlots] globaltimer stamps (NULL = off)
  int B, H, nh, S;
  int ncl, nb;          // clusters, blocks
  int ncr_max;          // clusters per row, rounded up
  int stages;
  int wob;              // W_o box width (64 or 128)
  int off_bars, off_xs, off_scr, off_misc, off_sc;
  float eps;
  float qk_scale_log2;  // log2(e) / sqrt(DQ)
  float turn_hi[DR / 2], turn_lo[DR / 2];  // RoPE turn rates theta^(-2i/DR) / (2 pi)
};

__host__ __device__ inline int c1_cols(int nh) { return nh * DQ + DL; }

// Phase stamps of the optional timeline (a tuning aid; one row per block).
enum MlaTimelineSlot {
  kMlaTlStart = 0,      // after the start-up cluster barrier
  kMlaTlNorm = 1,       // consumers: dependency wait and x * ln_weight done
  kMlaTlA = 2,          // projection tiles consumed and flushed
  kMlaTlBar1 = 3,       // grid barrier 1 passed
  kMlaTlB = 4,          // absorption / latent row done
  kMlaTlBar2 = 5,       // grid barrier 2 passed
  kMlaTlC0 = 6,         // first cache tile in hand (or no tile)
  kMlaTlC1 = 7,         // cache tiles and the new row folded in
  kMlaTlC2 = 8,         // sparse ClusterReduce merged and written
  kMlaTlBar3 = 9,       // grid barrier 3 passed
  kMlaTlD0 = 10,        // w_uv product done
  kMlaTlD1 = 11,        // DSMEM all-reduce of o_h done
  kMlaTlD2 = 12,        // w_o product and atomics done
  kMlaTlEnd = 13,       // before the final cluster barrier
  kMlaTlProdA = 14,     // producer: projection tiles issued
  kMlaTlProdC = 15,     // producer: cache tiles issued
  kMlaTlProdD = 16,     // producer: everything issued
  kMlaTlSlots = 32
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *word != old (written by other blocks of this fully
// resident grid), with acquire semantics.  On expiry it records
// kDevErrTimeout and returns false.
static __device__ __noinline__ bool wait_word_changes(const int* word, int old, int* errflag) {
  const long long t0 = clock64();
  for (uint32_t spins = 1;; ++spins) {
    if (ld_acquire_gpu(word) != old) return true;
    if ((spins & 255u) == 0) {
      if (*reinterpret_cast<volatile int*>(errflag) & kDevErrTimeout) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        atomicOr(errflag, kDevErrTimeout);
        return false;
      }
    }
    __nanosleep(32);
  }
}

// Grid-wide barrier of the consumer threads (thread 0 of each block takes
// part, after a block barrier, so its release covers the block's writes).
// The arrival is an acquire-release add; the last arrival resets the count
// and publishes a new generation with a release add; the others wait for it
// with acquire loads.  `gen` is the generation this block last saw (thread 0
// only).
__device__ __forceinline__ void grid_sync(const Params& p, int& gen, int tid) {
  named_sync(kBarConsumers, kConsumers);
  if (tid == 0) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                 : "=r"(old) : "l"(&p.bar[0]) : "memory");
    if (old == p.nb - 1) {
      asm volatile("st.relaxed.gpu.global.s32 [%0], 0;" ::"l"(&p.bar[0]) : "memory");
      asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(&p.bar[1]) : "memory");
    } else {
      wait_word_changes(&p.bar[1], gen, p.errflag);
    }
    ++gen;
  }
  named_sync(kBarConsumers, kConsumers);
}

// Ranges of the work of block `blk`: projection tiles [t0, t1); and for
// phase C the row, the sub-chunk index and count.
struct Plan {
  int ta0, ta1;   // projection tiles
  int row, sidx, nsub;
};
__device__ __forceinline__ Plan plan_of(const Params& p, int blk) {
  Plan q;
  const int ta = (p.nh + DL / GW) * (p.H / KT);
  q.ta0 = (int)((long long)blk * ta / p.nb);
  q.ta1 = (int)((long long)(blk + 1) * ta / p.nb);
  const int cl = blk / NCLU, r = blk % NCLU;
  q.row = cl % p.B;
  const int ncr = (p.ncl - q.row + p.B - 1) / p.B;
  q.sidx = (cl / p.B) * NCLU + r;
  q.nsub = ncr * NCLU;
  return q;
}

// Cached positions [t0, t1) of sub-chunk sidx of nsub over positions 0..pos-1.
__device__ __forceinline__ void sub_range(int pos, int sidx, int nsub, int& t0, int& t1) {
  const int n = pos > 0 ? pos : 0;
  t0 = (int)((long long)sidx * n / nsub);
  t1 = (int)((long long)(sidx + 1) * n / nsub);
}


// ------------------------------------------------------------------ kernel --
// HPW: query heads per consumer warp (n_heads = 8 * HPW).
template <typename T, int HPW>
__global__ void __launch_bounds__(kThreads, 1) cf_mla_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int blk = blockIdx.x;
  const int rank = (int)cluster_ctarank();
  const int cl = blk / NCLU;
  const int B = p.B, H = p.H, nh = p.nh;
  const int C1 = c1_cols(nh);
  uint8_t* ring = sm;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + p.off_bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + MAX_STAGES;
  uint64_t* rx = bars + 2 * MAX_STAGES;        // phase C: incoming head states
  uint64_t* ga = bars + 2 * MAX_STAGES + 1;    // phase D: all-reduce rounds [3]
  float* xs = reinterpret_cast<float*>(sm + p.off_xs);    // [B][H] x * ln_weight
  float* scr = reinterpret_cast<float*>(sm + p.off_scr);  // phase scratch
  int* s_pos = reinterpret_cast<int*>(sm + p.off_misc);   // [BMAX]
  float* s_rinv = reinterpret_cast<float*>(s_pos + BMAX); // [BMAX]
  int* s_flag = reinterpret_cast<int*>(s_rinv + BMAX);    // [4]
  float* s_red = reinterpret_cast<float*>(s_flag + 4);    // [8] block reductions
  const Plan pl = plan_of(p, blk);
  const int ab = p.B * DV;  // floats of the phase-D all-reduce
  auto stamp = [&](int slot) {
    if (p.timeline != nullptr && (tid == 0 || (slot >= kMlaTlProdA && lane == 0)))
      p.timeline[(size_t)blk * kMlaTlSlots + slot] = globaltimer_ns();
  };

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(rx, 1);
    for (int r = 0; r < 3; ++r) mbar_init(&ga[r], 1);
    fence_mbar_init_cluster();
    mbar_arrive_expect_tx(rx, (uint32_t)(NCLU * WPO * HPW * REC * 4));
    for (int r = 0; (1 << r) < NCLU; ++r) mbar_arrive_expect_tx(&ga[r], allreduce_round_bytes(ab));
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tensormap(&p.tm_wq);
    prefetch_tensormap(&p.tm_wdkv);
    prefetch_tensormap(&p.tm_wukv);
    prefetch_tensormap(&p.tm_wuv);
    prefetch_tensormap(&p.tm_wo);
    prefetch_tensormap(&p.tm_cache);
  }
  __syncthreads();
  cluster_sync_all();  // peers' barriers exist before any DSMEM traffic
  stamp(kMlaTlStart);

  const int KTN = H / KT;
  if (warp == kConsumerWarps) {
    // ================================================== TMA producer ====
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      RingPos rp(0, p.stages);
      auto slot = [&](uint32_t bytes, uint64_t*& bar) -> uint8_t* {
        const int s = rp.slot;
        if (it >= p.stages) mbar_wait(&empty[s], rp.phase ^ 1u, p.errflag);
        bar = &full[s];
        mbar_arrive_expect_tx(bar, bytes);
        ++it;
        rp.next(p.stages);
        return ring + (size_t)s * STAGE_BYTES;
      };
      uint64_t* bar;
      // A: projection tiles (weights: needed nothing from earlier kernels)
      for (int t = pl.ta0; t < pl.ta1; ++t) {
        const int g = t / KTN, kt = t % KTN;
        uint8_t* dst = slot(KT * GW * 2, bar);
        if (g < nh) tma_load_2d(dst, &p.tm_wq, g * GW, kt * KT, bar, pol);
        else tma_load_2d(dst, &p.tm_wdkv, (g - nh) * GW, kt * KT, bar, pol);
      }
      // B: the k part of w_ukv for absorption item (h, 64-row band)
      for (int item = blk; item < nh * (DC / KT); item += p.nb) {
        const int h = item / (DC / KT), ib = item % (DC / KT);
        uint8_t* dst = slot(KT * DN * 2, bar);
        tma_load_2d(dst, &p.tm_wukv, h * (DN + DV), ib * KT, bar, pol);
      }
      stamp(kMlaTlProdA);
      // C: this block's cached latent rows (written by earlier steps)
      asm volatile("griddepcontrol.wait;" ::: "memory");
      {
        const int pos = p.positions[pl.row];
        const int posv = (pos >= 0 && pos < p.S) ? pos : 0;
        int t0, t1;
        sub_range(posv, pl.sidx, pl.nsub, t0, t1);
        // each tile: RT rows as nine 64-column boxes with the 128-byte
        // swizzle (rows past the range arrive too and are zeroed by the
        // consumers; rows past the tensor read as zero)
        for (int t = t0; t < t1; t += RT) {
          uint8_t* dst = slot((uint32_t)STAGE_BYTES, bar);
          for (int i = 0; i < DL / 64; ++i)
            tma_load_2d(dst + i * RT * 128, &p.tm_cache, 64 * i, pl.row * p.S + t, bar, pol);
        }
      }
      stamp(kMlaTlProdC);
      // D: w_uv rows of this block's latent band, then w_o of its column
      // band, box by box (both 64-row halves of each)
      for (int h = cl; h < nh; h += p.ncl) {
        uint8_t* dst = slot(DCB * DV * 2, bar);
        tma_load_2d(dst, &p.tm_wuv, h * (DN + DV) + DN, rank * DCB, bar, pol);
        const int cb = H / NCLU;
        for (int cx = 0; cx < cb / p.wob; ++cx) {
          dst = slot((uint32_t)(DV * p.wob * 2), bar);
          tma_load_2d(dst, &p.tm_wo, rank * cb + cx * p.wob, h * DV, bar, pol);
        }
      }
      stamp(kMlaTlProdD);
    }
    __syncwarp();
  } else {
    // ================================================== consumers =======
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int gen = 0;
    if (tid == 0) gen = *reinterpret_cast<volatile int*>(&p.bar[1]);
    if (tid < BMAX) {
      int pos = -1;
      if (tid < B) {
        pos = p.positions[tid];
        if (pos < 0 || pos >= p.S) {
          if (blk == 0) atomicOr(p.errflag, kDevErrPosRange);
          pos = -1;
        }
      }
      s_pos[tid] = pos;
    }
    // n = x * ln_weight (fp32) and the rows' sums of squares
    {
      const T* hid = static_cast<const T*>(p.hidden);
      const T* lw = static_cast<const T*>(p.ln_w);
      for (int b = 0; b < B; ++b) {
        float ss = 0.f;
        for (int i = tid * 8; i < H; i += kConsumers * 8) {
          float xv[8], gv[8];
          load_cvt<T, 8>(hid + (size_t)b * H + i, xv);
          load_cvt<T, 8>(lw + i, gv);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            ss = fmaf(xv[e], xv[e], ss);
            xs[b * H + i + e] = xv[e] * gv[e];
          }
        }
        ss = warp_sum(ss);
        if (lane == 0) s_red[warp] = ss;
        named_sync(kBarConsumers, kConsumers);
        if (tid == 0) {
          float tot = 0.f;
          for (int w = 0; w < kConsumerWarps; ++w) tot += s_red[w];
          s_rinv[b] = 1.0f / sqrtf(tot / (float)H + p.eps);
        }
        named_sync(kBarConsumers, kConsumers);
      }
    }
    stamp(kMlaTlNorm);
    int it = 0;
    RingPos rc(0, p.stages);  // ring slot and parity of use `it`
    // ---- A: projection partial sums ---------------------------------------
    {
      float acc[BMAX][6];
      auto zero = [&]() {
#pragma unroll
        for (int b = 0; b < BMAX; ++b)
#pragma unroll
          for (int e = 0; e < 6; ++e) acc[b][e] = 0.f;
      };
      // lane's columns of a 192-column group: 64 j + 2 lane + {0, 1}, j < 3
      auto flush = [&](int g) {
#pragma unroll
        for (int b = 0; b < BMAX; ++b)
          if (b < B)
#pragma unroll
            for (int j = 0; j < 3; ++j)
              *reinterpret_cast<float2*>(scr + (warp * B + b) * GW + 64 * j + 2 * lane) =
                  make_float2(acc[b][2 * j], acc[b][2 * j + 1]);
        named_sync(kBarConsumers, kConsumers);
        for (int idx = tid; idx < B * GW; idx += kConsumers) {
          const int b = idx / GW, c = idx % GW;
          float v = 0.f;
          for (int w = 0; w < kConsumerWarps; ++w) v += scr[(w * B + b) * GW + c];
          atomicAdd(p.y + (size_t)b * C1 + g * GW + c, v * s_rinv[b]);
        }
        named_sync(kBarConsumers, kConsumers);
        zero();
      };
      zero();
      int cur = -1;
      for (int t = pl.ta0; t < pl.ta1; ++t, ++it, rc.next(p.stages)) {
        const int g = t / KTN, kt = t % KTN;
        if (g != cur && cur >= 0) flush(cur);
        cur = g;
        const int s = rc.slot;
        mbar_wait(&full[s], rc.phase, p.errflag);
        const T* tile = reinterpret_cast<const T*>(ring + (size_t)s * STAGE_BYTES);
        for (int r = warp; r < KT; r += kConsumerWarps) {
          float nv[BMAX];
#pragma unroll
          for (int b = 0; b < BMAX; ++b) nv[b] = b < B ? xs[b * H + kt * KT + r] : 0.f;
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            float w2[2];
            load_cvt<T, 2>(tile + r * GW + 64 * j + 2 * lane, w2);
#pragma unroll
            for (int b = 0; b < BMAX; ++b) {
              acc[b][2 * j] = fmaf(nv[b], w2[0], acc[b][2 * j]);
              acc[b][2 * j + 1] = fmaf(nv[b], w2[1], acc[b][2 * j + 1]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      if (cur >= 0) flush(cur);
    }
    stamp(kMlaTlA);
    grid_sync(p, gen, tid);
    stamp(kMlaTlBar1);

    // ---- B: absorption, query RoPE, the latent row ------------------------
    for (int item = blk; item < nh * (DC / KT); item += p.nb, ++it, rc.next(p.stages)) {
      const int h = item / (DC / KT), ib = item % (DC / KT);
      float qn[BMAX][4];
#pragma unroll
      for (int b = 0; b < BMAX; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          qn[b][e] = b < B ? __ldcg(p.y + (size_t)b * C1 + h * DQ + 4 * lane + e) : 0.f;
      const int s = rc.slot;
      mbar_wait(&full[s], rc.phase, p.errflag);
      const T* tile = reinterpret_cast<const T*>(ring + (size_t)s * STAGE_BYTES);
#pragma unroll
      for (int rr = 0; rr < KT / kConsumerWarps; ++rr) {
        const int i = warp * (KT / kConsumerWarps) + rr;
        float w4[4];
        load_cvt<T, 4>(tile + i * DN + 4 * lane, w4);
#pragma unroll
        for (int b = 0; b < BMAX; ++b) {
          if (b >= B) continue;
          float v = w4[0] * qn[b][0] + w4[1] * qn[b][1] + w4[2] * qn[b][2] + w4[3] * qn[b][3];
          v = warp_sum(v);
          if (lane == 0) p.qf[((size_t)b * nh + h) * DL + ib * KT + i] = v;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (ib == 0) {
        // RoPE of head h's query position part [LNA §三 rotate_half]
        for (int idx = tid; idx < B * (DR / 2); idx += kConsumers) {
          const int b = idx / (DR / 2), j = idx % (DR / 2);
          const int pos = s_pos[b] >= 0 ? s_pos[b] : 0;
          const float* src = p.y + (size_t)b * C1 + h * DQ + DN;
          const float a = __ldcg(src + j), bb = __ldcg(src + j + DR / 2);
          float c, sn;
          rope_cos_sin(pos, p.turn_hi[j], p.turn_lo[j], c, sn);
          float* dst = p.qf + ((size_t)b * nh + h) * DL + DC;
          dst[j] = a * c - bb * sn;
          dst[j + DR / 2] = bb * c + a * sn;
        }
      }
    }
    if (blk >= p.nb - B) {
      // the latent row of batch row b: c' = RMSNorm(c; g_kv), RoPE(kr), append
      const int b = p.nb - 1 - blk;
      const float* src = p.y + (size_t)b * C1 + nh * DQ;
      const T* gk = static_cast<const T*>(p.g_kv);
      float cv[DC / kConsumers];
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < DC / kConsumers; ++e) {
        cv[e] = __ldcg(src + tid + e * kConsumers);
        ss = fmaf(cv[e], cv[e], ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) s_red[warp] = ss;
      named_sync(kBarConsumers, kConsumers);
      float tot = 0.f;
      for (int w = 0; w < kConsumerWarps; ++w) tot += s_red[w];
      const float r = 1.0f / sqrtf(tot / (float)DC + p.eps);
      const int pos = s_pos[b];
      T* slot = static_cast<T*>(p.cache) + ((size_t)b * p.S + (pos >= 0 ? pos : 0)) * DL;
#pragma unroll
      for (int e = 0; e < DC / kConsumers; ++e) {
        const int i = tid + e * kConsumers;
        const float v = cv[e] * r * Elem<T>::to_f(gk[i]);
        p.lat[(size_t)b * DL + i] = v;
        if (pos >= 0) slot[i] = Elem<T>::from_f(v);
      }
      if (tid < DR / 2) {
        const int j = tid;
        const float a = __ldcg(src + DC + j), bb = __ldcg(src + DC + j + DR / 2);
        float c, sn;
        rope_cos_sin(pos >= 0 ? pos : 0, p.turn_hi[j], p.turn_lo[j], c, sn);
        const float ra = a * c - bb * sn, rb = bb * c + a * sn;
        p.lat[(size_t)b * DL + DC + j] = ra;
        p.lat[(size_t)b * DL + DC + j + DR / 2] = rb;
        if (pos >= 0) {
          slot[DC + j] = Elem<T>::from_f(ra);
          slot[DC + j + DR / 2] = Elem<T>::from_f(rb);
        }
      }
      named_sync(kBarConsumers, kConsumers);
    }
    stamp(kMlaTlB);
    grid_sync(p, gen, tid);
    stamp(kMlaTlBar2);

    // ---- C: attention over this block's share of the latent cache ---------
    {
      // y is no longer read in this launch: clear it for the next one
      for (int i = blk * kConsumers + tid; i < B * C1; i += p.nb * kConsumers) p.y[i] = 0.f;
      const int b = pl.row;
      const int pos = s_pos[b];
      int t0, t1;
      sub_range(pos >= 0 ? pos : 0, pl.sidx, pl.nsub, t0, t1);
      const bool fold_new = pos >= 0 && pl.sidx == pl.nsub - 1;
      // Tensor-core form of the latent attention [CF §5.2].  The 16 query
      // rows (heads; rows nh..15 zero) are the MMAs' M side.  Warp w owns the
      // latent dims [64 w, 64 w + 64) -- slab w of a cache tile -- and, for
      // w < 4, the position dims [512 + 16 w, 512 + 16 w + 16) of slab 8:
      // (1) its partial scores q[:, its dims] c[t, its dims]^T for the RT
      // positions of a tile (A = the scaled query as 16-bit fragments held in
      // registers for the whole phase, B = the tile's rows), summed over the
      // warps in shared memory; (2) warp w's heads 2w, 2w+1 take the
      // online-softmax step (lane = position) and write p and the factor of
      // the running sums; (3) o[:, its dims] = alpha o + p c (A = p, B = slab
      // w, transposed by ldmatrix).  The query and p enter as one fp16 value
      // or as bf16 hi + lo pairs (about fp32 accuracy).
      using MK = MmaKind<T>;
      constexpr bool kHiLo = MK::kAttnHiLo;
      const int nks = warp < 4 ? 5 : 4;  // k-steps of this warp's share of the scores
      const int g = lane >> 2, cq = 2 * (lane & 3);
      uint32_t qh[5][4], ql[5][4];
      {
        const float* qb = p.qf + (size_t)b * nh * DL;
#pragma unroll
        for (int ks = 0; ks < 5; ++ks) {
          const int k0 = ks < 4 ? 64 * warp + 16 * ks : DC + 16 * warp;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            // fragment register e: row g (+8 for odd e), columns k0 + cq (+8 for e >= 2)
            const int r = g + 8 * (e & 1), k = k0 + cq + 8 * (e >> 1);
            float v0 = 0.f, v1 = 0.f;
            if (ks < nks && r < nh) {
              const float2 v = __ldcg(reinterpret_cast<const float2*>(qb + (size_t)r * DL + k));
              v0 = v.x * p.qk_scale_log2;
              v1 = v.y * p.qk_scale_log2;
            }
            MK::split2(v0, v1, qh[ks][e], ql[ks][e]);
          }
        }
      }
      float o[8][4];
#pragma unroll
      for (int nb = 0; nb < 8; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[nb][e] = 0.f;
      float m2[2] = {-INFINITY, -INFINITY}, l2[2] = {0.f, 0.f};  // heads 2 warp + j
      float* sS = reinterpret_cast<float*>(sm + p.off_sc);         // [8][16][RT] partial scores
      T* sPh = reinterpret_cast<T*>(sS + kConsumerWarps * 16 * RT);  // [16][RT + 8] p (hi)
      T* sPl = sPh + 16 * (RT + 8);                                  // [16][RT + 8] p (lo)
      float* sAl = reinterpret_cast<float*>(sPl + 16 * (RT + 8));     // [16] factors
      float* sPn = sAl + 16;                                          // [16] p of the new row
      constexpr int PP = (RT + 8) * 2;  // p row pitch in bytes (not a multiple of 128)
      for (int tt = t0; tt < t1; tt += RT, ++it, rc.next(p.stages)) {
        const int n = min(RT, t1 - tt);
        const int s = rc.slot;
        mbar_wait(&full[s], rc.phase, p.errflag);
        if (tt == t0) stamp(kMlaTlC0);
        uint8_t* tile = ring + (size_t)s * STAGE_BYTES;  // [DL / 64][RT][64], 128-byte swizzle
        if (n < RT) {
          // rows past the range (later positions, another row's cache or the
          // zero fill) must not reach the sums: zero them
          const int zr = (RT - n) * 8;  // 16-byte chunks per slab
          for (int i = tid; i < (DL / 64) * zr; i += kConsumers) {
            const int sl = i / zr, w = i - sl * zr;
            *reinterpret_cast<uint4*>(tile + sl * RT * 128 + (n + w / 8) * 128 + (w % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();  // before the stage goes back to the TMA writes
          named_sync(kBarConsumers, kConsumers);
        }
        // (1) partial scores of this warp's dims
        {
          float acc[4][4];
#pragma unroll
          for (int nb = 0; nb < 4; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nb][e] = 0.f;
#pragma unroll
          for (int ks = 0; ks < 5; ++ks) {
            if (ks < nks) {
              const uint8_t* slab = tile + (ks < 4 ? warp : DC / 64) * (RT * 128);
              const int k0 = ks < 4 ? 16 * ks : 16 * warp;  // column within the slab
#pragma unroll
              for (int nb = 0; nb < RT / 8; ++nb) {
                uint32_t b0, b1;
                ldmatrix_bt_sw128(b0, b1, slab, 8 * nb, k0, lane);
                MK::mma(acc[nb], qh[ks], b0, b1);
                if constexpr (kHiLo) MK::mma(acc[nb], ql[ks], b0, b1);
              }
            }
          }
          float* dst = sS + warp * 16 * RT;
#pragma unroll
          for (int nb = 0; nb < RT / 8; ++nb) {
            *reinterpret_cast<float2*>(dst + g * RT + 8 * nb + cq) = make_float2(acc[nb][0], acc[nb][1]);
            *reinterpret_cast<float2*>(dst + (g + 8) * RT + 8 * nb + cq) =
                make_float2(acc[nb][2], acc[nb][3]);
          }
        }
        named_sync(kBarConsumers, kConsumers);
        // (2) online softmax of heads 2 warp + j over the tile
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int h = 2 * warp + j;
          float sc = -INFINITY;
          if (h < nh && lane < n) {
            sc = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) sc += sS[(w * 16 + h) * RT + lane];
          }
          float mt = sc;
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
          const float mn = fmaxf(m2[j], mt);
          const float alpha = mn == -INFINITY ? 1.f : exp2f(m2[j] - mn);
          const float pr = sc == -INFINITY ? 0.f : exp2f(sc - mn);
          float ps = pr;
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
          l2[j] = l2[j] * alpha + ps;
          m2[j] = mn;
          const T phv = Elem<T>::from_f(pr);
          sPh[h * (RT + 8) + lane] = phv;
          if constexpr (kHiLo) sPl[h * (RT + 8) + lane] = Elem<T>::from_f(pr - Elem<T>::to_f(phv));
          if (lane == 0) sAl[h] = alpha;
        }
        named_sync(kBarConsumers, kConsumers);
        // (3) o = alpha o + p c over this warp's 64 latent dims
        {
          const float a0 = sAl[g], a1 = sAl[g + 8];
#pragma unroll
          for (int nb = 0; nb < 8; ++nb) {
            o[nb][0] *= a0;
            o[nb][1] *= a0;
            o[nb][2] *= a1;
            o[nb][3] *= a1;
          }
          const uint8_t* slab = tile + warp * (RT * 128);
#pragma unroll
          for (int ks = 0; ks < RT / 16; ++ks) {
            uint32_t pa[4], pb[4];
            ldmatrix_a(pa, sPh + 16 * ks, PP, lane);
            if constexpr (kHiLo) ldmatrix_a(pb, sPl + 16 * ks, PP, lane);
#pragma unroll
            for (int nb = 0; nb < 8; ++nb) {
              uint32_t b0, b1;
              ldmatrix_b_sw128(b0, b1, slab, 16 * ks, 8 * nb, lane);
              MK::mma(o[nb], pa, b0, b1);
              if constexpr (kHiLo) MK::mma(o[nb], pb, b0, b1);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      if (fold_new) {
        // the new row (fp32, not yet rounded): its scores, the softmax step
        // and its term in o, on the CUDA cores
        named_sync(kBarConsumers, kConsumers);  // every warp is done with sAl
        const float* nl = p.lat + (size_t)b * DL;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int h = 2 * warp + j;
          float sc = 0.f;
          if (h < nh) {
            const float* qr = p.qf + ((size_t)b * nh + h) * DL;
            for (int d = lane; d < DL; d += 32) sc = fmaf(__ldcg(qr + d), __ldcg(nl + d), sc);
          }
          sc = warp_sum(sc) * p.qk_scale_log2;
          float alpha = 1.f, pn = 0.f;
          if (h < nh) {
            const float mn = fmaxf(m2[j], sc);
            alpha = exp2f(m2[j] - mn);
            pn = exp2f(sc - mn);
            l2[j] = l2[j] * alpha + pn;
            m2[j] = mn;
          }
          if (lane == 0) {
            sAl[h] = alpha;
            sPn[h] = pn;
          }
        }
        named_sync(kBarConsumers, kConsumers);
        const float a0 = sAl[g], a1 = sAl[g + 8], p0 = sPn[g], p1 = sPn[g + 8];
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
          const float2 c2 = __ldcg(reinterpret_cast<const float2*>(nl + 64 * warp + 8 * nb + cq));
          o[nb][0] = fmaf(p0, c2.x, o[nb][0] * a0);
          o[nb][1] = fmaf(p0, c2.y, o[nb][1] * a0);
          o[nb][2] = fmaf(p1, c2.x, o[nb][2] * a1);
          o[nb][3] = fmaf(p1, c2.y, o[nb][3] * a1);
        }
      }
      // sparse ClusterReduce: head h's state goes only to the cluster block
      // that owns it, block (h % 8) % NCLU, into slot
      // [rank][((h % 8) / NCLU) * HPW + h / 8] there; each warp sends its 64
      // dims of every head, lane 0 of warp w the (m, l) of heads 2w, 2w+1
      {
        float* rbuf = scr;  // [NCLU][WPO * HPW][REC]
        auto record = [&](int h, uint32_t& raddr, uint32_t& rbar) {
          const uint32_t owner = (uint32_t)((h % kConsumerWarps) % NCLU);
          const int j = ((h % kConsumerWarps) / NCLU) * HPW + h / kConsumerWarps;
          raddr = mapa(smem_u32(rbuf + ((size_t)rank * WPO * HPW + j) * REC), owner);
          rbar = mapa(smem_u32(rx), owner);
        };
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int h = g + 8 * hf;
          if (h < nh) {
            uint32_t raddr, rbar;
            record(h, raddr, rbar);
#pragma unroll
            for (int nb = 0; nb < 8; ++nb)
              st_async_v2(raddr + 4u * (64 * warp + 8 * nb + cq),
                          make_float2(o[nb][2 * hf], o[nb][2 * hf + 1]), rbar);
          }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int h = 2 * warp + j;
          if (h < nh && lane == 0) {
            uint32_t raddr, rbar;
            record(h, raddr, rbar);
            st_async_v4(raddr + 4u * DC, make_float4(m2[j], l2[j], 0.f, 0.f), rbar);
          }
        }
        stamp(kMlaTlC1);
        mbar_wait_cluster(rx, 0, p.errflag);
        // merge the NCLU states of each owned head: slot j = (w / NCLU) * HPW
        // + k holds head h = w + 8k of warp w = rank + NCLU * (j / HPW); the
        // slot's maximum and the sources' factors 2^(m_src - max) first
        const int ci = pl.sidx / NCLU;
        constexpr int JPB = WPO * HPW;
        float* sf = sS;  // [JPB][NCLU + 1]: factors, then the maximum
        if (tid < JPB) {
          float mm = -INFINITY;
          for (int src = 0; src < NCLU; ++src)
            mm = fmaxf(mm, rbuf[((size_t)src * JPB + tid) * REC + DC]);
          for (int src = 0; src < NCLU; ++src)
            sf[tid * (NCLU + 1) + src] =
                mm == -INFINITY ? 0.f : exp2f(rbuf[((size_t)src * JPB + tid) * REC + DC] - mm);
          sf[tid * (NCLU + 1) + NCLU] = mm;
        }
        named_sync(kBarConsumers, kConsumers);
        for (int idx = tid; idx < JPB * (DC + 2); idx += kConsumers) {
          const int j = idx / (DC + 2), e = idx % (DC + 2);
          float v = 0.f;
          if (e == DC) {
            v = sf[j * (NCLU + 1) + NCLU];
          } else {
            const int ee = e < DC ? e : DC + 1;
#pragma unroll
            for (int src = 0; src < NCLU; ++src)
              v = fmaf(rbuf[((size_t)src * JPB + j) * REC + ee], sf[j * (NCLU + 1) + src], v);
          }
          const int h = rank + NCLU * (j / HPW) + kConsumerWarps * (j % HPW);
          float* dst = p.part + (((size_t)b * p.ncr_max + ci) * nh + h) * REC;
          dst[e < DC ? e : (e == DC ? DC : DC + 1)] = v;
        }
      }
    }
    stamp(kMlaTlC2);
    grid_sync(p, gen, tid);
    stamp(kMlaTlBar3);

    // ---- D: per head: merge, w_uv, w_o, residual --------------------------
    {
      const int cb = H / NCLU;        // this block's output columns
      float* ol = scr;                          // [B][DCB] this block's o_lat rows
      float* red = ol + BMAX * DCB;             // [8][B][max(DV, wob)] warp partials
      float* ov = red + kConsumerWarps * BMAX * max(DV, p.wob);  // [B][DV]
      float* rb = ov + BMAX * DV;               // [log2 NCLU][B][DV] all-reduce receive
      const int cpl = p.wob / 32;               // w_o columns per lane (2 or 4)
      for (int h = cl; h < nh; h += p.ncl) {
        // merge of the row's cluster partials: warp b computes row b's
        // per-cluster factors 2^(m_c - M) / L into s_mf, then every thread
        // sums its latent rows over the clusters with independent loads
        float* s_mf = s_red + 8;  // [BMAX][kMaxClusters]
        if (warp < B) {
          const int b = warp;
          const int ncr = (p.ncl - b + B - 1) / B;
          float mc[kMaxClusters / 32], lc[kMaxClusters / 32];
          float mm = -INFINITY;
#pragma unroll
          for (int q = 0; q < kMaxClusters / 32; ++q) {
            const int c = lane + 32 * q;
            const float* ps = p.part + (((size_t)b * p.ncr_max + c) * nh + h) * REC;
            mc[q] = c < ncr ? __ldcg(ps + DC) : -INFINITY;
            lc[q] = c < ncr ? __ldcg(ps + DC + 1) : 0.f;
            mm = fmaxf(mm, mc[q]);
          }
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
          float L = 0.f, f[kMaxClusters / 32];
#pragma unroll
          for (int q = 0; q < kMaxClusters / 32; ++q) {
            f[q] = mm == -INFINITY ? 0.f : exp2f(mc[q] - mm);
            L = fmaf(lc[q], f[q], L);
          }
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
#pragma unroll
          for (int q = 0; q < kMaxClusters / 32; ++q)
            s_mf[b * kMaxClusters + lane + 32 * q] = L > 0.f ? f[q] / L : 0.f;
        }
        named_sync(kBarConsumers, kConsumers);
        {
          // with fewer (row, latent row) items than threads, SP threads share
          // an item's clusters; eight loads in flight per thread
          const int items = B * DCB;
          const int SP = items >= kConsumers ? 1 : kConsumers / items;
          float* half = red;  // [SP][items] partial sums
          for (int t = tid; t < items * SP; t += kConsumers) {
            const int idx = t % items, sp = t / items;
            const int b = idx / DCB, i = rank * DCB + idx % DCB;
            const int ncr = (p.ncl - b + B - 1) / B;
            const float* ps = p.part + ((size_t)b * p.ncr_max * nh + h) * REC + i;
            const size_t cstride = (size_t)nh * REC;
            float v0 = 0.f, v1 = 0.f;
            for (int c0 = sp; c0 < ncr; c0 += 8 * SP) {
              float x[8], f[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int c = c0 + k * SP;
                x[k] = c < ncr ? __ldcg(ps + c * cstride) : 0.f;
                f[k] = c < ncr ? s_mf[b * kMaxClusters + c] : 0.f;
              }
#pragma unroll
              for (int k = 0; k < 8; k += 2) {
                v0 = fmaf(x[k], f[k], v0);
                v1 = fmaf(x[k + 1], f[k + 1], v1);
              }
            }
            if (SP == 1) ol[idx] = v0 + v1;
            else half[sp * items + idx] = v0 + v1;
          }
          if (SP > 1) {
            named_sync(kBarConsumers, kConsumers);
            for (int idx = tid; idx < items; idx += kConsumers) {
              float v = 0.f;
              for (int sp = 0; sp < SP; ++sp) v += half[sp * items + idx];
              ol[idx] = v;
            }
          }
        }
        named_sync(kBarConsumers, kConsumers);
        // o_h partial over the block's latent rows, 64 per w_uv box: warp w
        // rows 8w..8w+7 of each box, lane columns 4l..4l+3
        {
          float a4[BMAX][4];
#pragma unroll
          for (int b = 0; b < BMAX; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) a4[b][e] = 0.f;
          {
            const int s = rc.slot;
            mbar_wait(&full[s], rc.phase, p.errflag);
            const T* tile = reinterpret_cast<const T*>(ring + (size_t)s * STAGE_BYTES);
#pragma unroll 4
            for (int rr = 0; rr < DCB / kConsumerWarps; ++rr) {
              const int i = warp * (DCB / kConsumerWarps) + rr;
              float w4[4];
              load_cvt<T, 4>(tile + i * DV + 4 * lane, w4);
#pragma unroll
              for (int b = 0; b < BMAX; ++b) {
                if (b >= B) continue;
                const float ov1 = ol[b * DCB + i];
#pragma unroll
                for (int e = 0; e < 4; ++e) a4[b][e] = fmaf(ov1, w4[e], a4[b][e]);
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++it;
            rc.next(p.stages);
          }
#pragma unroll
          for (int b = 0; b < BMAX; ++b)
            if (b < B)
              *reinterpret_cast<float4*>(red + (warp * B + b) * DV + 4 * lane) =
                  make_float4(a4[b][0], a4[b][1], a4[b][2], a4[b][3]);
          named_sync(kBarConsumers, kConsumers);
          for (int idx = tid; idx < B * DV; idx += kConsumers) {
            float v = 0.f;
            for (int w = 0; w < kConsumerWarps; ++w) v += red[w * B * DV + idx];
            ov[idx] = v;
          }
          named_sync(kBarConsumers, kConsumers);
        }
        stamp(kMlaTlD0);
        // o_h = sum over the cluster's latent bands [CF §3.1.1]
        cluster_allreduce<OpSum, kConsumers, kBarConsumers>(ov, ab, rb, ga, rank, NCLU, tid,
                                                            p.errflag);
        stamp(kMlaTlD1);
        // w_o rows h*DV.. of this block's column band, one box of wob columns
        // at a time (both 64-row halves), then its cross-warp sum and fp32
        // atomics into the accumulator [CF §3.2 原子写合并]
        for (int cx = 0; cx < cb / p.wob; ++cx) {
          float a[BMAX][4];
#pragma unroll
          for (int b = 0; b < BMAX; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) a[b][e] = 0.f;
          {
            const int s = rc.slot;
            mbar_wait(&full[s], rc.phase, p.errflag);
            const T* tile = reinterpret_cast<const T*>(ring + (size_t)s * STAGE_BYTES);
#pragma unroll 4
            for (int rr = 0; rr < DV / kConsumerWarps; ++rr) {
              const int j = warp * (DV / kConsumerWarps) + rr;
              float w[4] = {0.f, 0.f, 0.f, 0.f};
              if (cpl == 4) load_cvt<T, 4>(tile + j * p.wob + 4 * lane, w);
              else load_cvt<T, 2>(tile + j * p.wob + 2 * lane, w);
#pragma unroll
              for (int b = 0; b < BMAX; ++b) {
                if (b >= B) continue;
                const float ovj = ov[b * DV + j];
#pragma unroll
                for (int e = 0; e < 4; ++e) a[b][e] = fmaf(ovj, w[e], a[b][e]);
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++it;
            rc.next(p.stages);
          }
#pragma unroll
          for (int b = 0; b < BMAX; ++b)
            if (b < B)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (e < cpl) red[(warp * B + b) * p.wob + cpl * lane + e] = a[b][e];
          named_sync(kBarConsumers, kConsumers);
          for (int idx = tid; idx < B * p.wob; idx += kConsumers) {
            const int b = idx / p.wob, c = idx % p.wob;
            float v = 0.f;
            for (int w = 0; w < kConsumerWarps; ++w) v += red[(w * B + b) * p.wob + c];
            if (s_pos[b] >= 0) atomicAdd(p.acc + (size_t)b * H + rank * cb + cx * p.wob + c, v);
          }
          named_sync(kBarConsumers, kConsumers);
        }
        stamp(kMlaTlD2);
        __threadfence();
        named_sync(kBarConsumers, kConsumers);
        if (tid == 0) {
          const int last = atomicAdd(&p.tickets[rank], 1) == nh - 1;
          if (last) __threadfence();
          s_flag[0] = last;
        }
        named_sync(kBarConsumers, kConsumers);
        if (s_flag[0]) {
          // residual of the column band [LNA §一]
          const T* hid = static_cast<const T*>(p.hidden);
          T* out = static_cast<T*>(p.out);
          for (int idx = tid; idx < B * (cb / 4); idx += kConsumers) {
            const int b = idx / (cb / 4), c4 = idx % (cb / 4);
            const size_t off = (size_t)b * H + rank * cb + 4 * c4;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p.acc + off));
            __stcg(reinterpret_cast<float4*>(p.acc + off), make_float4(0.f, 0.f, 0.f, 0.f));
            float xv[4];
            load_cvt<T, 4>(hid + off, xv);
            const float r4[4] = {xv[0] + v.x, xv[1] + v.y, xv[2] + v.z, xv[3] + v.w};
            store4<T>(out + off, r4);
          }
          if (tid == 0) p.tickets[rank] = 0;
        }
        named_sync(kBarConsumers, kConsumers);
      }
    }
  }
  stamp(kMlaTlEnd);
  // no block leaves while a peer may still write into its shared memory
  __syncwarp();
  cluster_sync_exit();
}

// Dynamic shared memory of a plan (bytes past the 1024-aligned base).
struct Layout {
  int bars, xs, scr, misc, sc, total;
};
inline Layout layout_for(int stages, int max_batch, int H, int nh) {
  auto r128 = [](int v) { return (v + 127) / 128 * 128; };
  Layout L;
  int off = stages * STAGE_BYTES;
  L.bars = off;
  off += r128((2 * MAX_STAGES + 4) * 8);
  L.xs = off;
  off += r128(max_batch * H * 4);
  L.scr = off;
  const int hpw = nh / kConsumerWarps;
  const int cb = H / NCLU;
  const int scrA = kConsumerWarps * max_batch * GW;
  const int scrC = NCLU * WPO * hpw * REC;
  const int wob = cb % 128 == 0 ? 128 : 64;
  const int scrD = BMAX * DCB + kConsumerWarps * BMAX * std::max(DV, wob) + BMAX * DV +
                   3 * BMAX * DV;
  off += r128(4 * std::max(scrA, std::max(scrC, scrD)));
  L.misc = off;
  off += r128(4 * (2 * BMAX + 4 + 8 + BMAX * kMaxClusters));
  L.sc = off;
  // phase C: partial scores [8][16][RT] fp32, p hi and lo [16][RT + 8], factors [16], new-row p [16]
  off += r128(4 * kConsumerWarps * 16 * RT + 2 * 2 * 16 * (RT + 8) + 2 * 16 * 4);
  L.total = off + 1024;
  return L;
}

}  // namespace mla
}  // namespace cf

using namespace cf;
using namespace cf::mla;

struct cf_mla_handle {
  cf_mla_config cfg;
  int device = 0;
  int ncl = 0, nb = 0, stages = 0, wob = 128, ncr_max = 0;
  Layout L;
  const void* fn = nullptr;
  void* ws = nullptr;
  float *y = nullptr, *qf = nullptr, *lat = nullptr, *part = nullptr, *acc = nullptr;
  int *bar = nullptr, *tickets = nullptr, *errflag = nullptr;
  unsigned long long* timeline = nullptr;
  float turn_hi[DR / 2], turn_lo[DR / 2];
  struct MapSlot {
    const void* ptr = nullptr;
    CUtensorMap map;
  } m_wq, m_wdkv, m_wukv, m_wuv, m_wo;
  // latent cache [batch * S, DL] with the 128-byte swizzle, for the batch it was encoded for
  MapSlot m_cache;
  int cache_batch = 0;
};

namespace {

int resident_mla_clusters(const void* fn, int smem) {
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NCLU;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(NCLU, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.attrs = attr;
  lc.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &lc) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

const CUtensorMap* mla_map(cf_mla_handle::MapSlot& s, int dtype, const void* ptr, uint64_t inner,
                           uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  if (s.ptr != ptr) {
    s.ptr = nullptr;
    if (!encode_tmap_2d(&s.map, dtype, ptr, inner, outer, inner * 2, box_inner, box_outer, false))
      return nullptr;
    s.ptr = ptr;
  }
  return &s.map;
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" {

int cf_mla_create(const cf_mla_config* cfg, cf_mla_handle** out) {
  if (out == nullptr) return CF_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg == nullptr) return CF_ERR_INVALID_ARG;
  const cf_mla_config c = *cfg;
  if (c.hidden <= 0 || c.n_heads <= 0 || c.max_batch <= 0 || c.s_max <= 0 || c.d_nope <= 0 ||
      c.d_rope <= 0 || c.d_v <= 0 || c.d_latent <= 0)
    return CF_ERR_INVALID_ARG;
  if (!(c.rope_theta > 0.f) || !std::isfinite(c.rope_theta) || !(c.rms_eps >= 0.f) ||
      !std::isfinite(c.rms_eps))
    return CF_ERR_INVALID_ARG;
  if (c.dtype < CF_F32 || c.dtype > CF_BF16) return CF_ERR_INVALID_ARG;
  if (c.d_nope != DN || c.d_rope != DR || c.d_v != DV || c.d_latent != DC)
    return CF_ERR_UNSUPPORTED;
  if (c.dtype == CF_F32) return CF_ERR_UNSUPPORTED;
  {
    const int hpw = c.n_heads / kConsumerWarps;
    // 8 or 16 heads: one or two per consumer warp (and one cluster per head
    // in the last phase)
    if (c.n_heads % kConsumerWarps != 0 || !(hpw == 1 || hpw == 2)) return CF_ERR_UNSUPPORTED;
  }
  // column bands of the output projection: H / NCLU columns per block in
  // TMA boxes of 64 or 128 columns; the hidden state as 8-element vectors
  if (c.hidden % (NCLU * 64) != 0 || c.hidden > 16384) return CF_ERR_UNSUPPORTED;
  if (c.max_batch > BMAX) return CF_ERR_UNSUPPORTED;
  cf_mla_handle* h = new (std::nothrow) cf_mla_handle();
  if (h == nullptr) return CF_ERR_CUDA;
  h->cfg = c;
  auto fail = [&](int rc) {
    if (h->ws) cudaFree(h->ws);
    delete h;
    return rc;
  };
  if (cudaGetDevice(&h->device) != cudaSuccess) return fail(CF_ERR_CUDA);
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, h->device) != cudaSuccess) return fail(CF_ERR_CUDA);
  {
    const int hpw = c.n_heads / kConsumerWarps;
    const bool f16 = c.dtype == CF_F16;
    h->fn = hpw == 1 ? (f16 ? (const void*)&cf_mla_kernel<__half, 1>
                            : (const void*)&cf_mla_kernel<__nv_bfloat16, 1>)
                     : (f16 ? (const void*)&cf_mla_kernel<__half, 2>
                            : (const void*)&cf_mla_kernel<__nv_bfloat16, 2>);
  }
  h->wob = (c.hidden / NCLU) % 128 == 0 ? 128 : 64;
  const int budget = (int)prop.sharedMemPerBlockOptin;
  int stages = MAX_STAGES;
  for (; stages >= 2; --stages)
    if (layout_for(stages, c.max_batch, c.hidden, c.n_heads).total <= budget) break;
  if (stages < 2) return fail(CF_ERR_UNSUPPORTED);
  h->stages = stages;
  h->L = layout_for(stages, c.max_batch, c.hidden, c.n_heads);
  if (cudaFuncSetAttribute(h->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, h->L.total) !=
      cudaSuccess) {
    cudaGetLastError();
    return fail(CF_ERR_CUDA);
  }
  h->ncl = resident_mla_clusters(h->fn, h->L.total);
  // one cluster per head in the last phase, at least one per batch row
  if (h->ncl < c.n_heads || h->ncl < c.max_batch) return fail(CF_ERR_CLUSTER);
  h->ncl = std::min(h->ncl, kMaxClusters);
  h->nb = h->ncl * NCLU;
  // rows share the clusters (row b gets ceil((ncl - b) / batch)); sized for
  // a one-row call, which gives one row every cluster
  h->ncr_max = h->ncl;
  const int H = c.hidden, nh = c.n_heads, MB = c.max_batch;
  const size_t y_f = (size_t)MB * c1_cols(nh);
  const size_t qf_f = (size_t)MB * nh * DL;
  const size_t lat_f = (size_t)MB * DL;
  const size_t part_f = (size_t)MB * h->ncr_max * nh * REC;
  const size_t acc_f = (size_t)MB * H;
  const size_t floats = y_f + qf_f + lat_f + part_f + acc_f;
  const size_t ints = 2 + NCLU + 2;
  const size_t bytes = floats * 4 + ints * 4 + 256;
  if (cudaMalloc(&h->ws, bytes) != cudaSuccess) {
    h->ws = nullptr;
    return fail(CF_ERR_CUDA);
  }
  if (cudaMemset(h->ws, 0, bytes) != cudaSuccess) return fail(CF_ERR_CUDA);
  float* f = static_cast<float*>(h->ws);
  h->y = f;
  h->qf = h->y + y_f;
  h->lat = h->qf + qf_f;
  h->part = h->lat + lat_f;
  h->acc = h->part + part_f;
  int* ip = reinterpret_cast<int*>(h->acc + acc_f);
  h->bar = ip;
  h->tickets = ip + 2;
  h->errflag = ip + 2 + NCLU;
  for (int i = 0; i < DR / 2; ++i) {
    const double two_pi = 6.283185307179586476925286766559;
    const double rate = std::pow((double)c.rope_theta, -2.0 * i / (double)DR) / two_pi;
    h->turn_hi[i] = (float)rate;
    h->turn_lo[i] = (float)(rate - (double)h->turn_hi[i]);
  }
  *out = h;
  return CF_OK;
}

int cf_mla_decode(cf_mla_handle* h, int32_t batch, const void* hidden_states,
                  const void* ln_weight, const void* w_q, const void* w_dkv,
                  const void* kv_norm_weight, const void* w_ukv, const void* w_o,
                  void* latent_cache, const int32_t* positions, void* out, void* stream) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  const cf_mla_config& c = h->cfg;
  if (batch < 0 || batch > c.max_batch) return CF_ERR_INVALID_ARG;
  if (batch == 0) return CF_OK;
  const void* ptrs[] = {hidden_states, ln_weight, w_q,      w_dkv,    kv_norm_weight,
                        w_ukv,         w_o,       latent_cache, positions, out};
  for (const void* q : ptrs)
    if (q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u) != 0) return CF_ERR_INVALID_ARG;
  const int H = c.hidden, nh = c.n_heads, S = c.s_max;
  const size_t es = 2;
  const size_t ob = (size_t)batch * H * es;
  if (ranges_overlap(out, ob, hidden_states, ob) || ranges_overlap(out, ob, ln_weight, H * es) ||
      ranges_overlap(out, ob, w_q, (size_t)H * nh * DQ * es) ||
      ranges_overlap(out, ob, w_dkv, (size_t)H * DL * es) ||
      ranges_overlap(out, ob, kv_norm_weight, DC * es) ||
      ranges_overlap(out, ob, w_ukv, (size_t)DC * nh * (DN + DV) * es) ||
      ranges_overlap(out, ob, w_o, (size_t)nh * DV * H * es) ||
      ranges_overlap(out, ob, latent_cache, (size_t)batch * S * DL * es) ||
      ranges_overlap(out, ob, positions, (size_t)batch * 4))
    return CF_ERR_ALIAS;
  Params p;
  std::memset(&p, 0, sizeof(p));
  const CUtensorMap* m1 = mla_map(h->m_wq, c.dtype, w_q, (uint64_t)nh * DQ, H, GW, KT);
  const CUtensorMap* m2 = mla_map(h->m_wdkv, c.dtype, w_dkv, DL, H, GW, KT);
  const CUtensorMap* m3 = mla_map(h->m_wukv, c.dtype, w_ukv, (uint64_t)nh * (DN + DV), DC, 128, KT);
  const CUtensorMap* m5 = mla_map(h->m_wuv, c.dtype, w_ukv, (uint64_t)nh * (DN + DV), DC, 128, DCB);
  const CUtensorMap* m4 = mla_map(h->m_wo, c.dtype, w_o, H, (uint64_t)nh * DV, h->wob, DV);
  if (!m1 || !m2 || !m3 || !m4 || !m5) return CF_ERR_CUDA;
  p.tm_wq = *m1;
  p.tm_wdkv = *m2;
  p.tm_wukv = *m3;
  p.tm_wuv = *m5;
  p.tm_wo = *m4;
  if (h->m_cache.ptr != latent_cache || h->cache_batch != batch) {
    h->m_cache.ptr = nullptr;
    if (!encode_tmap_2d(&h->m_cache.map, c.dtype, latent_cache, DL, (uint64_t)batch * S, DL * 2,
                        64, RT, true))
      return CF_ERR_CUDA;
    h->m_cache.ptr = latent_cache;
    h->cache_batch = batch;
  }
  p.tm_cache = h->m_cache.map;
  p.hidden = hidden_states;
  p.ln_w = ln_weight;
  p.g_kv = kv_norm_weight;
  p.cache = latent_cache;
  p.positions = positions;
  p.out = out;
  p.y = h->y;
  p.qf = h->qf;
  p.lat = h->lat;
  p.part = h->part;
  p.acc = h->acc;
  p.bar = h->bar;
  p.tickets = h->tickets;
  p.errflag = h->errflag;
  p.timeline = h->timeline;
  p.B = batch;
  p.H = H;
  p.nh = nh;
  p.S = S;
  p.ncl = h->ncl;
  p.nb = h->nb;
  p.ncr_max = h->ncr_max;
  p.stages = h->stages;
  p.wob = h->wob;
  p.off_bars = h->L.bars;
  p.off_xs = h->L.xs;
  p.off_scr = h->L.scr;
  p.off_misc = h->L.misc;
  p.off_sc = h->L.sc;
  p.eps = c.rms_eps;
  p.qk_scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)DQ));
  for (int i = 0; i < DR / 2; ++i) {
    p.turn_hi[i] = h->turn_hi[i];
    p.turn_lo[i] = h->turn_lo[i];
  }
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NCLU;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = dim3(h->nb, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = h->L.total;
  lc.stream = static_cast<cudaStream_t>(stream);
  lc.attrs = attr;
  lc.numAttrs = 2;
  void* args[] = {&p};
  if (cudaLaunchKernelExC(&lc, h->fn, args) != cudaSuccess) {
    cudaGetLastError();
    return CF_ERR_CUDA;
  }
  return CF_OK;
}

int cf_mla_get_status(cf_mla_handle* h) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  int flag = 0;
  if (cudaMemcpy(&flag, h->errflag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CF_ERR_CUDA;
  if (flag != 0 && cudaMemset(h->errflag, 0, sizeof(int)) != cudaSuccess) return CF_ERR_CUDA;
  if (flag & kDevErrTimeout) return CF_ERR_DEVICE_TIMEOUT;
  if (flag & kDevErrPosRange) return CF_ERR_DEVICE_POS_RANGE;
  return CF_OK;
}

int cf_mla_launch_info(const cf_mla_handle* h, int32_t* clusters, int32_t* cluster_size,
                       int32_t* stages, int32_t* stage_bytes, int32_t* smem_bytes) {
  if (h == nullptr || clusters == nullptr || cluster_size == nullptr || stages == nullptr ||
      stage_bytes == nullptr || smem_bytes == nullptr)
    return CF_ERR_INVALID_ARG;
  *clusters = h->ncl;
  *cluster_size = NCLU;
  *stages = h->stages;
  *stage_bytes = STAGE_BYTES;
  *smem_bytes = h->L.total;
  return CF_OK;
}

int cf_mla_set_timeline(cf_mla_handle* h, unsigned long long* stamps) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  h->timeline = stamps;
  return CF_OK;
}

void cf_mla_destroy(cf_mla_handle* h) {
  if (h == nullptr) return;
  if (h->ws) cudaFree(h->ws);
  delete h;
}

}  // extern "C"
