// cf_ffn_tc.cuh -- the gated FFN of the decoder block for decode batches of
// 3 to 64 rows on the fifth-generation tensor cores (tcgen05, accumulators in
// tensor memory), as two kernels launched back to back (the second as a
// programmatic dependent of the first).
//
// Page cited by title and section:
//   [LNA] "大模型推理中的算子融合优化：LayerNorm + Attention 的 CUDA Kernel
//         手写与验证" (asdsk.com), §一 (the LLaMA block ends with a second
//         RMS Norm and the FFN) and §三 stage 1 (RMSNorm).
//
// Per batch row b (the same computation as the one- and two-row kernel):
//   n_b = h_b * g2 * rinv_b,   rinv_b = 1 / sqrt(mean(h_b^2) + eps)
//   a_bi = silu(Wg[i,:] . n_b) * (Wu[i,:] . n_b)
//   out_b = h_b + sum_i a_bi Wd[i,:]
//
// Kernel 1 (gate and up): one block per SM owns the intermediate units
// [i0, i1) (at most UB <= 128 of them).  Both products run transposed:
// M = 128 unit rows of W_gate / W_up (one TMA box of the block's rows, the
// [I, H] layout read as a K-major operand; the rows past the block's units
// are not used), N = the rows of n = h * g2 as 16-bit values -- one fp16 row
// per batch row, or for bf16 (8 significant bits) a hi row and a lo row, so
// that hi + lo carries about fp32 accuracy -- and K = the hidden dimension
// in 64-column slabs.  When 2 UB <= 128 the gate box and the up box, which
// lie next to each other in shared memory, form one M = 128 operand and one
// MMA serves both.  Phase 0 writes each block's share of the columns of n
// to a workspace and a grid barrier publishes it; every block then streams
// n with its weight boxes.  The norm scale rinv is applied in the epilogue
// (the rows' sums of squares are added up in phase 0).  The epilogue writes
// a in the operand layout kernel 2 loads: fp16 [B, I], or bf16 hi and lo
// arrays [B, I].
//
// Kernel 2 (down): (H / 128) column tiles x S splits of the units.  Each
// block computes out^T[128 columns, rows] = Wd^T a^T over its units: M = 128
// output columns (two swizzled 64-column TMA boxes of Wd, an M-major
// operand), N = a's rows (fp16, or bf16 hi rows then lo rows, loaded by TMA
// straight into a K-major slab), K = units.  The block's partial tile goes
// through shared memory to one bulk tensor reduction (add) into an fp32
// accumulator; the last split of a column tile adds the residual, writes
// `out` and clears the accumulator.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "cf_common.cuh"
#include "cf_mma.cuh"
#include "cf_params.h"
#include "cf_ptx.cuh"
#include "cf_tc05.cuh"

namespace cf {

constexpr int kFfnTcMaxStages = 8;

// Copies of the rows' sums of squares that kernel 1's blocks add into (block
// k into copy k % 8), so no word takes more than ~1/8 of the blocks' atomics.
constexpr int kFfnSsqCopies = 8;

struct FfnTcParams {
  CUtensorMap tm_wg;   // W_gate [I, H], box {64, UB}, 128-byte swizzle
  CUtensorMap tm_wu;   // W_up   [I, H], box {64, UB}
  CUtensorMap tm_n;    // n [NR, H] (h * g2: fp16 rows, or bf16 hi rows then lo rows), box {64, NR}
  CUtensorMap tm_wd;   // W_down [I, H], box {64, 64}
  CUtensorMap tm_ahi;  // a hi   [B, I], box {64, BP}
  CUtensorMap tm_alo;  // a lo   [B, I], box {64, BP}
  CUtensorMap tm_acc;  // acc    [B, H] fp32, box {128, B}, no swizzle (reduction target)
  const void* h;       // hidden [B, H] (residual)
  const void* g2;      // ln_weight [H]
  void* n;             // [NR, H] 16-bit
  float* ssq;          // [kFfnSsqCopies][BP] rows' sums of squares, zero between calls
  int* grid_count;     // arrivals at kernel 1's grid barrier, zero between calls
  int* grid_gen;       // generations of that barrier (only ever increases)
  void* a_hi;          // [B, Ip] 16-bit
  void* a_lo;          // [B, Ip] 16-bit
  void* out;           // [B, H]
  float* acc;          // [B, H] fp32, zero between calls
  int* counters;       // [H / 128], zero between calls
  int* errflag;
  int B, H, I;
  int Ip;              // row stride of a_hi / a_lo (I rounded up to 8)
  int UB;              // kernel 1: unit rows per box (multiple of 8, <= 128)
  int stacked;         // kernel 1: 2 UB <= 128, gate and up boxes as one M = 128 operand
  int nsl1, stages1, stage1_bytes;  // kernel 1: 64-column slabs per stage, ring
  int S;               // kernel 2: splits of the units
  int nsl2, stages2, stage2_bytes;  // kernel 2: 64-unit slabs per stage, ring
  int grid1;           // kernel 1's blocks (kernel 2's timeline rows follow them)
  float eps;
  unsigned long long* timeline;  // optional [grid1 + grid2][kFfnTlSlots] globaltimer
                                 // stamps (NULL = off)
};

// Stamps of the optional timeline, one row per block.  Kernel 1: start, the
// consumers' dependency wait done, phase 0 done, grid barrier passed, stage
// st landed at the MMA issuer (slot 4 + st, st < 48), every MMA complete
// (52), epilogue done (53).  Kernel 2: start, the consumers' dependency wait
// done, stage st landed (slot 4 + st), every MMA complete (52), partial tile
// reduced into the accumulator (53), done (54).
constexpr int kFfnTlSlots = 56;
constexpr int kFfnTlMaxStages = 48;

// Bounded wait until the grid-barrier generation differs from `gen0` (every
// block of this fully resident grid has arrived).  On expiry it records
// kDevErrTimeout and returns false.
static __device__ __noinline__ bool wait_generation(const int* gen, int gen0, int* errflag) {
  const long long t0 = clock64();
  for (uint32_t spins = 1;; ++spins) {
    if (*reinterpret_cast<const volatile int*>(gen) != gen0) return true;
    if ((spins & 255u) == 0) {
      if (*reinterpret_cast<volatile int*>(errflag) & kDevErrTimeout) return false;
      if (clock64() - t0 > kWaitLimitCycles) {
        atomicOr(errflag, kDevErrTimeout);
        return false;
      }
    }
    __nanosleep(64);
  }
}

// 16-bit hi + lo split of one fp32 value (hi = round(v), lo = round(v - hi)).
template <typename T>
__device__ __forceinline__ void split1(float v, T& hi, T& lo) {
  hi = Elem<T>::from_f(v);
  lo = Elem<T>::from_f(v - Elem<T>::to_f(hi));
}

// ------------------------------------------------------------ kernel 1 ---
template <typename T, int BP>
__global__ void __launch_bounds__(kThreads, 1)
    cf_ffn_gu_kernel(const __grid_constant__ FfnTcParams p) {
  using MK = MmaKind<T>;
  constexpr bool kHiLo = MK::kAttnHiLo;   // bf16: n as hi + lo rows
  constexpr int NR = kHiLo ? 2 * BP : BP;  // rows of n (the MMA's N)
  constexpr int TCOLS = tmem_cols_for(2 * NR);  // gate and up accumulators
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int slab1 = (2 * p.UB + NR) * 128;  // gate box | up box | n box
  uint8_t* ring = sm;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + (size_t)p.stages1 * p.stage1_bytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kFfnTcMaxStages;
  uint64_t* done = bars + 2 * kFfnTcMaxStages;
  // consumer thread 0 arrives here once the grid barrier has passed, i.e.
  // once every block's columns of n are published
  uint64_t* n_ready = bars + 2 * kFfnTcMaxStages + 1;
  float* rinv = reinterpret_cast<float*>(bars + 2 * kFfnTcMaxStages + 2);  // [BP]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(rinv + BP);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int i0 = (int)((long long)blockIdx.x * p.I / G);
  const int i1 = (int)((long long)(blockIdx.x + 1) * p.I / G);
  const int nslab = p.H / 64;
  const int nst = (nslab + p.nsl1 - 1) / p.nsl1;  // stages of the stream
  // 2 UB <= 128: one M = 128 MMA covers the gate box (rows 0..UB-1) and the
  // up box right after it (rows UB..2UB-1), so gate unit u accumulates in
  // TMEM lane u and up unit u in lane UB + u
  const bool stacked = p.stacked != 0;

  auto stamp = [&](int slot) {
    if (p.timeline != nullptr && tid == 0)
      p.timeline[(size_t)blockIdx.x * kFfnTlSlots + slot] = globaltimer_ns();
  };
  stamp(0);
  if (tid == 0) {
    for (int s = 0; s < p.stages1; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(done, 1);
    mbar_init(n_ready, 1);
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, TCOLS);
    tmem_relinquish();
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kConsumerWarps) {
    // ================================================ TMA producer ====
    if (lane == 0) {
      prefetch_tensormap(&p.tm_wg);
      prefetch_tensormap(&p.tm_wu);
      prefetch_tensormap(&p.tm_n);
      const uint64_t pol_w = policy_evict_first(), pol_n = policy_evict_normal();
      auto stage_slabs = [&](int st) { return min(p.nsl1, nslab - st * p.nsl1); };
      // stage st goes to ring slot s
      auto load_w = [&](int st, int s) {
        uint8_t* base = ring + (size_t)s * p.stage1_bytes;
        for (int j = 0; j < stage_slabs(st); ++j) {
          const int x = (st * p.nsl1 + j) * 64;
          tma_load_2d(base + j * slab1, &p.tm_wg, x, i0, &full[s], pol_w);
          tma_load_2d(base + j * slab1 + p.UB * 128, &p.tm_wu, x, i0, &full[s], pol_w);
        }
      };
      auto load_n = [&](int st, int s) {
        uint8_t* base = ring + (size_t)s * p.stage1_bytes;
        for (int j = 0; j < stage_slabs(st); ++j)
          tma_load_2d(base + j * slab1 + 2 * p.UB * 128, &p.tm_n, (st * p.nsl1 + j) * 64, 0,
                      &full[s], pol_n);
      };
      // The weights need nothing from this launch or the previous kernel:
      // the first stages' weight boxes go out at once, their n boxes once
      // consumer thread 0 reports that the grid barrier publishing n has
      // passed.  The barrier's words are read by that consumer only, after
      // its dependency wait: with programmatic dependent launch an earlier
      // launch of this kernel (the previous layer's) may still be inside its
      // own barrier while this one starts.
      const int fill = min(p.stages1, nst);
      for (int st = 0; st < fill; ++st) {
        mbar_arrive_expect_tx(&full[st], (uint32_t)(stage_slabs(st) * slab1));
        load_w(st, st);
      }
      mbar_wait(n_ready, 0, p.errflag);
      fence_proxy_async_global();  // n was written by other blocks' threads
      for (int st = 0; st < fill; ++st) load_n(st, st);
      RingPos rp(fill, p.stages1);
      for (int st = fill; st < nst; ++st, rp.next(p.stages1)) {
        const int s = rp.slot;
        mbar_wait(&empty[s], rp.phase ^ 1u, p.errflag);
        mbar_arrive_expect_tx(&full[s], (uint32_t)(stage_slabs(st) * slab1));
        load_w(st, s);
        load_n(st, s);
      }
    }
    __syncwarp();
  } else {
    // ================================================ consumers ========
    // h comes from the previous kernel; n, a, the row sums and the grid
    // barrier's words are reused across calls, so none of them is read or
    // written before this wait.  Once it returns, every earlier kernel of the
    // stream has completed: each launch in the chain waits for its own
    // predecessor before it can complete.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // generation of the grid barrier before this block arrives: it cannot
    // advance until every block of this launch, this one included, has
    // arrived
    const int gen0 = tid == 0 ? *reinterpret_cast<volatile int*>(p.grid_gen) : 0;
    stamp(1);
    // ---- Phase 0: this block's columns of n = h * g2 (fp16: one row per
    // batch row; bf16: hi rows 0..BP-1, lo rows BP..2BP-1 of n [NR, H]), and
    // the rows' sums of squares over them [LNA §三 stage 1] ------------------
    {
      const T* __restrict__ hid = static_cast<const T*>(p.h);
      const T* __restrict__ g2 = static_cast<const T*>(p.g2);
      T* n = static_cast<T*>(p.n);
      const int H8 = p.H / 8;
      const int c0 = (int)((long long)blockIdx.x * H8 / G);
      const int nc = (int)((long long)(blockIdx.x + 1) * H8 / G) - c0;
      // the block's (row, 8-column group) items spread over all consumer
      // threads, so their loads are in flight together; the rows' sums of
      // squares meet in shared memory (rinv holds them until the barrier)
      if (tid < BP) rinv[tid] = 0.f;
      named_sync(kBarConsumers, kConsumers);
      for (int item = tid; item < BP * nc; item += kConsumers) {
        const int b = item / nc, c = c0 + item % nc;
        float g[8], x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        load_cvt<T, 8>(g2 + 8 * c, g);
        if (b < p.B) load_cvt<T, 8>(hid + (size_t)b * p.H + 8 * c, x);
        float ss = 0.f;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ss = fmaf(x[2 * e], x[2 * e], fmaf(x[2 * e + 1], x[2 * e + 1], ss));
          MK::split2(x[2 * e] * g[2 * e], x[2 * e + 1] * g[2 * e + 1], hi[e], lo[e]);
        }
        *reinterpret_cast<uint4*>(n + (size_t)b * p.H + 8 * c) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if constexpr (kHiLo)
          *reinterpret_cast<uint4*>(n + (size_t)(BP + b) * p.H + 8 * c) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
        if (ss != 0.f) atomicAdd(&rinv[b], ss);
      }
      named_sync(kBarConsumers, kConsumers);
      if (tid < p.B && tid < BP && rinv[tid] != 0.f)
        atomicAdd(p.ssq + (blockIdx.x % kFfnSsqCopies) * BP + tid, rinv[tid]);
      // grid barrier: every block's n columns and row sums are published
      __threadfence();
      named_sync(kBarConsumers, kConsumers);
      stamp(2);
      if (tid == 0) {
        if (atomicAdd(p.grid_count, 1) == G - 1) {
          *reinterpret_cast<volatile int*>(p.grid_count) = 0;
          __threadfence();
          atomicAdd(p.grid_gen, 1);
        } else {
          wait_generation(p.grid_gen, gen0, p.errflag);
        }
        __threadfence();
        mbar_arrive(n_ready);  // the producer may now load n (also after a timeout)
      }
      named_sync(kBarConsumers, kConsumers);
      stamp(3);
    }
    if (tid < BP) {
      float t = 0.f;
#pragma unroll
      for (int k = 0; k < kFfnSsqCopies; ++k) t += __ldcg(p.ssq + k * BP + tid);
      rinv[tid] = tid < p.B ? 1.0f / sqrtf(t / (float)p.H + p.eps) : 0.f;
    }
    // ---- gate and up: one thread issues each stage's MMAs as it lands ----
    const uint32_t tmem = *s_tmem;
    const uint32_t idesc = idesc_kind_f16(MK::kBf16, 128, NR, false);
    if (tid == 0) {
      RingPos rp(0, p.stages1);
      for (int st = 0; st < nst; ++st, rp.next(p.stages1)) {
        const int s = rp.slot;
        mbar_wait(&full[s], rp.phase, p.errflag);
        if (st < kFfnTlMaxStages) stamp(4 + st);
        tc05_fence_after();
        const int ns = min(p.nsl1, nslab - st * p.nsl1);
        uint8_t* base = ring + (size_t)s * p.stage1_bytes;
        for (int j = 0; j < ns; ++j) {
          const uint32_t ag = smem_u32(base + j * slab1), au = ag + (uint32_t)p.UB * 128u;
          const uint32_t bn = ag + 2u * (uint32_t)p.UB * 128u;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const bool acc = st > 0 || j > 0 || ks > 0;
            const uint64_t bd = smem_desc_k_sw128(bn + ks * 32u, 1024);
            tc05_mma_f16(tmem, smem_desc_k_sw128(ag + ks * 32u, 1024), bd, idesc, acc);
            if (!stacked)
              tc05_mma_f16(tmem + (uint32_t)NR, smem_desc_k_sw128(au + ks * 32u, 1024), bd, idesc,
                           acc);
          }
        }
        mbar_arrive_cnt(&empty[s], kConsumerWarps - 1);
        tc05_commit(&empty[s]);
      }
      tc05_commit(done);
    }
    __syncwarp();
    named_sync(kBarConsumers, kConsumers);  // rinv
    mbar_wait(done, 0, p.errflag);
    stamp(4 + kFfnTlMaxStages);
    tc05_fence_after();
    // a = silu(gate) * up.  Warp w reads TMEM lane quarter w % 4 (lanes
    // 32 (w % 4) + lane) for rows [h BP/2, (h+1) BP/2), h = w / 4; the hi
    // and lo columns of a row are summed and scaled by the row's rinv.
    T* __restrict__ ahi = static_cast<T*>(p.a_hi);
    T* __restrict__ alo = static_cast<T*>(p.a_lo);
    const int qd = warp & 3, hrow = (warp >> 2) * (BP / 2);
    const int tl = 32 * qd + lane;  // this thread's TMEM lane
    const uint32_t dq = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)hrow;
    constexpr int RB = BP / 2 < 16 ? BP / 2 : 16;  // rows per TMEM load batch
    if (stacked) {
      // gate (lanes < UB) and up (lanes UB..2UB-1) of a unit sit in different
      // lanes: every lane's scaled sums go to shared memory (the ring is idle
      // once every MMA is complete) as S[row][lane], then each (row, unit)
      // pair is finished from there
      float* S = reinterpret_cast<float*>(ring);
      if (32 * qd < 2 * p.UB) {
#pragma unroll
        for (int r0 = 0; r0 < BP / 2; r0 += RB) {
          uint32_t vh[RB], vl[RB];
          tmem_ld_32x32b_nowait<RB>(dq + (uint32_t)r0, vh);
          if constexpr (kHiLo) tmem_ld_32x32b_nowait<RB>(dq + (uint32_t)(BP + r0), vl);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < RB; ++e) {
            const int b = hrow + r0 + e;
            float v = __uint_as_float(vh[e]);
            if constexpr (kHiLo) v += __uint_as_float(vl[e]);
            S[b * 128 + tl] = v * rinv[b];
          }
        }
      }
      named_sync(kBarConsumers, kConsumers);
      // four independent (row, unit) pairs per pass, so their shared-memory
      // reads and arithmetic overlap
      const int nu = i1 - i0, total = p.B * nu;
      for (int i = tid; i < total; i += 4 * kConsumers) {
        float z[4], up[4];
        int off[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int idx = min(i + k * kConsumers, total - 1);
          const int b = idx / nu, u = idx - b * nu;
          z[k] = S[b * 128 + u];
          up[k] = S[b * 128 + p.UB + u];
          off[k] = b * p.Ip + i0 + u;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          T hi, lo;
          split1<T>(z[k] * __frcp_rn(1.0f + __expf(-z[k])) * up[k], hi, lo);
          if (i + k * kConsumers < total) {
            ahi[off[k]] = hi;
            if constexpr (kHiLo) alo[off[k]] = lo;
          }
        }
      }
    } else if (i0 + 32 * qd < i1) {
      // gate in columns [0, NR), up in [NR, 2 NR) of the same lane (unit)
      const int unit = i0 + tl;
      const bool own = unit < i1;
#pragma unroll
      for (int r0 = 0; r0 < BP / 2; r0 += RB) {
        float rv[RB];
#pragma unroll
        for (int e = 0; e < RB; ++e) rv[e] = rinv[hrow + r0 + e];
        uint32_t gh[RB], gl[RB], uh[RB], ul[RB];
        tmem_ld_32x32b_nowait<RB>(dq + (uint32_t)r0, gh);
        tmem_ld_32x32b_nowait<RB>(dq + (uint32_t)(NR + r0), uh);
        if constexpr (kHiLo) {
          tmem_ld_32x32b_nowait<RB>(dq + (uint32_t)(BP + r0), gl);
          tmem_ld_32x32b_nowait<RB>(dq + (uint32_t)(NR + BP + r0), ul);
        }
        tmem_wait_ld();
        T hv[RB], lv[RB];
#pragma unroll
        for (int e = 0; e < RB; ++e) {
          float z = __uint_as_float(gh[e]), u = __uint_as_float(uh[e]);
          if constexpr (kHiLo) {
            z += __uint_as_float(gl[e]);
            u += __uint_as_float(ul[e]);
          }
          z *= rv[e];
          u *= rv[e];
          split1<T>(z * __frcp_rn(1.0f + __expf(-z)) * u, hv[e], lv[e]);
        }
#pragma unroll
        for (int e = 0; e < RB; ++e) {
          const int b = hrow + r0 + e;
          if (b < p.B && own) {
            ahi[(size_t)b * p.Ip + unit] = hv[e];
            if constexpr (kHiLo) alo[(size_t)b * p.Ip + unit] = lv[e];
          }
        }
      }
    }
  }
  stamp(5 + kFfnTlMaxStages);
  tc05_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc05_fence_after();
    tmem_dealloc(*s_tmem, TCOLS);
  }
}


// ------------------------------------------------------------ kernel 2 ---
template <typename T, int BP>
__global__ void __launch_bounds__(kThreads, 1)
    cf_ffn_down_kernel(const __grid_constant__ FfnTcParams p) {
  using MK = MmaKind<T>;
  constexpr bool kHiLo = MK::kAttnHiLo;   // bf16: a as hi + lo rows
  constexpr int N5 = kHiLo ? 2 * BP : BP;  // rows of the B operand (the MMA's N)
  constexpr int TCOLS = tmem_cols_for(N5);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  // slab: Wd box of columns j0..j0+63 | Wd box j0+64.. | a hi box | a lo box
  constexpr int kWBox = 64 * 128;
  constexpr int kSlab = 2 * kWBox + N5 * 128;
  uint8_t* ring = sm;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + (size_t)p.stages2 * p.stage2_bytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kFfnTcMaxStages;
  uint64_t* done = bars + 2 * kFfnTcMaxStages;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * kFfnTcMaxStages + 1);
  int* s_flag = reinterpret_cast<int*>(s_tmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int jt = blockIdx.x / p.S, split = blockIdx.x % p.S;
  const int j0 = jt * 128;
  const int nslab_all = (p.I + 63) / 64;
  const int sl0 = (int)((long long)split * nslab_all / p.S);
  const int sl1 = (int)((long long)(split + 1) * nslab_all / p.S);
  const int nslab = sl1 - sl0;
  const int nst = (nslab + p.nsl2 - 1) / p.nsl2;

  auto stamp = [&](int slot) {
    if (p.timeline != nullptr && tid == 0)
      p.timeline[(size_t)(p.grid1 + blockIdx.x) * kFfnTlSlots + slot] = globaltimer_ns();
  };
  stamp(0);
  if (tid == 0) {
    for (int s = 0; s < p.stages2; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(done, 1);
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, TCOLS);
    tmem_relinquish();
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kConsumerWarps) {
    // ================================================ TMA producer ====
    if (lane == 0) {
      prefetch_tensormap(&p.tm_wd);
      prefetch_tensormap(&p.tm_ahi);
      prefetch_tensormap(&p.tm_alo);
      prefetch_tensormap(&p.tm_acc);
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_normal();
      auto stage_slabs = [&](int st) { return min(p.nsl2, nslab - st * p.nsl2); };
      // stage st goes to ring slot s
      auto load_w = [&](int st, int s) {
        uint8_t* base = ring + (size_t)s * p.stage2_bytes;
        for (int j = 0; j < stage_slabs(st); ++j) {
          const int u = (sl0 + st * p.nsl2 + j) * 64;
          tma_load_2d(base + j * kSlab, &p.tm_wd, j0, u, &full[s], pol_w);
          tma_load_2d(base + j * kSlab + kWBox, &p.tm_wd, j0 + 64, u, &full[s], pol_w);
        }
      };
      auto load_a = [&](int st, int s) {
        uint8_t* base = ring + (size_t)s * p.stage2_bytes;
        for (int j = 0; j < stage_slabs(st); ++j) {
          const int u = (sl0 + st * p.nsl2 + j) * 64;
          tma_load_2d(base + j * kSlab + 2 * kWBox, &p.tm_ahi, u, 0, &full[s], pol_a);
          if constexpr (kHiLo)
            tma_load_2d(base + j * kSlab + 2 * kWBox + BP * 128, &p.tm_alo, u, 0, &full[s],
                        pol_a);
        }
      };
      const int fill = min(p.stages2, nst);
      for (int st = 0; st < fill; ++st) {
        mbar_arrive_expect_tx(&full[st], (uint32_t)(stage_slabs(st) * kSlab));
        load_w(st, st);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");  // a comes from kernel 1
      for (int st = 0; st < fill; ++st) load_a(st, st);
      RingPos rp(fill, p.stages2);
      for (int st = fill; st < nst; ++st, rp.next(p.stages2)) {
        const int s = rp.slot;
        mbar_wait(&empty[s], rp.phase ^ 1u, p.errflag);
        mbar_arrive_expect_tx(&full[s], (uint32_t)(stage_slabs(st) * kSlab));
        load_w(st, s);
        load_a(st, s);
      }
    }
    __syncwarp();
  } else {
    // ================================================ consumers ========
    asm volatile("griddepcontrol.wait;" ::: "memory");
    stamp(1);
    // kernel 1 of this call is complete: clear its row sums for the next call
    if (blockIdx.x == 0)
      for (int i = tid; i < kFfnSsqCopies * BP; i += kConsumers) p.ssq[i] = 0.f;
    const uint32_t tmem = *s_tmem;
    const uint32_t idesc = idesc_kind_f16(MK::kBf16, 128, N5, true);
    if (tid == 0) {
      RingPos rp(0, p.stages2);
      for (int st = 0; st < nst; ++st, rp.next(p.stages2)) {
        const int s = rp.slot;
        mbar_wait(&full[s], rp.phase, p.errflag);
        if (st < kFfnTlMaxStages) stamp(4 + st);
        tc05_fence_after();
        const int ns = min(p.nsl2, nslab - st * p.nsl2);
        uint8_t* base = ring + (size_t)s * p.stage2_bytes;
        for (int j = 0; j < ns; ++j) {
          const uint32_t aw = smem_u32(base + j * kSlab);
          const uint32_t ba = smem_u32(base + j * kSlab + 2 * kWBox);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc05_mma_f16(tmem, smem_desc_mn_sw128(aw + ks * 2048u, kWBox, 1024),
                         smem_desc_k_sw128(ba + ks * 32u, 1024), idesc, st > 0 || j > 0 || ks > 0);
        }
        mbar_arrive_cnt(&empty[s], kConsumerWarps - 1);
        tc05_commit(&empty[s]);
      }
      tc05_commit(done);
    }
    __syncwarp();
    mbar_wait(done, 0, p.errflag);
    stamp(4 + kFfnTlMaxStages);
    tc05_fence_after();
    // The partial tile [rows][128 columns] (hi + lo products summed) goes to
    // shared memory -- the ring is idle once every MMA is complete -- and
    // from there to one bulk tensor reduction (add) into the accumulator of
    // the call's B rows (the box is B rows high: rows B.. of the tile are not
    // read).  Lane = output column j0 + 32 (w % 4) + lane; rows
    // [h BP/2, (h+1) BP/2), h = w / 4.
    float* tile = reinterpret_cast<float*>(ring);
    const int qd = warp & 3, hrow = (warp >> 2) * (BP / 2);
    const int cl = 32 * qd + lane;
    const uint32_t dq = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)hrow;
    if (nslab > 0) {
#pragma unroll
      for (int r8 = 0; r8 < BP / 2; r8 += 8) {
        float vh[8], vl[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        tmem_ld_32x32b_x8(dq + (uint32_t)r8, vh);
        if constexpr (kHiLo) tmem_ld_32x32b_x8(dq + (uint32_t)(BP + r8), vl);
#pragma unroll
        for (int e = 0; e < 8; ++e) tile[(hrow + r8 + e) * 128 + cl] = vh[e] + vl[e];
      }
      fence_proxy_async_smem();
    }
    tc05_fence_before();
    named_sync(kBarConsumers, kConsumers);
    if (tid == 0) {
      if (nslab > 0) {
        tma_reduce_add_2d(&p.tm_acc, j0, 0, tile);
        bulk_commit_group();
        bulk_wait_group_0();          // the reduction's writes are performed
        fence_proxy_async_global();   // ... and ordered before the ticket below
      }
      stamp(5 + kFfnTlMaxStages);
      __threadfence();
      const int last = atomicAdd(&p.counters[jt], 1) == p.S - 1;
      if (last) __threadfence();
      s_flag[0] = last;
    }
    named_sync(kBarConsumers, kConsumers);
    if (s_flag[0]) {
      // residual of the column tile [LNA §一]
      // eight (row, 4-column) items per thread and pass (all 64 rows in one
      // pass), all loads first
      constexpr int U = 8;
      const T* __restrict__ hid = static_cast<const T*>(p.h);
      T* __restrict__ out = static_cast<T*>(p.out);
      const int items = p.B * 32;
      for (int i0 = tid; i0 < items; i0 += U * kConsumers) {
        float4 v[U];
        float x[U][4];
        size_t off[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int idx = i0 + k * kConsumers;
          off[k] = (size_t)(idx < items ? idx / 32 : 0) * p.H + j0 + 4 * (idx % 32);
          if (idx < items) {
            v[k] = __ldcg(reinterpret_cast<const float4*>(p.acc + off[k]));
            load_cvt<T, 4>(hid + off[k], x[k]);
          }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
          if (i0 + k * kConsumers < items) {
            const float r4[4] = {x[k][0] + v[k].x, x[k][1] + v[k].y, x[k][2] + v[k].z,
                                 x[k][3] + v[k].w};
            store4<T>(out + off[k], r4);
            __stcg(reinterpret_cast<float4*>(p.acc + off[k]), make_float4(0.f, 0.f, 0.f, 0.f));
          }
        }
      }
      if (tid == 0) p.counters[jt] = 0;
    }
    stamp(6 + kFfnTlMaxStages);
  }
  tc05_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc05_fence_after();
    tmem_dealloc(*s_tmem, TCOLS);
  }
}

}  // namespace cf
