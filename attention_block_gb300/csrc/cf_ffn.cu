// cf_ffn.cu -- second RMSNorm + gated FFN + residual for decode batches, as
// one kernel on sm_103a, and its C ABI (include/cf_ffn.h).
//
// Page cited by title and section:
//   [LNA] "大模型推理中的算子融合优化：LayerNorm + Attention 的 CUDA Kernel
//         手写与验证" (asdsk.com), §一 (the LLaMA block ends with a second
//         RMS Norm and the FFN) and §三 stage 1 (RMSNorm with warp-shuffle
//         reductions).
//
// The whole step is weight streaming: 3·I·H weights per call against a few
// KB of activations.  The mapping is chosen so that every byte crosses HBM
// once and in long contiguous runs:
//   * one block per SM; block k owns intermediate units [k·I/G, (k+1)·I/G)
//     (balanced to one unit), whose gate, up and down rows are contiguous
//     in the [I, H] weight layout, so each shared-memory stage is ONE bulk
//     copy of R whole rows (cp.async.bulk, mbarrier completion);
//   * a producer warp streams first the gate and up rows of all the block's
//     units (R units per stage, gate and up alternating), then their down
//     rows; it needs nothing from the previous kernel, so with programmatic
//     dependent launch the stream starts while that kernel drains (the
//     consumers wait for it before reading `hidden`);
//   * the normalized rows n live in the consumers' registers in fp32 (each
//     thread owns 4-element chunks q = tid + 256 j of the hidden dimension);
//     for a gate or up stage every warp reduces its threads' dot-product
//     partials with one transposed shuffle reduction (all R·B sums at once)
//     and stores one sum per (unit, row) in its own shared-memory slot, so
//     no block barrier stalls the stream; after the last up stage one
//     barrier, a = silu(gate) * up for all the block's units, and another
//     barrier; the down rows are then accumulated into per-thread partial
//     outputs over the owned chunks.  Measured on the Llama-2-7B shape: a
//     block barrier per group of R units cost 23 % of the step, one
//     5-shuffle butterfly per (row, batch row) another 23 %;
//   * the blocks' partial outputs meet in an fp32 accumulator through float4
//     atomics; the last block (ticket) adds the residual, writes `out` and
//     clears the accumulator for the next call.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>

#include "cf.h"
#include "cf_common.cuh"
#include "cf_ffn.h"
#include "cf_ffn_tc.cuh"
#include "cf_params.h"
#include "cf_ptx.cuh"
#include "cf_test.h"
#include "cf_tmap.h"

namespace cf {
namespace {

constexpr int kFfnMaxH = 4096;                          // hidden size the registers hold
constexpr int kFfnKC = kFfnMaxH / (4 * kConsumers);     // 4-element chunks per thread
constexpr int kFfnMaxR = 16;                            // weight rows per stage
constexpr int kFfnMaxUnits = 128;                       // intermediate units per block
constexpr int kFfnMaxStages = 8;

struct FfnParams {
  const void* h;
  const void* g2;
  const void* wg;
  const void* wu;
  const void* wd;
  void* out;
  float* acc;    // [max_batch, H], zero between calls
  int* counter;  // zero between calls
  int* errflag;
  int B, H, I, R, stages, stage_bytes;
  float eps;
};

// Shared memory after the ring: mbarriers, then float scratch.
__host__ __device__ constexpr int ffn_scratch_floats(int bmax) {
  return kConsumerWarps * 2 * kFfnMaxUnits * bmax  // per-warp gate / up sums
         + kFfnMaxUnits * bmax                     // activations
         + kConsumerWarps * bmax + 4;              // sums of squares, flag
}

// Sum of V values (V a power of two <= 32) over the 32 lanes of a warp as a
// transposed reduction: each round every lane keeps half of its values and
// adds the partner's copies of them, so after five rounds lane l holds the
// full sum of value l / (32 / V) -- V - 1 + (5 - log2 V) shuffles with a
// dependency depth of five, against 5 V for one butterfly per value.
template <int V>
__device__ __forceinline__ float warp_transposed_sum(float (&pv)[V], int lane) {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two <= 32");
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int c = V >> step;  // values held before this round
    if (c >= 2) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < c / 2; ++i) {
        const float send = upper ? pv[i] : pv[i + c / 2];
        const float keep = upper ? pv[i + c / 2] : pv[i];
        pv[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    } else {
      pv[0] += __shfl_xor_sync(0xffffffffu, pv[0], o);
    }
  }
  return pv[0];
}

template <typename T, int BMAX>
__global__ void __launch_bounds__(kThreads, 1) cf_ffn_kernel(const __grid_constant__ FfnParams p) {
  constexpr int UB = kFfnMaxUnits * BMAX;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                           ~uintptr_t(127));
  uint8_t* ring = sm;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)p.stages * p.stage_bytes);
  uint64_t* empty = full + kFfnMaxStages;
  float* wsum = reinterpret_cast<float*>(empty + kFfnMaxStages);  // [8][2][units][BMAX]
  float* av = wsum + kConsumerWarps * 2 * UB;                      // [units][BMAX]
  float* ssq = av + UB;                                            // [8][BMAX]
  int* flag = reinterpret_cast<int*>(ssq + kConsumerWarps * BMAX);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int i0 = (int)((long long)blockIdx.x * p.I / G);
  const int i1 = (int)((long long)(blockIdx.x + 1) * p.I / G);
  const int nchunk = (i1 - i0 + p.R - 1) / p.R;
  const size_t row_bytes = (size_t)p.H * sizeof(T);

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_mbar_init_cluster();
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kConsumerWarps) {
    // ============================================== weight stream ====
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint8_t* mats[3] = {static_cast<const uint8_t*>(p.wg),
                                static_cast<const uint8_t*>(p.wu),
                                static_cast<const uint8_t*>(p.wd)};
      int it = 0;
      RingPos rp(0, p.stages);
      // gate and up rows of every group, then the down rows
      for (int pass = 0; pass < 2; ++pass)
        for (int c = 0; c < nchunk; ++c) {
          const int r0 = i0 + c * p.R;
          const uint32_t bytes = (uint32_t)(min(p.R, i1 - r0) * row_bytes);
          for (int m = pass * 2; m < (pass ? 3 : 2); ++m, ++it, rp.next(p.stages)) {
            const int s = rp.slot;
            if (it >= p.stages) mbar_wait(&empty[s], rp.phase ^ 1u, p.errflag);
            mbar_arrive_expect_tx(&full[s], bytes);
            bulk_load_1d(ring + (size_t)s * p.stage_bytes, mats[m] + (size_t)r0 * row_bytes,
                         bytes, &full[s], pol);
          }
        }
    }
    __syncwarp();
    return;
  }

  // ================================================== consumer warps ====
  asm volatile("griddepcontrol.wait;" ::: "memory");  // `hidden` comes from the previous kernel
  const T* __restrict__ hid = static_cast<const T*>(p.h);
  const T* __restrict__ g2 = static_cast<const T*>(p.g2);
  const int HC = p.H / 4;

  // ---- Second RMSNorm [LNA §一, §三 stage 1]: this thread's chunks of every
  // row, the sums of squares reduced by warp shuffles and across warps --------
  float n[kFfnKC][BMAX][4];
  float ss[BMAX];
#pragma unroll
  for (int b = 0; b < BMAX; ++b) ss[b] = 0.f;
#pragma unroll
  for (int j = 0; j < kFfnKC; ++j) {
    const int q = tid + j * kConsumers;
#pragma unroll
    for (int b = 0; b < BMAX; ++b) {
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (q < HC && b < p.B) load_cvt<T, 4>(hid + (size_t)b * p.H + 4 * q, x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        n[j][b][e] = x[e];
        ss[b] = fmaf(x[e], x[e], ss[b]);
      }
    }
  }
#pragma unroll
  for (int b = 0; b < BMAX; ++b) {
    const float v = warp_sum(ss[b]);
    if (lane == 0) ssq[warp * BMAX + b] = v;
  }
  named_sync(kBarConsumers, kConsumers);
#pragma unroll
  for (int b = 0; b < BMAX; ++b) {
    float t = 0.f;
    for (int w = 0; w < kConsumerWarps; ++w) t += ssq[w * BMAX + b];
    ss[b] = b < p.B ? 1.0f / sqrtf(t / (float)p.H + p.eps) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < kFfnKC; ++j) {
    const int q = tid + j * kConsumers;
    float g[4] = {0.f, 0.f, 0.f, 0.f};
    if (q < HC) load_cvt<T, 4>(g2 + 4 * q, g);
#pragma unroll
    for (int b = 0; b < BMAX; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) n[j][b][e] = n[j][b][e] * ss[b] * g[e];
  }

  // ---- Phase A: gate and up dot products of every unit; each warp keeps
  // its own shuffle-reduced sums (no block barrier while the stream runs) --
  const int nunits = i1 - i0;
  int it = 0;
  RingPos rp(0, p.stages);
  for (int c = 0; c < nchunk; ++c) {
    const int rc = min(p.R, nunits - c * p.R);
#pragma unroll
    for (int m = 0; m < 2; ++m, ++it, rp.next(p.stages)) {
      const int s = rp.slot;
      mbar_wait(&full[s], rp.phase, p.errflag);
      const uint8_t* st = ring + (size_t)s * p.stage_bytes;
      constexpr int V = kFfnMaxR * BMAX;  // (row, batch row) partials per thread
      float part[V];
#pragma unroll
      for (int r = 0; r < kFfnMaxR; ++r) {
#pragma unroll
        for (int b = 0; b < BMAX; ++b) part[r * BMAX + b] = 0.f;
        if (r < rc) {
          const T* row = reinterpret_cast<const T*>(st + (size_t)r * row_bytes);
#pragma unroll
          for (int j = 0; j < kFfnKC; ++j) {
            const int q = tid + j * kConsumers;
            if (q < HC) {
              float w[4];
              load_cvt<T, 4>(row + 4 * q, w);
#pragma unroll
              for (int b = 0; b < BMAX; ++b)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  part[r * BMAX + b] = fmaf(w[e], n[j][b][e], part[r * BMAX + b]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      // lanes (v * 32/V .. ) end up with value v's warp sum; one of them stores it
      const float v = warp_transposed_sum<V>(part, lane);
      const int vi = lane / (32 / V);
      if (lane % (32 / V) == 0 && vi < rc * BMAX)
        wsum[(warp * 2 + m) * UB + c * p.R * BMAX + vi] = v;
    }
  }
  named_sync(kBarConsumers, kConsumers);
  for (int idx = tid; idx < nunits * BMAX; idx += kConsumers) {
    float gs = 0.f, us = 0.f;
    for (int w = 0; w < kConsumerWarps; ++w) {
      gs += wsum[(w * 2) * UB + idx];
      us += wsum[(w * 2 + 1) * UB + idx];
    }
    av[idx] = gs / (1.0f + expf(-gs)) * us;  // silu(gate) * up
  }
  named_sync(kBarConsumers, kConsumers);

  // ---- Phase B: down rows, o += a_u * Wd[u, owned chunks] -----------------
  float o[kFfnKC][BMAX][4];
#pragma unroll
  for (int j = 0; j < kFfnKC; ++j)
#pragma unroll
    for (int b = 0; b < BMAX; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[j][b][e] = 0.f;
  for (int c = 0; c < nchunk; ++c, ++it, rp.next(p.stages)) {
    const int rc = min(p.R, nunits - c * p.R);
    const int s = rp.slot;
    mbar_wait(&full[s], rp.phase, p.errflag);
    const uint8_t* st = ring + (size_t)s * p.stage_bytes;
    for (int r = 0; r < rc; ++r) {
      const T* row = reinterpret_cast<const T*>(st + (size_t)r * row_bytes);
      float a[BMAX];
#pragma unroll
      for (int b = 0; b < BMAX; ++b) a[b] = av[(c * p.R + r) * BMAX + b];
#pragma unroll
      for (int j = 0; j < kFfnKC; ++j) {
        const int q = tid + j * kConsumers;
        if (q < HC) {
          float w[4];
          load_cvt<T, 4>(row + 4 * q, w);
#pragma unroll
          for (int b = 0; b < BMAX; ++b)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[j][b][e] = fmaf(a[b], w[e], o[j][b][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- Merge the blocks' partial outputs, then residual by the last block --
#pragma unroll
  for (int j = 0; j < kFfnKC; ++j) {
    const int q = tid + j * kConsumers;
    if (q < HC) {
#pragma unroll
      for (int b = 0; b < BMAX; ++b)
        if (b < p.B)
          atomicAdd(reinterpret_cast<float4*>(p.acc + (size_t)b * p.H + 4 * q),
                    make_float4(o[j][b][0], o[j][b][1], o[j][b][2], o[j][b][3]));
    }
  }
  __threadfence();
  named_sync(kBarConsumers, kConsumers);
  if (tid == 0) {
    const int last = (atomicAdd(p.counter, 1) == G - 1);
    if (last) __threadfence();
    flag[0] = last;
  }
  named_sync(kBarConsumers, kConsumers);
  if (flag[0]) {
    T* out = static_cast<T*>(p.out);
    for (int idx = tid; idx < p.B * HC; idx += kConsumers) {
      const int b = idx / HC, q = idx % HC;
      const size_t off = (size_t)b * p.H + 4 * q;
      const float4 v = __ldcg(reinterpret_cast<const float4*>(p.acc + off));
      float x[4];
      load_cvt<T, 4>(hid + off, x);
      const float r4[4] = {x[0] + v.x, x[1] + v.y, x[2] + v.z, x[3] + v.w};
      store4<T>(out + off, r4);
      __stcg(reinterpret_cast<float4*>(p.acc + off), make_float4(0.f, 0.f, 0.f, 0.f));
    }
    if (tid == 0) *p.counter = 0;
  }
}

using FfnFn = void (*)(FfnParams);
using FfnTcFn = void (*)(FfnTcParams);

// Tensor-core pair for batches of 3..64 rows: batch tile BP = 16, 32 or 64.
void ffn_tc_entries(int dtype, int bp, FfnTcFn& gu, FfnTcFn& down) {
  if (dtype == CF_F16) {
    gu = bp == 16 ? cf_ffn_gu_kernel<__half, 16>
                  : (bp == 32 ? cf_ffn_gu_kernel<__half, 32> : cf_ffn_gu_kernel<__half, 64>);
    down = bp == 16 ? cf_ffn_down_kernel<__half, 16>
                    : (bp == 32 ? cf_ffn_down_kernel<__half, 32> : cf_ffn_down_kernel<__half, 64>);
  } else {
    gu = bp == 16 ? cf_ffn_gu_kernel<__nv_bfloat16, 16>
                  : (bp == 32 ? cf_ffn_gu_kernel<__nv_bfloat16, 32>
                              : cf_ffn_gu_kernel<__nv_bfloat16, 64>);
    down = bp == 16 ? cf_ffn_down_kernel<__nv_bfloat16, 16>
                    : (bp == 32 ? cf_ffn_down_kernel<__nv_bfloat16, 32>
                                : cf_ffn_down_kernel<__nv_bfloat16, 64>);
  }
}

// Raise a kernel's dynamic shared-memory limit to `bytes`, never lowering it
// (the attribute belongs to the function, shared by every handle).
bool raise_smem(const void* fn, int bytes) {
  cudaFuncAttributes cur;
  if (cudaFuncGetAttributes(&cur, fn) != cudaSuccess) return false;
  return cur.maxDynamicSharedSizeBytes >= bytes ||
         cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
             cudaSuccess;
}

// One cached tensor map per operand, keyed by (pointer, outer extent).
struct TmapSlot {
  const void* ptr = nullptr;
  int outer = 0;
  CUtensorMap map;
};

FfnFn ffn_entry(int dtype, int bmax) {
  if (dtype == CF_F32) return bmax == 1 ? cf_ffn_kernel<float, 1> : cf_ffn_kernel<float, 2>;
  if (dtype == CF_F16) return bmax == 1 ? cf_ffn_kernel<__half, 1> : cf_ffn_kernel<__half, 2>;
  return bmax == 1 ? cf_ffn_kernel<__nv_bfloat16, 1> : cf_ffn_kernel<__nv_bfloat16, 2>;
}

int dtype_bytes(int dtype) { return dtype == CF_F32 ? 4 : 2; }

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace cf

using namespace cf;

struct cf_ffn_handle {
  cf_ffn_config cfg;
  FfnFn fn = nullptr;
  int blocks = 0, R = 0, stages = 0, stage_bytes = 0, smem = 0, bmax = 1;
  void* ws = nullptr;  // acc | counters | errflag | a_hi | a_lo
  float* acc = nullptr;
  int* counter = nullptr;
  int* errflag = nullptr;
  // tensor-core pair (max_batch >= 3): kernel 1 gate/up, kernel 2 down
  bool tc = false;
  int BP = 0, Ip = 0;
  FfnTcFn fn_gu = nullptr, fn_down = nullptr;
  int blocks1 = 0, UB = 0, nsl1 = 0, stages1 = 0, stage1_bytes = 0, smem1 = 0;
  bool stacked = false;
  int blocks2 = 0, S = 0, nsl2 = 0, stages2 = 0, stage2_bytes = 0, smem2 = 0;
  void* a_hi = nullptr;
  void* a_lo = nullptr;
  void* n = nullptr;      // [NR, H] 16-bit: h * g2 (fp16 rows, or bf16 hi rows then lo rows)
  float* ssq = nullptr;   // [8][BP] rows' sums of squares (copies)
  int* grid = nullptr;    // kernel 1's grid barrier: [0] arrivals, [1] generation
  TmapSlot m_wg, m_wu, m_wd;
  int acc_batch = 0;      // batch the accumulator's tensor map was encoded for
  CUtensorMap m_acc;      // acc [acc_batch, H] fp32: kernel 2's reduction target
  unsigned long long* timeline = nullptr;  // optional stamps of both kernels
  CUtensorMap m_ahi, m_alo, m_n;
};

namespace {

// Plan of the tensor-core pair on a device with `sms` SMs and `budget` bytes
// of shared memory per block.  False when the shape does not fit.
bool plan_ffn_tc(cf_ffn_handle* h, int sms, int budget) {
  const cf_ffn_config& c = h->cfg;
  const int H = c.hidden, I = c.intermediate;
  h->BP = c.max_batch <= 16 ? 16 : (c.max_batch <= 32 ? 32 : 64);
  // activations (h * g2, a) as one fp16 value each, or as bf16 hi + lo pairs
  const int BP = h->BP, N5 = c.dtype == CF_BF16 ? 2 * BP : BP;
  h->Ip = (I + 7) / 8 * 8;
  // kernel 1: one block per SM, each at most UB (multiple of 8) units
  h->blocks1 = std::min(sms, I);
  const int umax = (I + h->blocks1 - 1) / h->blocks1;
  h->UB = (umax + 7) / 8 * 8;
  if (h->UB > 128) return false;
  h->stacked = 2 * h->UB <= 128;
  const int slab1 = (2 * h->UB + N5) * 128;  // gate box | up box | n box
  int extras1 = (2 * kFfnTcMaxStages + 2) * 8 + BP * 4 + 16;  // barriers, rinv, TMEM word
  // the M = 128 operand reads of a slab's gate and up boxes run up to 16 KB
  // past the box start: keep that much shared memory after the ring
  extras1 = std::max(extras1, 16384 - (h->UB + N5) * 128);
  extras1 = (extras1 + 1023) / 1024 * 1024;
  h->nsl1 = std::max(1, std::min(H / 64, 65536 / slab1));
  for (;; --h->nsl1) {
    h->stage1_bytes = h->nsl1 * slab1;
    h->stages1 = std::min(kFfnTcMaxStages, (budget - extras1) / h->stage1_bytes);
    if (h->stages1 >= 2 || h->nsl1 == 1) break;
  }
  if (h->stages1 < 2) return false;
  h->smem1 = h->stages1 * h->stage1_bytes + extras1 + 1024;
  // the stacked epilogue stages the fp32 sums [BP][128] in the idle ring
  if (h->stacked && BP * 128 * (int)sizeof(float) > h->stages1 * h->stage1_bytes) return false;
  // kernel 2: H / 128 column tiles x S splits of the 64-unit slabs
  const int tiles = H / 128, slabs = (I + 63) / 64;
  h->S = std::max(1, std::min(slabs, sms / tiles));
  h->blocks2 = tiles * h->S;
  const int slab2 = (128 + N5) * 128;
  const int extras2 = 1024;
  h->nsl2 = std::max(1, std::min((slabs + h->S - 1) / h->S, 65536 / slab2));
  h->stage2_bytes = h->nsl2 * slab2;
  h->stages2 = std::min(kFfnTcMaxStages, (budget - extras2) / h->stage2_bytes);
  // the epilogue stages the fp32 partial tile [BP][128] in the idle ring
  if (h->stages2 < 2 || BP * 128 * (int)sizeof(float) > h->stage2_bytes) return false;
  h->smem2 = h->stages2 * h->stage2_bytes + extras2 + 1024;
  ffn_tc_entries(c.dtype, BP, h->fn_gu, h->fn_down);
  if (!raise_smem(reinterpret_cast<const void*>(h->fn_gu), h->smem1) ||
      !raise_smem(reinterpret_cast<const void*>(h->fn_down), h->smem2)) {
    cudaGetLastError();
    return false;
  }
  return true;
}

const CUtensorMap* cached_map(TmapSlot& slot, int dtype, const void* ptr, uint64_t inner,
                              uint64_t outer, uint32_t box_outer) {
  if (slot.ptr != ptr || slot.outer != (int)outer) {
    if (!encode_tmap_2d(&slot.map, dtype, ptr, inner, outer, inner * 2, 64, box_outer, true)) {
      slot.ptr = nullptr;
      return nullptr;
    }
    slot.ptr = ptr;
    slot.outer = (int)outer;
  }
  return &slot.map;
}

}  // namespace

extern "C" int cf_ffn_create(const cf_ffn_config* cfg, cf_ffn_handle** out) {
  if (out == nullptr) return CF_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg == nullptr) return CF_ERR_INVALID_ARG;
  const cf_ffn_config c = *cfg;
  if (c.hidden <= 0 || c.hidden % 8 != 0 || c.intermediate <= 0 || c.max_batch <= 0 ||
      c.dtype < CF_F32 || c.dtype > CF_BF16 || !(c.rms_eps >= 0.f) || c.stage_bytes < 0)
    return CF_ERR_INVALID_ARG;
  // batches of 3+ rows: the tensor-core pair (16-bit storage, H a multiple
  // of 128, at most 64 rows)
  if (c.hidden > kFfnMaxH || c.max_batch > 64) return CF_ERR_UNSUPPORTED;
  if (c.max_batch > 2 && (c.dtype == CF_F32 || c.hidden % 128 != 0)) return CF_ERR_UNSUPPORTED;
  const int row_bytes = c.hidden * dtype_bytes(c.dtype);
  if (c.stage_bytes != 0 && c.stage_bytes < row_bytes) return CF_ERR_INVALID_ARG;
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
    return CF_ERR_CUDA;
  cf_ffn_handle* h = new (std::nothrow) cf_ffn_handle();
  if (h == nullptr) return CF_ERR_CUDA;
  h->cfg = c;
  h->bmax = c.max_batch <= 1 ? 1 : 2;
  h->fn = ffn_entry(c.dtype, h->bmax);
  const int extras = 2 * kFfnMaxStages * 8 + ffn_scratch_floats(h->bmax) * 4 + 128;
  const int budget = (int)prop.sharedMemPerBlockOptin;
  // Default: the largest stage of whole rows that still leaves two stages.
  // Measured (fraction of the copy bandwidth, Llama-2-7B FFN / Llama-3-8B FFN
  // at B = 2): 2 x 104 KB 0.96 / 0.92, 3 x 64 KB 0.98 / 0.88, 4 x 48 KB
  // 0.90 / 0.78, 6 x 32 KB 0.73 / 0.63 -- the cost per stage outweighs the
  // depth of the ring.
  const int req = c.stage_bytes ? c.stage_bytes : (budget - extras) / 2 / 128 * 128;
  h->R = std::min(kFfnMaxR, req / row_bytes);
  if (h->R < 1) {
    delete h;
    return CF_ERR_UNSUPPORTED;
  }
  h->stage_bytes = (h->R * row_bytes + 127) / 128 * 128;
  h->stages = std::min(kFfnMaxStages, (budget - extras) / h->stage_bytes);
  if (h->stages < 2) {
    delete h;
    return CF_ERR_UNSUPPORTED;
  }
  h->smem = h->stages * h->stage_bytes + extras;
  h->blocks = std::min(prop.multiProcessorCount, c.intermediate);
  if ((c.intermediate + h->blocks - 1) / h->blocks > kFfnMaxUnits) {
    delete h;
    return CF_ERR_UNSUPPORTED;
  }
  if (!raise_smem(reinterpret_cast<const void*>(h->fn), h->smem)) {
    cudaGetLastError();
    delete h;
    return CF_ERR_CUDA;
  }
  h->tc = c.max_batch > 2;
  if (h->tc && !plan_ffn_tc(h, prop.multiProcessorCount,
                            (int)prop.sharedMemPerBlockOptin - 1024)) {
    delete h;
    return CF_ERR_UNSUPPORTED;
  }
  // workspace: acc | 512-byte control block (counters [32], errflag, grid
  // barrier [2]) | row sums [8][64] | a_hi | a_lo | n
  const size_t acc_bytes = (size_t)c.max_batch * c.hidden * sizeof(float);
  const size_t a_bytes = h->tc ? (size_t)c.max_batch * h->Ip * 2 : 0;
  const int n_rows = c.dtype == CF_BF16 ? 2 * h->BP : h->BP;
  const size_t n_bytes = h->tc ? (size_t)n_rows * c.hidden * 2 : 0;
  const size_t ssq_bytes = (size_t)kFfnSsqCopies * 64 * sizeof(float);
  const size_t total = acc_bytes + 512 + ssq_bytes + 2 * a_bytes + n_bytes;
  if (cudaMalloc(&h->ws, total) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return CF_ERR_CUDA;
  }
  if (cudaMemset(h->ws, 0, total) != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return CF_ERR_CUDA;
  }
  h->acc = static_cast<float*>(h->ws);
  h->counter = reinterpret_cast<int*>(static_cast<char*>(h->ws) + acc_bytes);  // [32]
  h->errflag = h->counter + 32;
  if (h->tc) {
    h->grid = h->errflag + 1;
    h->ssq = reinterpret_cast<float*>(static_cast<char*>(h->ws) + acc_bytes + 512);
    h->a_hi = static_cast<char*>(h->ws) + acc_bytes + 512 + ssq_bytes;
    h->a_lo = static_cast<char*>(h->a_hi) + a_bytes;
    h->n = static_cast<char*>(h->a_lo) + a_bytes;
    if (!encode_tmap_2d(&h->m_n, c.dtype, h->n, c.hidden, n_rows, (uint64_t)c.hidden * 2, 64,
                        n_rows, true)) {
      cudaFree(h->ws);
      delete h;
      return CF_ERR_CUDA;
    }
    if (!encode_tmap_2d(&h->m_ahi, c.dtype, h->a_hi, c.intermediate, c.max_batch, h->Ip * 2, 64,
                        h->BP, true) ||
        !encode_tmap_2d(&h->m_alo, c.dtype, h->a_lo, c.intermediate, c.max_batch, h->Ip * 2, 64,
                        h->BP, true)) {
      cudaFree(h->ws);
      delete h;
      return CF_ERR_CUDA;
    }
  }
  *out = h;
  return CF_OK;
}

namespace {

// Batches of 3+ rows: gate/up kernel, then the down kernel as its
// programmatic dependent.
int ffn_forward_tc(cf_ffn_handle* h, int batch, const void* hidden, const void* ln_weight,
                   const void* w_gate, const void* w_up, const void* w_down, void* out,
                   void* stream) {
  const cf_ffn_config& c = h->cfg;
  const uint64_t H = c.hidden, I = c.intermediate;
  const CUtensorMap* mg = cached_map(h->m_wg, c.dtype, w_gate, H, I, h->UB);
  const CUtensorMap* mu = cached_map(h->m_wu, c.dtype, w_up, H, I, h->UB);
  const CUtensorMap* md = cached_map(h->m_wd, c.dtype, w_down, H, I, 64);
  if (!mg || !mu || !md) return CF_ERR_CUDA;
  if (h->acc_batch != batch) {
    // box = exactly the call's rows, so the reduction never leaves the tensor
    if (!encode_tmap_2d(&h->m_acc, CF_F32, h->acc, H, (uint64_t)batch, H * sizeof(float), 128,
                        (uint32_t)batch, false)) {
      h->acc_batch = 0;
      return CF_ERR_CUDA;
    }
    h->acc_batch = batch;
  }
  FfnTcParams p;
  std::memset(&p, 0, sizeof(p));
  p.tm_wg = *mg;
  p.tm_wu = *mu;
  p.tm_n = h->m_n;
  p.n = h->n;
  p.ssq = h->ssq;
  p.grid_count = h->grid;
  p.grid_gen = h->grid + 1;
  p.tm_acc = h->m_acc;
  p.tm_wd = *md;
  p.tm_ahi = h->m_ahi;
  p.tm_alo = h->m_alo;
  p.h = hidden;
  p.g2 = ln_weight;
  p.a_hi = h->a_hi;
  p.a_lo = h->a_lo;
  p.out = out;
  p.acc = h->acc;
  p.counters = h->counter;
  p.errflag = h->errflag;
  p.B = batch;
  p.H = c.hidden;
  p.I = c.intermediate;
  p.Ip = h->Ip;
  p.UB = h->UB;
  p.stacked = h->stacked ? 1 : 0;
  p.nsl1 = h->nsl1;
  p.stages1 = h->stages1;
  p.stage1_bytes = h->stage1_bytes;
  p.S = h->S;
  p.nsl2 = h->nsl2;
  p.stages2 = h->stages2;
  p.stage2_bytes = h->stage2_bytes;
  p.grid1 = h->blocks1;
  p.eps = c.rms_eps;
  p.timeline = h->timeline;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  void* args[] = {&p};
  const FfnTcFn fns[2] = {h->fn_gu, h->fn_down};
  const int grids[2] = {h->blocks1, h->blocks2}, smems[2] = {h->smem1, h->smem2};
  for (int k = 0; k < 2; ++k) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grids[k], 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = smems[k];
    lc.stream = static_cast<cudaStream_t>(stream);
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (cudaLaunchKernelExC(&lc, reinterpret_cast<const void*>(fns[k]), args) != cudaSuccess) {
      cudaGetLastError();
      return CF_ERR_CUDA;
    }
  }
  return CF_OK;
}

}  // namespace

extern "C" int cf_ffn_forward(cf_ffn_handle* h, int32_t batch, const void* hidden,
                              const void* ln_weight, const void* w_gate, const void* w_up,
                              const void* w_down, void* out, void* stream) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  const cf_ffn_config& c = h->cfg;
  if (batch < 0 || batch > c.max_batch) return CF_ERR_INVALID_ARG;
  if (batch == 0) return CF_OK;
  const void* ptrs[] = {hidden, ln_weight, w_gate, w_up, w_down, out};
  for (const void* q : ptrs)
    if (q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u) != 0) return CF_ERR_INVALID_ARG;
  const size_t es = dtype_bytes(c.dtype);
  const size_t act = (size_t)batch * c.hidden * es, mat = (size_t)c.intermediate * c.hidden * es;
  if (ranges_overlap(out, act, hidden, act) ||
      ranges_overlap(out, act, ln_weight, (size_t)c.hidden * es) ||
      ranges_overlap(out, act, w_gate, mat) || ranges_overlap(out, act, w_up, mat) ||
      ranges_overlap(out, act, w_down, mat))
    return CF_ERR_ALIAS;
  if (batch > 2) return ffn_forward_tc(h, batch, hidden, ln_weight, w_gate, w_up, w_down, out,
                                       stream);
  FfnParams p;
  std::memset(&p, 0, sizeof(p));
  p.h = hidden;
  p.g2 = ln_weight;
  p.wg = w_gate;
  p.wu = w_up;
  p.wd = w_down;
  p.out = out;
  p.acc = h->acc;
  p.counter = h->counter;
  p.errflag = h->errflag;
  p.B = batch;
  p.H = c.hidden;
  p.I = c.intermediate;
  p.R = h->R;
  p.stages = h->stages;
  p.stage_bytes = h->stage_bytes;
  p.eps = c.rms_eps;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = dim3(h->blocks, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = h->smem;
  lc.stream = static_cast<cudaStream_t>(stream);
  lc.attrs = attr;
  lc.numAttrs = 1;
  void* args[] = {&p};
  if (cudaLaunchKernelExC(&lc, reinterpret_cast<const void*>(h->fn), args) != cudaSuccess) {
    cudaGetLastError();
    return CF_ERR_CUDA;
  }
  return CF_OK;
}

extern "C" int cf_ffn_get_status(cf_ffn_handle* h) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  int flag = 0;
  if (cudaMemcpy(&flag, h->errflag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CF_ERR_CUDA;
  if (flag != 0 && cudaMemset(h->errflag, 0, sizeof(int)) != cudaSuccess) return CF_ERR_CUDA;
  return (flag & kDevErrTimeout) ? CF_ERR_DEVICE_TIMEOUT : CF_OK;
}

extern "C" int cf_ffn_launch_info(const cf_ffn_handle* h, int32_t* blocks, int32_t* rows_per_stage,
                                  int32_t* stages) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  if (blocks) *blocks = h->blocks;
  if (rows_per_stage) *rows_per_stage = h->R;
  if (stages) *stages = h->stages;
  return CF_OK;
}

extern "C" int cf_ffn_set_timeline(cf_ffn_handle* h, unsigned long long* stamps) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  h->timeline = stamps;
  return CF_OK;
}

extern "C" int cf_ffn_kernels(const cf_ffn_handle* h, int32_t batch, int32_t* blocks1,
                              int32_t* blocks2) {
  if (h == nullptr || batch < 1 || batch > h->cfg.max_batch) return CF_ERR_INVALID_ARG;
  const bool tc = batch > 2;
  if (blocks1) *blocks1 = tc ? h->blocks1 : h->blocks;
  if (blocks2) *blocks2 = tc ? h->blocks2 : 0;
  return tc ? 2 : 1;
}

extern "C" int cf_ffn_debug_a(const cf_ffn_handle* h, int32_t batch, float* a_out) {
  if (h == nullptr || a_out == nullptr || batch < 1 || batch > h->cfg.max_batch)
    return CF_ERR_INVALID_ARG;
  if (!h->tc) return CF_ERR_UNSUPPORTED;
  const int I = h->cfg.intermediate, Ip = h->Ip;
  const size_t n = (size_t)batch * Ip;
  uint16_t* hi = new (std::nothrow) uint16_t[2 * n];
  if (hi == nullptr) return CF_ERR_CUDA;
  uint16_t* lo = hi + n;
  const bool ok = cudaMemcpy(hi, h->a_hi, n * 2, cudaMemcpyDeviceToHost) == cudaSuccess &&
                  cudaMemcpy(lo, h->a_lo, n * 2, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (ok) {
    // bf16: a = hi + lo; fp16: a = hi alone
    const bool bf = h->cfg.dtype == CF_BF16;
    for (int b = 0; b < batch; ++b)
      for (int i = 0; i < I; ++i) {
        const size_t k = (size_t)b * Ip + i;
        a_out[(size_t)b * I + i] =
            bf ? __bfloat162float(*reinterpret_cast<__nv_bfloat16*>(&hi[k])) +
                     __bfloat162float(*reinterpret_cast<__nv_bfloat16*>(&lo[k]))
               : __half2float(*reinterpret_cast<__half*>(&hi[k]));
      }
  }
  delete[] hi;
  return ok ? CF_OK : CF_ERR_CUDA;
}

extern "C" void cf_ffn_destroy(cf_ffn_handle* h) {
  if (h == nullptr) return;
  if (h->ws) cudaFree(h->ws);
  delete h;
}
