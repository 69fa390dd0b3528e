// cf_params.h -- launch parameters shared by the host planner (cf_api.cu) and
// the fused decode kernel (cf_kernel.cuh).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace cf {

// Device-side error bits (the host maps them to CF_ERR_* codes).
constexpr int kDevErrPosRange = 1;
constexpr int kDevErrTimeout = 2;

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;   // 256 compute threads
constexpr int kThreads = kConsumers + 32;         // + one TMA producer warp
constexpr int kMaxCluster = 16;
constexpr int kMaxRounds = 4;                     // log2(kMaxCluster)
constexpr int kMaxStages = 32;

// Batched kernel: 64-column boxes per W_qkv stage.  The head group's NC
// projection columns come in NC/64/CB stages per slice of Rw hidden rows.  A
// few tall boxes per stage stream faster than many short ones (the TMA cost
// grows with the number of boxes and stages, not only with the bytes), so a
// stage holds four boxes where NC/64 allows.
__host__ __device__ constexpr int rows_wqkv_boxes(int NC) {
  return (NC / 64) % 4 == 0 ? 4 : ((NC / 64) % 3 == 0 ? 3 : NC / 64);
}

// Phase stamps of the optional timeline (one row of kTimelineSlots per block).
enum TimelineSlot {
  kTlStart = 0,       // after the start-up cluster barrier
  kTlNorm = 1,        // RMSNorm done
  kTlProj = 2,        // last W_qkv tile consumed and partials summed
  kTlReduceScatter = 3,
  kTlGather = 4,
  kTlAttn = 5,        // all rows' attention partials merged inside the block
  kTlMax = 6,
  kTlSum = 7,         // final o available
  kTlOproj = 8,
  kTlFinal = 9,
  kTlProdW = 10,      // producer: last W_qkv tile issued
  kTlProdKV = 11,     // producer: last K/V tile issued
  kTlProdAll = 12,    // producer: last W_o tile issued
  kTlEnd = 13,
  kTlProjLoop = 14,   // last W_qkv tile consumed by warp 0 (before the norm scale)
  kTlProjLoopLast = 15,  // same, slowest consumer warp (atomic max)
  kTlRinv = 16,       // norm scale ready
  kTlAttnFirst = 17,  // first K/V tile in hand
  kTlOprojFirst = 18, // first W_o tile in hand
  kTlOprojLoop = 19,  // last W_o tile consumed
  kTlTicket = 20,     // accumulator fence + ticket done
  kTlOprojTile1 = 21, // W_o tiles 1..3 in hand (slots 21..23)
  kTlAttnLoop = 24,   // last K/V tile and the new token consumed (row 0)
  kTlAttnWarps = 25,  // warp states written (row 0)
  kTlSmid = 26,       // not a time: the SM the block ran on
  kTimelineSlots = 32
};

// Byte offsets of the shared-memory regions (from a 1024-aligned base).  The
// comments give the sequence-split kernel's use; the batched kernel
// (cf_kernel_rows.cuh) reuses the fields for its own regions: red = partial
// sums [N][slice], scratch = x*g staging / warp states / O-projection A
// operand, xn = attention Q fragments, qkv = its rows' o, sm = attention
// record, scale = ln_weight band.
struct SmemLayout {
  int ring;      // stages * stage_bytes       TMA ring
  int bars;      // mbarriers (see BarIdx)
  int xn;        // [BT][Hc] f32               RMS-normalized hidden, own K band
  int red;       // [N][SE] f32                projection partials / gathered slices
  int scratch;   // reduce-scatter receive buffers, later warp states, later O-proj buffer
  int qkv;       // [BT][NSEG][D] f32          full q', k', v (q' reused for o)
  int sm;        // [BT*G][D+4] f32 + log2N receive: partial (o, m, l) records
  int scale;     // [BT*G][2] f32              combine factors of one round
  int rope;      // [BT][P][2] f32             cos/sin of own pairs
  int misc;      // positions [BT] i32, flags [4] i32, rinv [BT] f32, RMS partials [8][BT] f32
  int total;     // bytes incl. 1024 alignment slack
};

// mbarrier slots inside the `bars` region.
struct BarIdx {
  static constexpr int full = 0;                       // [kMaxStages]
  static constexpr int empty = kMaxStages;             // [kMaxStages]
  static constexpr int rs = 2 * kMaxStages;            // [kMaxRounds] reduce-scatter
  static constexpr int ga = rs + kMaxRounds;           // [kMaxRounds] gather
  static constexpr int sm = ga + kMaxRounds;           // [kMaxRounds] softmax-merge all-reduce
                                                       // (the batched kernel: tensor-core
                                                       // completions)
  static constexpr int count = sm + kMaxRounds;
};

struct KParams {  // 128-byte aligned through its CUtensorMap members
  CUtensorMap tm_wqkv;   // 2D {C, H},            box {D, Rw}
  CUtensorMap tm_wo;     // 2D {H, nq*D},         box {Co, Ro}
  CUtensorMap tm_k;      // 4D {D, nkv, S, B},    box {D, 1, Rt, 1}
  CUtensorMap tm_v;      // 4D {D, nkv, S, B},    box {D, 1, Rt, 1}
  CUtensorMap tm_x;      // 2D {H, B},            box {Rw, BT} (batched kernel only)
  const void* hidden;    // [B, H]
  const void* ln_w;      // [H]
  void* k_cache;         // [B, S, nkv, D]
  void* v_cache;         // [B, S, nkv, D]
  const int* positions;  // [B]
  void* out;             // [B, H]
  float* acc;            // [B, H] fp32 workspace, zero between launches
  int* counters;         // [nbt * N] completion counters, zero between launches
  int* errflag;          // device error bits
  float* dbg;            // optional intermediate dump (NULL = off)
  unsigned long long* timeline;  // optional [grid][kTimelineSlots] globaltimer stamps (NULL = off)
  int fin_split;         // batched kernel: blocks sharing the finalize of a
                         // (tile, band) (<= 1: the last block alone)
  int B, H, nq, nkv, S;
  int N;                 // cluster size
  int nbt;               // batch tiles
  int Rw, Rt, Ro, Co;
  int stages, stage_bytes;
  float eps;
  float qk_scale_log2;   // log2(e) / sqrt(D)
  SmemLayout L;
  float turn_hi[64];     // RoPE turn rate theta^(-2i/D) / (2 pi), i < D/2, as an
  float turn_lo[64];     // unevaluated float pair hi + lo computed in float64
};

}  // namespace cf
