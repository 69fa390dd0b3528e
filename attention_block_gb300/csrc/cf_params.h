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

// Byte offsets of the shared-memory regions (from a 1024-aligned base).
struct SmemLayout {
  int ring;      // stages * stage_bytes       TMA ring
  int bars;      // mbarriers (see BarIdx)
  int xn;        // [BT][Hc] f32               RMS-normalized hidden, own K band
  int red;       // [N][SE] f32                projection partials / gathered slices
  int scratch;   // reduce-scatter receive buffers, later warp states, later O-proj buffer
  int qkv;       // [BT][NSEG][D] f32          full q', k', v (q' reused for o)
  int mx;        // [MXP] f32 + log2N receive  softmax max statistics
  int sm;        // [SMP] f32 + log2N receive  rescaled (o, l) partials
  int mloc;      // [MXP] f32                  local max copy
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
  static constexpr int mx = ga + kMaxRounds;           // [kMaxRounds] max all-reduce
  static constexpr int sm = mx + kMaxRounds;           // [kMaxRounds] sum all-reduce
  static constexpr int count = sm + kMaxRounds;
};

struct KParams {  // 128-byte aligned through its CUtensorMap members
  CUtensorMap tm_wqkv;   // 2D {C, H},            box {D, Rw}
  CUtensorMap tm_wo;     // 2D {H, nq*D},         box {Co, Ro}
  CUtensorMap tm_k;      // 4D {D, nkv, S, B},    box {D, 1, Rt, 1}
  CUtensorMap tm_v;      // 4D {D, nkv, S, B},    box {D, 1, Rt, 1}
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
  int B, H, nq, nkv, S;
  int N;                 // cluster size
  int nbt;               // batch tiles
  int Rw, Rt, Ro, Co;
  int stages, stage_bytes;
  float eps;
  float qk_scale_log2;   // log2(e) / sqrt(D)
  SmemLayout L;
  double inv_freq[64];   // theta^(-2i/D), i < D/2, computed in float64
};

}  // namespace cf
