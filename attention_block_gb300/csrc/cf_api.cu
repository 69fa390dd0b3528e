// cf_api.cu -- host side of the C ABI declared in include/cf.h: argument
// validation, kernel-instance choice, shared-memory planning, TMA tensor-map
// encoding (cached per pointer), the handle's device workspace and the
// cluster launch.  No allocation, synchronization or host copy happens on the
// cf_decode_attn_block path, so it can be captured in a CUDA graph.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "cf.h"
#include "cf_params.h"
#include "cf_registry.h"
#include "cf_test.h"
#include "cf_unfused.h"

using namespace cf;

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

int esize(int dt) { return dt == CF_F32 ? 4 : 2; }

CUtensorMapDataType tm_type(int dt) {
  return dt == CF_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                      : (dt == CF_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
int pow2_floor(int v) {
  int p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}
// Largest power of two <= cap that divides v (v > 0).
int pow2_divisor(int v, int cap) {
  int p = 1;
  while (p * 2 <= cap && v % (p * 2) == 0) p *= 2;
  return p;
}
int round_up(int v, int a) { return (v + a - 1) / a * a; }

const KernelEntry* find_entry(int dtype, int D, int G, int BT) {
  const KernelEntry* e = nullptr;
  int n = dtype == CF_F32 ? registry_f32(&e) : (dtype == CF_F16 ? registry_f16(&e) : registry_bf16(&e));
  for (int i = 0; i < n; ++i)
    if (e[i].D == D && e[i].G == G && e[i].BT == BT) return &e[i];
  return nullptr;
}

// Largest compiled batch tile <= want for (dtype, D, G); 0 if none.
int best_batch_tile(int dtype, int D, int G, int want) {
  const KernelEntry* e = nullptr;
  int n = dtype == CF_F32 ? registry_f32(&e) : (dtype == CF_F16 ? registry_f16(&e) : registry_bf16(&e));
  int best = 0;
  for (int i = 0; i < n; ++i)
    if (e[i].D == D && e[i].G == G && e[i].BT <= want && e[i].BT > best) best = e[i].BT;
  return best;
}

// Small per-handle cache of encoded tensor maps keyed by (pointer, extent).
struct MapCache {
  static constexpr int kSlots = 64;
  const void* ptr[kSlots] = {};
  int extent[kSlots] = {};
  CUtensorMap map[kSlots];
  int next = 0;
  const CUtensorMap* find(const void* p, int e) const {
    for (int i = 0; i < kSlots; ++i)
      if (ptr[i] == p && extent[i] == e && p != nullptr) return &map[i];
    return nullptr;
  }
  CUtensorMap* insert(const void* p, int e) {
    const int i = next;
    next = (next + 1) % kSlots;
    ptr[i] = p;
    extent[i] = e;
    return &map[i];
  }
};

struct Plan {
  int N, BT, G, Rw, Rt, Ro, Co, stages, stage_bytes, ctas_per_sm;
  SmemLayout L;
  int mode = 0;  // 0 sequence-split kernel, 1 batched row-split kernel
  int RPC = 0;   // rows per block (mode 1)
};

// Shared-memory plan of the batched row-split kernel (one block per SM):
// N = BT / RPC blocks per cluster, K band Hc = H / N.  Returns false when the
// shape does not fit (the caller then tries another instance).
bool make_plan_rows(const cf_config& c, int BT, int RPC, int stage_req, const cudaDeviceProp& prop,
                    Plan& pl) {
  const int es = esize(c.dtype), D = c.head_dim, H = c.hidden;
  const int G = c.n_q_heads / c.n_kv_heads, NSEG = G + 2, NC = NSEG * D, GD = G * D;
  const int N = BT / RPC;
  if (N < 1 || N > kMaxCluster || (N & (N - 1)) != 0 || H % (64 * N) != 0) return false;
  const int Hc = H / N;
  pl.mode = 1;
  pl.RPC = RPC;
  pl.N = N;
  pl.BT = BT;
  pl.G = G;
  pl.ctas_per_sm = 1;
  pl.Co = (Hc % 256 == 0) ? 256 : ((Hc % 128 == 0) ? 128 : 64);
  // tiles of 16+ rows run the O projection on tcgen05 in 128-column tiles
  const bool tc5 = BT >= 16;
  if (tc5 && pl.Co < 128) return false;
  // W_qkv stage: Rw rows of CB 64-column boxes of the group's NC columns;
  // the first stage of each slice of Rw rows also holds the [BT x Rw] slice
  // of x
  const int CB = rows_wqkv_boxes(NC);
  int rw = 16;
  while (rw * 2 <= 256 && Hc % (rw * 2) == 0 && (rw * 2) * CB * 64 * es <= stage_req) rw *= 2;
  pl.Rw = rw;
  // K/V tile: Rt positions of K and of V (32 <= Rt <= 256, a power of two:
  // the attention hands out 32-position chunks)
  pl.Rt = std::min(256, pow2_floor(std::max(32, stage_req / (2 * D * es))));
  int ro = 16;
  while (ro * 2 <= 256 && GD % (ro * 2) == 0 && (ro * 2) * pl.Co * es <= stage_req) ro *= 2;
  pl.Ro = ro;
  const int item =
      std::max((CB * 64 + BT) * pl.Rw * es, std::max(2 * pl.Rt * D * es, pl.Ro * pl.Co * es));
  pl.stage_bytes = round_up(item, 1024);

  const int SE = RPC * NC + (RPC + 3) / 4 * 4;  // reduce-scatter slice (floats)
  const int OP = 4 * GD + 16;                   // O-projection A row (bytes)
  const int apitch = (pl.Rw + 8) * 2;           // staged x*g row (bytes)
  int off = 0;
  SmemLayout& L = pl.L;
  auto take = [&](int bytes) {
    const int o = off;
    off += round_up(bytes, 128);
    return o;
  };
  L.bars = take(BarIdx::count * 8);
  L.red = take(N * SE * 4);
  // one region, three lifetimes: x*g staging of the BT rows (projection),
  // warp states (attention merge), the O-projection A operand of the BT
  // rows (after attention); rows BT..15 of a 16-row MMA tile read a zero chunk
  const int slots = G > 1 ? 4 : 8;  // warp-state slots of the attention merge
  int scratch = std::max(4 * BT * apitch, std::max(slots * G * (D + 4) * 4, BT * OP));
  if (tc5) {
    // tcgen05 operands in 128-byte-swizzled slabs (1024-byte aligned): two
    // x buffers of ceil(Rw/64) slabs of 2*BT rows, later o in G*D/64 slabs
    scratch = std::max(scratch, std::max(2 * ((pl.Rw + 63) / 64) * 256 * BT, (GD / 64) * 256 * BT));
    off = round_up(off, 1024);
  }
  L.scratch = take(scratch);
  L.xn = take((D / 16) * 32 * 16);  // Q fragments of the attention
  L.qkv = take(RPC * GD * 4);       // own rows' o
  L.sm = take(G * (D + 4) * 4);     // attention record
  L.scale = 0;                      // unused (ln_weight is read from L2)
  L.rope = take(RPC * (D / 2) * 2 * 4);
  L.misc = take((4 + BT + 4 + RPC) * 4);  // zero chunk, positions, flags, norm scales
  const int extras = round_up(off, 1024);
  int budget = std::min((int)prop.sharedMemPerBlockOptin,
                        (int)prop.sharedMemPerMultiprocessor - (int)prop.reservedSharedMemPerBlock);
  budget -= 1024;
  int stages = std::min((budget - extras) / pl.stage_bytes, kMaxStages);
  if (c.max_stages > 0) stages = std::min(stages, c.max_stages);
  // On tcgen05 only the MMA-issuing thread waits for every W_qkv stage; the
  // other consumers wait for the first stage of each K slice only, NC/64/CB
  // ring slots after the previous one.  The ring must hold a whole slice's
  // stages, or that wait could meet a slot whose earlier fill is still
  // pending and take its parity as complete.
  const int min_stages = tc5 ? std::max(2, NC / 64 / CB) : 2;
  if (stages < min_stages) {
    // a default stage size larger than 32 KB that leaves too few stages:
    // retry with 32 KB
    if (c.stage_bytes == 0 && stage_req > 32768)
      return make_plan_rows(c, BT, RPC, 32768, prop, pl);
    return false;
  }
  pl.stages = stages;
  const int ring = stages * pl.stage_bytes;
  L.ring = 0;
  for (int* f : {&L.bars, &L.red, &L.scratch, &L.xn, &L.qkv, &L.sm, &L.rope, &L.misc})
    *f += ring;
  L.total = ring + extras + 1024;
  return true;
}

// Completion counters for `batch_cap` rows: one per (batch tile, column
// band).
size_t counter_slots(const Plan& pl, int batch_cap) {
  return (size_t)((batch_cap + pl.BT - 1) / pl.BT) * pl.N;
}

// Shared-memory plan for one (config, N, BT, stage size, CTAs/SM).  Returns
// false when not even two ring stages fit.
bool make_plan(const cf_config& c, int N, int BT, int stage_req, int ctas_per_sm,
               const cudaDeviceProp& prop, Plan& pl) {
  const int es = esize(c.dtype), D = c.head_dim, H = c.hidden;
  const int G = c.n_q_heads / c.n_kv_heads, NSEG = G + 2;
  const int P = D / (2 * N), SE = BT * NSEG * 2 * P;
  const int Hc = H / N;
  const int nrounds = __builtin_ctz((unsigned)N);
  pl.N = N;
  pl.BT = BT;
  pl.G = G;
  pl.Co = pow2_divisor(Hc, 256);
  pl.Rw = pow2_divisor(Hc, std::min(256, std::max(1, stage_req / (NSEG * D * es))));
  pl.Rt = std::min(256, pow2_floor(std::max(1, stage_req / (2 * D * es))));
  pl.Ro = pow2_divisor(G * D, std::min(256, std::max(1, stage_req / (pl.Co * es))));
  int item = std::max(NSEG * pl.Rw * D * es, std::max(2 * pl.Rt * D * es, pl.Ro * pl.Co * es));
  // A held stage also serves as the buffer of the projection's cross-warp
  // tree (at least 4 slots of BT*NSEG*(D/32) floats per lane) and of the
  // O projection's row-group partials ([RG][BT][Co] floats, RG*Co = 256 *
  // (16 / element size)).
  item = std::max(item, std::max(4 * BT * NSEG * (D / 32) * 32 * 4, 256 * (16 / es) * BT * 4));
  pl.stage_bytes = round_up(item, 1024);

  const int SMP = BT * G * (D + 4);
  int off = 0;
  SmemLayout& L = pl.L;
  auto take = [&](int bytes) {
    const int o = off;
    off += round_up(bytes, 128);
    return o;
  };
  L.bars = take(BarIdx::count * 8);
  L.xn = take(BT * Hc * 4);
  L.red = take(N * SE * 4);
  L.scratch = take(std::max((N - 1) * SE, kConsumerWarps * G * (D + 4)) * 4);
  L.qkv = take(BT * NSEG * D * 4);
  L.sm = take(SMP * 4 * (1 + nrounds));
  L.scale = take(BT * G * 2 * 4);
  L.rope = take(BT * P * 2 * 4);
  L.misc = take((BT + 4 + BT + kConsumerWarps * BT) * 4);
  const int extras = round_up(off, 1024);

  const int per_sm = (int)prop.sharedMemPerMultiprocessor;
  const int per_block_max = (int)prop.sharedMemPerBlockOptin;
  int budget = std::min(per_block_max, per_sm / ctas_per_sm - (int)prop.reservedSharedMemPerBlock);
  budget -= 1024;  // alignment slack of the dynamic base
  int stages = (budget - extras) / pl.stage_bytes;
  stages = std::min(stages, kMaxStages);
  if (c.max_stages > 0) stages = std::min(stages, c.max_stages);
  if (stages < 2) return false;
  pl.stages = stages;
  pl.ctas_per_sm = ctas_per_sm;
  // ring first, then the other regions (all offsets from the 1024-aligned base)
  const int ring = stages * pl.stage_bytes;
  L.ring = 0;
  L.bars += ring;
  L.xn += ring;
  L.red += ring;
  L.scratch += ring;
  L.qkv += ring;
  L.sm += ring;
  L.scale += ring;
  L.rope += ring;
  L.misc += ring;
  L.total = ring + extras + 1024;
  return true;
}

}  // namespace

// One launch shape of a handle, used for batches of at most `cap` rows.
struct PlanSlot {
  int cap = 0;
  Plan plan;
  const void* fn = nullptr;
  int max_active_clusters = 0;
  MapCache m_wqkv, m_wo, m_k, m_v, m_x;  // tensor maps have the plan's box shapes
};
constexpr int kMaxPlanSlots = 8;

struct cf_handle {
  cf_config cfg;
  int device = 0, sm_count = 0;
  // Launch shapes in ascending batch capacity; the last serves max_batch.
  // A call uses the first slot whose capacity holds its batch (runtime choice
  // of the kernel instance and cluster shape per batch).
  PlanSlot slots[kMaxPlanSlots];
  int nslots = 0;
  PlanSlot& main() { return slots[nslots - 1]; }
  const PlanSlot& main() const { return slots[nslots - 1]; }
  const PlanSlot& slot_for(int batch) const {
    for (int i = 0; i < nslots; ++i)
      if (batch <= slots[i].cap) return slots[i];
    return main();
  }
  void* ws = nullptr;       // one allocation: acc | counters | errflag
  float* acc = nullptr;
  int* counters = nullptr;
  int* errflag = nullptr;
  float* dbg = nullptr;
  unsigned long long* timeline = nullptr;
  bool pdl = true;
  float turn_hi[64], turn_lo[64];  // RoPE turn rates as float pairs (see KParams)
  // three-kernel (unfused) path: HBM intermediates and counters
  void* uf_ws = nullptr;
  float *uf_y = nullptr, *uf_part = nullptr, *uf_o32 = nullptr;
  int *uf_cnt_attn = nullptr, *uf_cnt_out = nullptr;
  float* uf_rinv = nullptr;
  int uf_NS = 1, uf_KS = 1, uf_KS1 = 1;
};

namespace {

int validate_config(const cf_config* c) {
  if (c == nullptr) return CF_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->hidden % 64 != 0) return CF_ERR_INVALID_ARG;
  if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->n_q_heads % c->n_kv_heads != 0)
    return CF_ERR_INVALID_ARG;
  if (c->head_dim <= 0 || c->head_dim % 2 != 0) return CF_ERR_INVALID_ARG;
  if (c->max_batch <= 0 || c->s_max <= 0) return CF_ERR_INVALID_ARG;
  if (c->dtype < CF_F32 || c->dtype > CF_BF16) return CF_ERR_INVALID_ARG;
  if (!(c->rope_theta > 0.f) || !std::isfinite(c->rope_theta)) return CF_ERR_INVALID_ARG;
  if (!(c->rms_eps >= 0.f) || !std::isfinite(c->rms_eps)) return CF_ERR_INVALID_ARG;
  const int N = c->cluster_size;
  if (N != 0 && !(N == 1 || N == 2 || N == 4 || N == 8 || N == 16)) return CF_ERR_INVALID_ARG;
  if (c->batch_tile < 0 || c->stage_bytes < 0) return CF_ERR_INVALID_ARG;
  if (c->stage_bytes != 0 && (c->stage_bytes < 2048 || c->stage_bytes > 131072))
    return CF_ERR_INVALID_ARG;
  if (c->ctas_per_sm < 0 || c->ctas_per_sm > 2) return CF_ERR_INVALID_ARG;
  if (c->adaptive < -1 || c->adaptive > 1) return CF_ERR_INVALID_ARG;
  if (c->pdl < -1 || c->pdl > 1) return CF_ERR_INVALID_ARG;
  if (c->max_stages < 0 || c->max_stages == 1 || c->max_stages > kMaxStages)
    return CF_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return CF_ERR_UNSUPPORTED;
  if (N != 0 && N > c->head_dim / 4) return CF_ERR_INVALID_ARG;
  if (N != 0 && ((c->hidden / N) * esize(c->dtype)) % 16 != 0) return CF_ERR_INVALID_ARG;
  // The 4D KV map's extents must fit its index range.
  if ((long long)c->s_max * c->n_kv_heads * c->head_dim > (1LL << 40)) return CF_ERR_INVALID_ARG;
  return CF_OK;
}

bool encode(CUtensorMap* m, int dtype, int rank, const void* base, const uint64_t* dims,
            const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128 = false) {
  uint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(m, tm_type(dtype), (cuuint32_t)rank, const_cast<void*>(base),
                        (const cuuint64_t*)dims, (const cuuint64_t*)strides_bytes,
                        (const cuuint32_t*)box, (const cuuint32_t*)estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

// Raise the function's dynamic shared-memory limit to `bytes` (never lower
// it: the attribute is per function, shared by every handle) and allow
// clusters above 8 blocks when needed.
int prepare_function(const void* fn, int bytes, int N) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  cudaFuncAttributes cur;
  if (cudaFuncGetAttributes(&cur, fn) != cudaSuccess) return CF_ERR_CUDA;
  if (cur.maxDynamicSharedSizeBytes < bytes &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return CF_ERR_CUDA;
  if (N > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                   cudaSuccess)
    return CF_ERR_CLUSTER;
  return CF_OK;
}

// Clusters of N blocks with `smem` bytes each that can be resident at once
// (0 when none, or on error).
int resident_clusters(const void* fn, int N, int smem) {
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = N;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(N, 1, 1);
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

// Whether c takes the batched row-split kernel: 16-bit storage and either a
// batch of at least 16 rows (by default) or an explicit rows_per_block or
// batch tile of 16 or more.
bool wants_rows(const cf_config& c) {
  if (c.dtype == CF_F32) return false;
  if (c.rows_per_block > 0 || c.batch_tile >= 16) return true;
  return c.batch_tile == 0 && c.max_batch >= 16;
}

// The batched row-split instance for c with its plan, or nullptr.  Among the
// instances whose plan fits, prefer those whose whole grid is resident at
// once (one wave) and, among them, the one with the most blocks (more SMs
// streaming), then the larger batch tile (fewer weight reads); if no grid
// fits in one wave, the fewest waves, then the larger batch tile.
const KernelEntry* pick_rows_entry(const cf_config& c, int stage_req, const cudaDeviceProp& prop,
                                   Plan& pl) {
  if (!wants_rows(c)) return nullptr;
  const int D = c.head_dim, G = c.n_q_heads / c.n_kv_heads;
  const KernelEntry* e0 = nullptr;
  const KernelEntry* e1 = nullptr;
  const int n0 = registry_rows(&e0);
  const int n = n0 + registry_rows_sweep(&e1);
  const KernelEntry* best = nullptr;
  long long best_waves = 0, best_blocks = 0;
  for (int i = 0; i < n; ++i) {
    const KernelEntry& k = i < n0 ? e0[i] : e1[i - n0];
    if (k.dtype != c.dtype || k.D != D || k.G != G) continue;
    if (k.explicit_only && !(c.batch_tile == k.BT && c.rows_per_block == k.RPC)) continue;
    if (c.batch_tile > 0 && k.BT != c.batch_tile) continue;
    if (c.rows_per_block > 0 && k.RPC != c.rows_per_block) continue;
    if (c.batch_tile == 0 && k.BT > std::max(4, c.max_batch)) continue;
    Plan trial;
    if (!make_plan_rows(c, k.BT, k.RPC, stage_req, prop, trial)) continue;
    if (prepare_function(k.fn, trial.L.total, trial.N) != CF_OK) continue;
    const int resident = resident_clusters(k.fn, trial.N, trial.L.total);
    if (resident <= 0) continue;
    const long long clusters = (long long)c.n_kv_heads * ((c.max_batch + k.BT - 1) / k.BT);
    const long long waves = (clusters + resident - 1) / resident;
    const long long blocks = std::min(clusters, (long long)resident) * trial.N;
    bool better = best == nullptr;
    if (!better) {
      const bool one = waves == 1, best_one = best_waves == 1;
      if (one != best_one) better = one;
      else if (one) better = blocks > best_blocks || (blocks == best_blocks && k.BT > best->BT);
      else better = waves < best_waves || (waves == best_waves && k.BT > best->BT);
    }
    if (better) {
      best = &k;
      pl = trial;
      best_waves = waves;
      best_blocks = blocks;
    }
  }
  return best;
}

// Kernel instance, launch shape and shared-memory plan of config c on the
// current device, written into h (all but the workspace pointers).
int plan_handle(const cf_config& c, cf_handle& h) {
  const int D = c.head_dim, G = c.n_q_heads / c.n_kv_heads;
  if (!get_encode()) return CF_ERR_CUDA;
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess) return CF_ERR_CUDA;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return CF_ERR_CUDA;
  const int stage_req = c.stage_bytes ? c.stage_bytes : 32768;
  Plan pl;
  // batched kernel: 64 KB stages for head_dim 128 (fewer, larger TMA boxes;
  // measured faster on the Llama-3 GQA layer), 32 KB otherwise
  const int stage_rows = c.stage_bytes ? c.stage_bytes : (D >= 128 ? 65536 : 32768);
  const KernelEntry* ke = pick_rows_entry(c, stage_rows, prop, pl);
  if (ke == nullptr) {
    // an explicit batched request with no fitting instance is an error; a
    // default choice falls back to the sequence-split kernel
    if (c.batch_tile >= 16 || c.rows_per_block > 0) return CF_ERR_UNSUPPORTED;
    // Batch tile: requested, else the largest compiled one <= max_batch.
    int BT = c.batch_tile;
    if (BT == 0) {
      BT = best_batch_tile(c.dtype, D, G, std::min(c.max_batch, 4));
      if (G > 1) BT = best_batch_tile(c.dtype, D, G, std::min(c.max_batch, 2));
    }
    if (BT <= 0) return CF_ERR_UNSUPPORTED;
    ke = find_entry(c.dtype, D, G, BT);
    if (ke == nullptr) return CF_ERR_UNSUPPORTED;
    // Cluster size: requested, else the smallest power of two >= 2 that gives
    // about two blocks per SM over the whole grid (capped by head_dim/4, by
    // the hidden size's 16-byte column bands and by a K band of at least 64
    // rows per block), then halved while the grid's clusters would not all be
    // resident at once (measured: a second wave costs more than a smaller
    // cluster -- the GQA layer at batch 1 runs 1.3x faster with 8 clusters of
    // 8 than with 8 clusters of 16, of which only 7 fit).
    const int clusters = c.n_kv_heads * ((c.max_batch + BT - 1) / BT);
    int N = c.cluster_size;
    if (N == 0) {
      N = 2;
      while (N < 16 && N * 2 <= D / 4 && ((c.hidden / (N * 2)) * esize(c.dtype)) % 16 == 0 &&
             c.hidden / (N * 2) >= 64 &&
             (long long)clusters * N * 2 <= 2LL * prop.multiProcessorCount)
        N *= 2;
    }
    if (N > D / 4 || ((c.hidden / N) * esize(c.dtype)) % 16 != 0) return CF_ERR_INVALID_ARG;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, ke->fn) != cudaSuccess) return CF_ERR_CUDA;
    for (;;) {
      int cps = c.ctas_per_sm;
      if (cps == 0) {
        // registers are allocated per thread in multiples of 8
        const int regs = (fa.numRegs + 7) / 8 * 8;
        const bool regs_ok = regs * kThreads * 2 <= prop.regsPerMultiprocessor;
        cps = (regs_ok && (long long)clusters * N > prop.multiProcessorCount) ? 2 : 1;
      }
      // When the weights dominate the stream (the cached K/V of every row at
      // s_max below half the W_qkv bytes), 48 KB stages: the W_qkv phase then
      // moves 64-row tiles, fewer stages through each SM's TMA unit, which
      // bounds the SMs that hold two blocks; K/V and W_o tiles stay 32 KB.
      // Measured: Llama-2 1K layer 32.78 -> 32.31 us; a 16K-position layer
      // keeps 32 KB stages (48 KB: 2145 -> 2154 us per 32-layer step).
      const bool weight_bound =
          (long long)c.s_max * 2 * BT < (long long)c.hidden * (G + 2) / 2;
      const int req = (c.stage_bytes == 0 && weight_bound) ? 49152 : stage_req;
      if (!make_plan(c, N, BT, req, cps, prop, pl) &&
          !(cps == 2 && make_plan(c, N, BT, req, 1, prop, pl)) &&
          !(req != stage_req && make_plan(c, N, BT, stage_req, cps, prop, pl)))
        return CF_ERR_UNSUPPORTED;
      if (c.cluster_size != 0 || N <= 2) break;
      const int rc = prepare_function(ke->fn, pl.L.total, N);
      if (rc != CF_OK) return rc;
      if (resident_clusters(ke->fn, N, pl.L.total) >= clusters) break;
      N /= 2;
    }
  }
  const int N = pl.N;
  {
    const int rc = prepare_function(ke->fn, pl.L.total, N);
    if (rc != CF_OK) return rc;
  }
  const int nclusters = resident_clusters(ke->fn, N, pl.L.total);
  if (nclusters <= 0) return CF_ERR_CLUSTER;
  h.cfg = c;
  h.device = dev;
  h.sm_count = prop.multiProcessorCount;
  h.nslots = 1;
  h.slots[0] = PlanSlot();
  h.slots[0].cap = c.max_batch;
  h.slots[0].plan = pl;
  h.slots[0].fn = ke->fn;
  h.slots[0].max_active_clusters = nclusters;
  h.pdl = c.pdl != -1;
  for (int i = 0; i < 64; ++i) {
    // turns per position: theta^(-2i/d) / (2 pi), split into hi + lo floats
    const double two_pi = 6.283185307179586476925286766559;
    const double rate = (i < D / 2) ? std::pow((double)c.rope_theta, -2.0 * i / (double)D) / two_pi
                                    : 0.0;
    h.turn_hi[i] = (float)rate;
    h.turn_lo[i] = (float)(rate - (double)h.turn_hi[i]);
  }
  return CF_OK;
}

}  // namespace

extern "C" {

const char* cf_strerror(int code) {
  switch (code) {
    case CF_OK: return "ok";
    case CF_ERR_INVALID_ARG: return "invalid argument";
    case CF_ERR_UNSUPPORTED: return "unsupported configuration (no kernel built for it)";
    case CF_ERR_ALIAS: return "output overlaps an input";
    case CF_ERR_CLUSTER: return "thread-block cluster shape cannot be resident on this device";
    case CF_ERR_CUDA: return "CUDA runtime or driver error";
    case CF_ERR_DEVICE_POS_RANGE: return "a positions[] value was outside [0, s_max)";
    case CF_ERR_DEVICE_TIMEOUT: return "an in-kernel wait timed out";
    default: return "unknown error code";
  }
}

int cf_create(const cf_config* cfg, cf_handle** out) {
  if (out == nullptr) return CF_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc != CF_OK) return rc;
  const cf_config c = *cfg;
  cf_handle* h = new (std::nothrow) cf_handle();
  if (h == nullptr) return CF_ERR_CUDA;
  rc = plan_handle(c, *h);
  if (rc != CF_OK) {
    delete h;
    return rc;
  }
  // Runtime choice per batch: unless the launch shape was fixed by the
  // caller, also plan for batch caps 1, 2, 4 and 8 below max_batch and keep
  // each plan that differs from the next larger one.  Measured (one GB300):
  // a handle for the 64-row, head_dim-64 MHA layer runs 1-, 2-, 4- and 8-row
  // calls 2.2-2.8x faster on the sequence-split plans of those caps than on
  // its 64-row tile; for GQA (several query heads per KV head) the batched
  // 4-row-tile plan of the Llama-3 layer beat the sequence-split plans at
  // 2-8 rows by 1.4-3.1x and tied at one row, so GQA handles keep one plan.
  const bool fixed_shape = c.cluster_size || c.batch_tile || c.stage_bytes || c.ctas_per_sm ||
                           c.rows_per_block || c.max_stages || c.adaptive == -1;
  if (!fixed_shape && c.n_q_heads == c.n_kv_heads) {
    PlanSlot top = h->slots[0];
    PlanSlot found[kMaxPlanSlots];
    int nfound = 0;
    for (int cap = 1; cap < c.max_batch && cap <= 8 && nfound < kMaxPlanSlots - 1; cap *= 2) {
      cf_config cc = c;
      cc.max_batch = cap;
      cf_handle tmp;
      if (plan_handle(cc, tmp) != CF_OK) continue;
      found[nfound++] = tmp.slots[0];
    }
    // keep a slot only if it differs from the next kept larger one
    PlanSlot kept[kMaxPlanSlots];
    int nk = 0;
    kept[nk++] = top;
    for (int i = nfound - 1; i >= 0; --i) {
      const PlanSlot& up = kept[nk - 1];
      const bool same = found[i].fn == up.fn && found[i].plan.N == up.plan.N &&
                        found[i].plan.BT == up.plan.BT && found[i].plan.RPC == up.plan.RPC &&
                        found[i].plan.L.total == up.plan.L.total;
      if (!same) kept[nk++] = found[i];  // else the larger slot serves these batches
    }
    h->nslots = nk;
    for (int i = 0; i < nk; ++i) h->slots[i] = kept[nk - 1 - i];
  }
  const size_t acc_bytes = (size_t)c.max_batch * c.hidden * sizeof(float);
  size_t cnt_slots = 0;
  for (int i = 0; i < h->nslots; ++i)
    cnt_slots = std::max(cnt_slots, counter_slots(h->slots[i].plan, h->slots[i].cap));
  const size_t cnt_bytes = cnt_slots * sizeof(int);
  const size_t total = acc_bytes + cnt_bytes + 256;
  if (cudaMalloc(&h->ws, total) != cudaSuccess) {
    delete h;
    return CF_ERR_CUDA;
  }
  if (cudaMemset(h->ws, 0, total) != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return CF_ERR_CUDA;
  }
  h->acc = static_cast<float*>(h->ws);
  h->counters = reinterpret_cast<int*>(static_cast<char*>(h->ws) + acc_bytes);
  h->errflag = reinterpret_cast<int*>(static_cast<char*>(h->ws) + acc_bytes + cnt_bytes);
  // Workspace of the three-kernel path (cf_decode_attn_block_unfused).
  {
    const int D = c.head_dim, G = c.n_q_heads / c.n_kv_heads, H = c.hidden;
    const int Cq = (c.n_q_heads + 2 * c.n_kv_heads) * D;
    const int sms = h->sm_count;
    // about four blocks per SM in each of the three kernels
    int NS = (4 * sms + c.max_batch * c.n_kv_heads - 1) / (c.max_batch * c.n_kv_heads);
    NS = std::max(1, std::min(32, NS));
    const int nbt = c.max_batch == 1 ? 1 : (c.max_batch + 7) / 8;
    auto splits = [&](int bands, int K) {
      int ks = 1;
      while (ks < 16 && bands * nbt * ks * 2 <= 4 * sms && K % (ks * 2 * 64) == 0) ks *= 2;
      return ks;
    };
    h->uf_NS = NS;
    h->uf_KS1 = splits(Cq % 128 == 0 ? Cq / 128 : Cq / 64, H);
    h->uf_KS = splits(H % 128 == 0 ? H / 128 : H / 64, c.n_q_heads * D);
    const size_t y_b = (size_t)c.max_batch * Cq * 4;
    const size_t part_b = (size_t)c.max_batch * c.n_kv_heads * NS * G * (D + 4) * 4;
    const size_t o_b = (size_t)c.max_batch * c.n_q_heads * D * 4;
    const size_t ca_b = (size_t)c.max_batch * c.n_kv_heads * 4;
    const size_t co_b = (size_t)c.max_batch * (H / 64) * 4;
    const size_t ri_b = ((size_t)c.max_batch * 4 + 255) / 256 * 256;
    const size_t tot = y_b + part_b + o_b + ca_b + co_b + ri_b + 256;
    if (cudaMalloc(&h->uf_ws, tot) != cudaSuccess || cudaMemset(h->uf_ws, 0, tot) != cudaSuccess) {
      if (h->uf_ws) cudaFree(h->uf_ws);
      cudaFree(h->ws);
      delete h;
      return CF_ERR_CUDA;
    }
    char* w = static_cast<char*>(h->uf_ws);
    h->uf_y = reinterpret_cast<float*>(w);
    h->uf_part = reinterpret_cast<float*>(w + y_b);
    h->uf_o32 = reinterpret_cast<float*>(w + y_b + part_b);
    h->uf_cnt_attn = reinterpret_cast<int*>(w + y_b + part_b + o_b);
    h->uf_cnt_out = reinterpret_cast<int*>(w + y_b + part_b + o_b + ca_b);
    h->uf_rinv = reinterpret_cast<float*>(w + y_b + part_b + o_b + ca_b + co_b);
  }
  *out = h;
  return CF_OK;
}

int cf_decode_attn_block(cf_handle* h, int32_t batch, const void* hidden_states,
                         const void* ln_weight, const void* w_qkv, const void* w_o,
                         void* k_cache, void* v_cache, const int32_t* positions, void* out,
                         void* stream) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  const cf_config& c = h->cfg;
  if (batch < 0 || batch > c.max_batch) return CF_ERR_INVALID_ARG;
  if (batch == 0) return CF_OK;
  const void* ptrs[] = {hidden_states, ln_weight, w_qkv, w_o, k_cache, v_cache, positions, out};
  for (const void* p : ptrs)
    if (p == nullptr || ((uintptr_t)p & 15u) != 0) return CF_ERR_INVALID_ARG;

  const int es = esize(c.dtype), D = c.head_dim, H = c.hidden;
  const int nq = c.n_q_heads, nkv = c.n_kv_heads, S = c.s_max;
  const int C = (nq + 2 * nkv) * D;
  const size_t out_bytes = (size_t)batch * H * es;
  const size_t cache_bytes = (size_t)batch * S * nkv * D * es;
  if (overlaps(out, out_bytes, hidden_states, (size_t)batch * H * es) ||
      overlaps(out, out_bytes, ln_weight, (size_t)H * es) ||
      overlaps(out, out_bytes, w_qkv, (size_t)H * C * es) ||
      overlaps(out, out_bytes, w_o, (size_t)nq * D * H * es) ||
      overlaps(out, out_bytes, k_cache, cache_bytes) ||
      overlaps(out, out_bytes, v_cache, cache_bytes) ||
      overlaps(out, out_bytes, positions, (size_t)batch * 4))
    return CF_ERR_ALIAS;

  PlanSlot& ps = const_cast<PlanSlot&>(h->slot_for(batch));
  const Plan& pl = ps.plan;
  KParams kp;
  std::memset(&kp, 0, sizeof(kp));
  // Tensor maps (encoded on the host, cached per pointer and extent).
  auto get_map = [&](MapCache& mc, const void* base, int key, int rank, const uint64_t* dims,
                     const uint64_t* str, const uint32_t* box, bool swz,
                     CUtensorMap& dst) -> bool {
    const CUtensorMap* m = mc.find(base, key);
    if (!m) {
      CUtensorMap* n = mc.insert(base, key);
      if (!encode(n, c.dtype, rank, base, dims, str, box, swz)) {
        mc.ptr[(mc.next + MapCache::kSlots - 1) % MapCache::kSlots] = nullptr;
        return false;
      }
      m = n;
    }
    dst = *m;
    return true;
  };
  // The batched kernel reads weights as 64-column boxes (128 bytes) with the
  // 128-byte swizzle, and x as [BT x Rw] tiles.
  const bool rows = pl.mode == 1;
  {
    const uint64_t dims[2] = {(uint64_t)C, (uint64_t)H};
    const uint64_t str[1] = {(uint64_t)C * es};
    const uint32_t box[2] = {(uint32_t)(rows ? 64 : D), (uint32_t)pl.Rw};
    if (!get_map(ps.m_wqkv, w_qkv, 0, 2, dims, str, box, rows, kp.tm_wqkv)) return CF_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {(uint64_t)H, (uint64_t)nq * D};
    const uint64_t str[1] = {(uint64_t)H * es};
    const uint32_t box[2] = {(uint32_t)(rows ? 64 : pl.Co), (uint32_t)pl.Ro};
    if (!get_map(ps.m_wo, w_o, 0, 2, dims, str, box, rows, kp.tm_wo)) return CF_ERR_CUDA;
  }
  for (int which = 0; which < 2; ++which) {
    const void* base = which == 0 ? k_cache : v_cache;
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)nkv, (uint64_t)S, (uint64_t)batch};
    const uint64_t str[3] = {(uint64_t)D * es, (uint64_t)nkv * D * es, (uint64_t)S * nkv * D * es};
    const uint32_t box[4] = {(uint32_t)(rows ? 64 : D), 1u, (uint32_t)pl.Rt, 1u};
    if (!get_map(which == 0 ? ps.m_k : ps.m_v, base, batch, 4, dims, str, box, rows,
                 which == 0 ? kp.tm_k : kp.tm_v))
      return CF_ERR_CUDA;
  }
  if (rows) {
    const uint64_t dims[2] = {(uint64_t)H, (uint64_t)batch};
    const uint64_t str[1] = {(uint64_t)H * es};
    const uint32_t box[2] = {(uint32_t)pl.Rw, (uint32_t)pl.BT};
    if (!get_map(ps.m_x, hidden_states, batch, 2, dims, str, box, false, kp.tm_x))
      return CF_ERR_CUDA;
  }

  kp.hidden = hidden_states;
  kp.ln_w = ln_weight;
  kp.k_cache = k_cache;
  kp.v_cache = v_cache;
  kp.positions = positions;
  kp.out = out;
  kp.acc = h->acc;
  kp.counters = h->counters;
  kp.errflag = h->errflag;
  kp.dbg = h->dbg;
  kp.timeline = h->timeline;
  // The last min(8, nkv) blocks of a (tile, band) share its finalize when the
  // whole grid is resident at once (the earlier ones wait for the later).
  const long long grid_clusters = (long long)nkv * ((batch + pl.BT - 1) / pl.BT);
  kp.fin_split =
      (rows && pl.BT >= 16 && grid_clusters <= ps.max_active_clusters) ? std::min(8, nkv) : 1;
  kp.B = batch;
  kp.H = H;
  kp.nq = nq;
  kp.nkv = nkv;
  kp.S = S;
  kp.N = pl.N;
  kp.nbt = (batch + pl.BT - 1) / pl.BT;
  kp.Rw = pl.Rw;
  kp.Rt = pl.Rt;
  kp.Ro = pl.Ro;
  kp.Co = pl.Co;
  kp.stages = pl.stages;
  kp.stage_bytes = pl.stage_bytes;
  kp.eps = c.rms_eps;
  kp.qk_scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  kp.L = pl.L;
  for (int i = 0; i < 64; ++i) {
    kp.turn_hi[i] = h->turn_hi[i];
    kp.turn_lo[i] = h->turn_lo[i];
  }

  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.N;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // Programmatic dependent launch: the kernel may be scheduled while the
  // previous kernel on the stream drains; it waits for that kernel's
  // completion (griddepcontrol.wait) before reading any global memory.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = dim3(pl.N * nkv * kp.nbt, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = pl.L.total;
  lc.stream = static_cast<cudaStream_t>(stream);
  lc.attrs = attr;
  lc.numAttrs = h->pdl ? 2 : 1;
  void* args[] = {&kp};
  if (cudaLaunchKernelExC(&lc, ps.fn, args) != cudaSuccess) {
    cudaGetLastError();
    return CF_ERR_CUDA;
  }
  return CF_OK;
}

int cf_get_status(cf_handle* h) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  int flag = 0;
  if (cudaMemcpy(&flag, h->errflag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CF_ERR_CUDA;
  if (flag != 0 && cudaMemset(h->errflag, 0, sizeof(int)) != cudaSuccess) return CF_ERR_CUDA;
  if (flag & kDevErrTimeout) return CF_ERR_DEVICE_TIMEOUT;
  if (flag & kDevErrPosRange) return CF_ERR_DEVICE_POS_RANGE;
  return CF_OK;
}

int cf_set_debug(cf_handle* h, float* dbg) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  h->dbg = dbg;
  return CF_OK;
}

int cf_set_timeline(cf_handle* h, unsigned long long* stamps) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  h->timeline = stamps;
  return CF_OK;
}

int cf_get_launch_info(const cf_handle* h, cf_launch_info* info) {
  if (h == nullptr) return CF_ERR_INVALID_ARG;
  return cf_get_launch_info_batch(h, h->cfg.max_batch, info);
}

int cf_get_launch_info_batch(const cf_handle* h, int32_t batch, cf_launch_info* info) {
  if (h == nullptr || info == nullptr || batch < 1 || batch > h->cfg.max_batch)
    return CF_ERR_INVALID_ARG;
  const PlanSlot& ps = h->slot_for(batch);
  const Plan& pl = ps.plan;
  info->cluster_size = pl.N;
  info->batch_tile = pl.BT;
  info->group = pl.G;
  info->rows_per_wtile = pl.Rw;
  info->pos_per_ktile = pl.Rt;
  info->wo_rows_per_tile = pl.Ro;
  info->wo_cols_per_tile = pl.Co;
  info->stages = pl.stages;
  info->stage_bytes = pl.stage_bytes;
  info->smem_bytes = pl.L.total;
  info->threads = kThreads;
  info->max_active_clusters = ps.max_active_clusters;
  info->sm_count = h->sm_count;
  info->mode = pl.mode;
  info->rows_per_block = pl.RPC;
  return CF_OK;
}

int cf_decode_attn_block_unfused(cf_handle* h, int32_t batch, const void* hidden_states,
                                 const void* ln_weight, const void* w_qkv, const void* w_o,
                                 void* k_cache, void* v_cache, const int32_t* positions, void* out,
                                 void* stream) {
  if (h == nullptr || h->uf_ws == nullptr) return CF_ERR_INVALID_ARG;
  const cf_config& c = h->cfg;
  if (batch < 0 || batch > c.max_batch) return CF_ERR_INVALID_ARG;
  if (batch == 0) return CF_OK;
  const void* ptrs[] = {hidden_states, ln_weight, w_qkv, w_o, k_cache, v_cache, positions, out};
  for (const void* p : ptrs)
    if (p == nullptr || ((uintptr_t)p & 15u) != 0) return CF_ERR_INVALID_ARG;
  const int es = esize(c.dtype), D = c.head_dim, H = c.hidden;
  const int nq = c.n_q_heads, nkv = c.n_kv_heads, S = c.s_max;
  const size_t out_bytes = (size_t)batch * H * es;
  const size_t cache_bytes = (size_t)batch * S * nkv * D * es;
  if (overlaps(out, out_bytes, hidden_states, (size_t)batch * H * es) ||
      overlaps(out, out_bytes, ln_weight, (size_t)H * es) ||
      overlaps(out, out_bytes, w_qkv, (size_t)H * (nq + 2 * nkv) * D * es) ||
      overlaps(out, out_bytes, w_o, (size_t)nq * D * H * es) ||
      overlaps(out, out_bytes, k_cache, cache_bytes) ||
      overlaps(out, out_bytes, v_cache, cache_bytes) ||
      overlaps(out, out_bytes, positions, (size_t)batch * 4))
    return CF_ERR_ALIAS;
  UfParams p;
  p.hidden = hidden_states;
  p.ln_w = ln_weight;
  p.w_qkv = w_qkv;
  p.w_o = w_o;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.positions = positions;
  p.out = out;
  p.y = h->uf_y;
  p.part = h->uf_part;
  p.o32 = h->uf_o32;
  p.rinv = h->uf_rinv;
  p.acc = h->acc;
  p.cnt_attn = h->uf_cnt_attn;
  p.cnt_out = h->uf_cnt_out;
  p.errflag = h->errflag;
  p.B = batch;
  p.H = H;
  p.nq = nq;
  p.nkv = nkv;
  p.D = D;
  p.S = S;
  p.NS = h->uf_NS;
  p.KS = h->uf_KS;
  p.KS1 = h->uf_KS1;
  p.eps = c.rms_eps;
  p.qk_scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  for (int i = 0; i < 64; ++i) {
    p.turn_hi[i] = h->turn_hi[i];
    p.turn_lo[i] = h->turn_lo[i];
  }
  return unfused_launch(p, c.dtype, nq / nkv, static_cast<cudaStream_t>(stream));
}

void cf_destroy(cf_handle* h) {
  if (h == nullptr) return;
  if (h->uf_ws) cudaFree(h->uf_ws);
  if (h->ws) cudaFree(h->ws);
  delete h;
}

}  // extern "C"

// ===========================================================================
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc at all: code running inside a CUDA
// graph capture region that must not allocate, custom allocators that own all
// device memory, or embeddings in runtimes that forbid allocation after
// start-up.  cf_decode_attn_block_noalloc serves them: it needs no handle, and
// its scratch -- the fp32 output accumulator, the completion counters and the
// error flag that cf_create would otherwise allocate -- lives in the
// file-scope device array below, which every GPU that loads this library
// holds until the process exits.  Its planning state lives in static host
// storage, one slot per device, so no host heap is touched either.
// ===========================================================================
namespace {

constexpr size_t kNoAllocAccFloats = size_t(1) << 19;  // 2 MiB: batch * hidden <= 524288
constexpr size_t kNoAllocCounters = 8192;
constexpr size_t kNoAllocBytes = kNoAllocAccFloats * 4 + kNoAllocCounters * 4 + 256;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

struct NoAllocSlot {
  bool ready = false;        // device address of the scratch obtained
  unsigned char* scratch = nullptr;
  bool planned = false;      // `h` prepared for `cfg`
  cf_config cfg;
  cf_handle h;
};
NoAllocSlot g_noalloc[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

// The planning half of cf_create (kernel instance, cluster size, shared-memory
// plan, function attributes) with the handle's workspace pointed at the
// static scratch instead of a fresh allocation.
int noalloc_prepare(const cf_config& c, unsigned char* scratch, cf_handle& h) {
  const int rc = plan_handle(c, h);
  if (rc != CF_OK) return rc;
  if (counter_slots(h.main().plan, c.max_batch) > kNoAllocCounters)
    return CF_ERR_INVALID_ARG;
  h.ws = nullptr;  // nothing to free: the workspace is the static scratch
  h.acc = reinterpret_cast<float*>(scratch);
  h.counters = reinterpret_cast<int*>(scratch + kNoAllocAccFloats * 4);
  h.errflag = reinterpret_cast<int*>(scratch + kNoAllocAccFloats * 4 + kNoAllocCounters * 4);
  h.dbg = nullptr;
  h.timeline = nullptr;
  PlanSlot& ps = h.main();
  for (MapCache* mc : {&ps.m_wqkv, &ps.m_wo, &ps.m_k, &ps.m_v, &ps.m_x}) {
    for (int i = 0; i < MapCache::kSlots; ++i) mc->ptr[i] = nullptr;
    mc->next = 0;
  }
  return CF_OK;
}

}  // namespace

extern "C" int cf_decode_attn_block_noalloc(const cf_config* cfg, int32_t batch,
                                            const void* hidden_states, const void* ln_weight,
                                            const void* w_qkv, const void* w_o, void* k_cache,
                                            void* v_cache, const int32_t* positions, void* out,
                                            void* stream) {
  int rc = validate_config(cfg);
  if (rc != CF_OK) return rc;
  if (batch < 0 || batch > cfg->max_batch) return CF_ERR_INVALID_ARG;
  if ((size_t)cfg->max_batch * (size_t)cfg->hidden > kNoAllocAccFloats) return CF_ERR_INVALID_ARG;
  if (batch == 0) return CF_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CF_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return CF_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocSlot& s = g_noalloc[dev];
  if (!s.ready) {
    // Once per device, with that device current: the host-side name of the
    // array is only a stand-in, so fetch its real device address.
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return CF_ERR_CUDA;
    }
    s.scratch = static_cast<unsigned char*>(p);
    s.ready = true;
  }
  if (!s.planned || std::memcmp(&s.cfg, cfg, sizeof(cf_config)) != 0) {
    s.planned = false;
    rc = noalloc_prepare(*cfg, s.scratch, s.h);
    if (rc != CF_OK) return rc;
    s.cfg = *cfg;
    s.planned = true;
  }
  // The kernel leaves the accumulator and counters at zero, but the array
  // keeps whatever the previous call left (e.g. one stopped by an error), so
  // the regions this call uses are cleared first, on the same stream.  The
  // error word is not: it collects the device-detected errors of every call
  // until cf_noalloc_get_status reads and clears it.
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t acc_bytes = (size_t)batch * cfg->hidden * sizeof(float);
  const size_t cnt_bytes = counter_slots(s.h.main().plan, batch) * sizeof(int);
  if (cudaMemsetAsync(s.h.acc, 0, acc_bytes, st) != cudaSuccess ||
      cudaMemsetAsync(s.h.counters, 0, cnt_bytes, st) != cudaSuccess) {
    cudaGetLastError();
    return CF_ERR_CUDA;
  }
  return cf_decode_attn_block(&s.h, batch, hidden_states, ln_weight, w_qkv, w_o, k_cache, v_cache,
                              positions, out, stream);
}

extern "C" int cf_noalloc_get_status(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CF_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return CF_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocSlot& s = g_noalloc[dev];
  if (!s.ready) return CF_OK;  // no call has run on this device
  int* flag_dev =
      reinterpret_cast<int*>(s.scratch + kNoAllocAccFloats * 4 + kNoAllocCounters * 4);
  int flag = 0;
  if (cudaMemcpy(&flag, flag_dev, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CF_ERR_CUDA;
  if (flag != 0 && cudaMemset(flag_dev, 0, sizeof(int)) != cudaSuccess) return CF_ERR_CUDA;
  if (flag & kDevErrTimeout) return CF_ERR_DEVICE_TIMEOUT;
  if (flag & kDevErrPosRange) return CF_ERR_DEVICE_POS_RANGE;
  return CF_OK;
}
