/*
 * cf.h -- C ABI of the GB300-native fused decode attention block.
 *
 * One call runs, for every batch row b, the single-token decode step of a
 * transformer attention block as ONE fused sm_103a kernel launch:
 *
 *   n   = RMSNorm(x_b)                           [LNA §三 stage 1]
 *   y   = n . W_qkv   (merged QKV projection)    [CF §5.1], [LNA §三 stage 2]
 *   q_h, k_g <- RoPE(., p_b)  (rotate-half)      [LNA §三]
 *   k_cache[b,p_b,g,:] = k_g, v_cache[b,p_b,g,:] = v_g   [LNA §三 stage 3]
 *   o_h = softmax(q_h K_g^T / sqrt(d)) V_g over positions 0..p_b,
 *         g = h / (nq/nkv)                        [CF §3.2], [LNA §三 GQA]
 *   out_b = x_b + concat_h(o_h) . W_o             [CF §3.2], [LNA §一]
 *
 * Each (KV head, batch tile) maps to one thread-block cluster [CF §3.2
 * 空间映射策略]; the cluster's blocks split the hidden (reduction) dimension
 * of the projections, the KV sequence of the attention and the output
 * columns of the O projection, and exchange partial results over distributed
 * shared memory with the ClusterReduce / ClusterGather primitives [CF §3.1.1,
 * §3.1.2].  The per-head output contributions are merged with global atomics
 * [CF §3.2 原子写合并].
 *
 * Pages cited by title and section:
 *   [CF]  "ClusterFusion框架深度解析：LLM推理优化的集群级通信革命" (devpress.csdn.net)
 *   [LNA] "大模型推理中的算子融合优化：LayerNorm + Attention 的 CUDA Kernel 手写与验证"
 *         (asdsk.com)
 *
 * Conventions for every function:
 *   - returns CF_OK (0) or a negative CF_ERR_* code; no exception crosses
 *     the ABI; nothing is printed;
 *   - "device" pointers are CUDA device (or managed) pointers on the device
 *     that was current at cf_create; the caller owns all tensors;
 *   - all tensors are dense, row-major, in the handle's storage dtype, and
 *     16-byte aligned.
 */
#ifndef CF_H
#define CF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CF_OK 0
#define CF_ERR_INVALID_ARG (-1)      /* bad pointer, size or config value      */
#define CF_ERR_UNSUPPORTED (-2)      /* valid but not built (dtype/d/group/..) */
#define CF_ERR_ALIAS (-3)            /* out overlaps an input                  */
#define CF_ERR_CLUSTER (-4)          /* the cluster shape cannot be resident   */
#define CF_ERR_CUDA (-5)             /* a CUDA runtime/driver call failed      */
#define CF_ERR_DEVICE_POS_RANGE (-6) /* a positions[b] was outside [0, S_max)  */
#define CF_ERR_DEVICE_TIMEOUT (-7)   /* a bounded in-kernel wait expired       */

typedef enum { CF_F32 = 0, CF_F16 = 1, CF_BF16 = 2 } cf_dtype;

/* Problem statement [CF §3.2 fused_qkv_attention_out], [LNA §三 kernel
 * signature].  Zero in a tuning field selects the measured default. */
typedef struct cf_config {
  int32_t hidden;       /* H; multiple of 64                                  */
  int32_t n_q_heads;    /* nq                                                 */
  int32_t n_kv_heads;   /* nkv; nq % nkv == 0 (nkv == nq is MHA)              */
  int32_t head_dim;     /* d: 64 or 128                                       */
  int32_t max_batch;    /* upper bound on `batch` in cf_decode_attn_block     */
  int32_t s_max;        /* S: KV-cache capacity per sequence                  */
  float rope_theta;     /* RoPE base, e.g. 1e4 or 5e5                         */
  float rms_eps;        /* RMSNorm eps (inside the square root)               */
  int32_t dtype;        /* cf_dtype: storage of every tensor; math is fp32    */
  int32_t cluster_size; /* 0 = default, else 1, 2, 4, 8 or 16 blocks/cluster  */
  int32_t batch_tile;   /* 0 = default, else batch rows per cluster           */
  int32_t stage_bytes;  /* 0 = default, else bytes per shared-memory stage    */
  int32_t ctas_per_sm;  /* 0 = default, else 1 or 2 (shared-memory split)    */
  int32_t pdl;            /* programmatic dependent launch: 0 = default (on),
                             -1 = off                                         */
  int32_t max_stages;     /* 0 = as many ring stages as fit, else at most this
                             many (>= 2)                                      */
  int32_t rows_per_block; /* batched mode (batch_tile >= 16, fp16/bf16): batch
                             rows each block of a cluster owns; 0 = default  */
  int32_t adaptive;       /* 0 or 1 = default: for MHA (nq == nkv), besides the
                             max_batch plan, plan for batch caps 1, 2, 4 and 8
                             and give each call the smallest one that holds
                             its batch (kept only where the instance or shape
                             differs; off whenever a launch-shape field above
                             is set); -1 = one plan                           */
} cf_config;

typedef struct cf_handle cf_handle; /* opaque */

/* What cf_create chose (for tests, tuning and the roofline report). */
typedef struct cf_launch_info {
  int32_t cluster_size, batch_tile, group;      /* N, BT, nq/nkv            */
  int32_t rows_per_wtile, pos_per_ktile;        /* Rw, Rt                   */
  int32_t wo_rows_per_tile, wo_cols_per_tile;   /* Ro, Co                   */
  int32_t stages, stage_bytes, smem_bytes;      /* per CTA                  */
  int32_t threads, max_active_clusters, sm_count;
  int32_t mode;            /* 0: sequence-split kernel, 1: batched row-split kernel */
  int32_t rows_per_block;  /* mode 1 */
} cf_launch_info;

/* Validate cfg, pick the kernel instance and launch shape, and allocate the
 * handle's device workspace (fp32 output accumulator [max_batch, H],
 * completion counters, error flag, and the intermediates of the three-kernel
 * path below) on the current device.  On failure
 * nothing stays allocated and *out is NULL.
 * Errors: INVALID_ARG (NULL, non-positive sizes, nq % nkv != 0, odd d, H not
 * a multiple of 64, cluster_size not in {0,1,2,4,8,16} or > d/4),
 * UNSUPPORTED (d, dtype or nq/nkv without a built kernel), CLUSTER (no
 * cluster of the chosen shape fits on the device), CUDA. */
int cf_create(const cf_config* cfg, cf_handle** out);

/* Enqueue one decode step for `batch` rows on `stream` (a cudaStream_t; NULL
 * means the legacy default stream).  Asynchronous: it never synchronizes,
 * allocates or copies to the host, so it can be captured in a CUDA graph.
 *   hidden_states [batch, H]             device, read
 *   ln_weight     [H]                    device, read
 *   w_qkv         [H, (nq+2nkv)*d]       device, read; columns [Q | K | V],
 *                                        each head's d columns contiguous
 *   w_o           [nq*d, H]              device, read
 *   k_cache, v_cache [batch, S, nkv, d]  device; slot [b, positions[b]] is
 *                                        overwritten with the new token's
 *                                        (RoPE'd) key and value, nothing else
 *                                        is written
 *   positions     [batch] int32          device; the new token's slot, which
 *                                        is also its RoPE position; the
 *                                        attention covers 0..positions[b]
 *   out           [batch, H]             device, written; must not overlap
 *                                        any input (CF_ERR_ALIAS)
 * A positions[b] outside [0, S) is reported by cf_get_status as
 * CF_ERR_DEVICE_POS_RANGE; that row's cache is left untouched and its out
 * row equals its hidden row.  batch == 0 is a no-op.
 * Not thread-safe per handle: use one handle per stream. */
int cf_decode_attn_block(cf_handle* h, int32_t batch, const void* hidden_states,
                         const void* ln_weight, const void* w_qkv,
                         const void* w_o, void* k_cache, void* v_cache,
                         const int32_t* positions, void* out, void* stream);

/* The same decode step as three separate kernels with fp32 intermediates in
 * HBM -- the unfused layout [CF §1.1] compares the fused kernel with: (1)
 * (x ∘ g) · W_qkv; (2) RMSNorm scale, RoPE, KV append and split-KV attention;
 * (3) the output projection and residual.  It exists to measure the fusion
 * gain.  Same arguments, results (within the parity tolerance) and errors
 * as cf_decode_attn_block, on the same handle (whose workspace cf_create
 * sizes for it too); head_dim 64 or 128, query heads per KV head 1 or 4.
 * Asynchronous, no allocation. */
int cf_decode_attn_block_unfused(cf_handle* h, int32_t batch, const void* hidden_states,
                                 const void* ln_weight, const void* w_qkv, const void* w_o,
                                 void* k_cache, void* v_cache, const int32_t* positions,
                                 void* out, void* stream);

/* Read and clear the device-side error flag.  Call after the work has
 * finished (synchronize the stream first).  Returns CF_OK,
 * CF_ERR_DEVICE_POS_RANGE, CF_ERR_DEVICE_TIMEOUT or CF_ERR_CUDA. */
int cf_get_status(cf_handle* h);

/* Optional intermediate dump for tests: when dbg is a device float buffer of
 * batch*(2*nq*d + 2*nkv*d + H) floats, later calls write, per row b, the
 * post-RoPE q [nq*d], post-RoPE k [nkv*d], v [nkv*d], attention output o
 * [nq*d] and the pre-residual projection [H], in that order (each block
 * [batch, .]).  NULL turns it off.  Diagnostics only; not for timing. */
int cf_set_debug(cf_handle* h, float* dbg);

int cf_get_launch_info(const cf_handle* h, cf_launch_info* info);

/* What a call with `batch` rows (1 <= batch <= max_batch) launches: the plan
 * of the smallest batch cap that holds it (see cf_config.adaptive).  Errors:
 * CF_ERR_INVALID_ARG. */
int cf_get_launch_info_batch(const cf_handle* h, int32_t batch, cf_launch_info* info);

/* Static message for a CF_* code. */
const char* cf_strerror(int code);

/* Free the handle and its workspace.  NULL is a no-op. */
void cf_destroy(cf_handle* h);

/* The same decode step for callers that cannot allocate device memory at all
 * -- for example code that runs while a CUDA graph is being captured under a
 * no-allocation policy, or runtimes whose own allocator owns all device
 * memory.  The pages have no counterpart of this entry point.
 *
 * It takes the configuration directly (no handle) and calls no cudaMalloc,
 * cudaFree or other allocating routine.  Its scratch (fp32 output
 * accumulator, completion counters, error flag) is a fixed file-scope device
 * array of about 2 MiB that every GPU which loads this library keeps until
 * the process exits; calls are rejected with CF_ERR_INVALID_ARG when
 * cfg->max_batch * cfg->hidden exceeds 524288.  The first call on each
 * device looks up that array's device address (cudaGetSymbolAddress) and
 * sets kernel attributes, so make the first call on a device before any
 * stream capture.  Each call first clears, on `stream`, the part of the
 * array it uses.  All calls share the one array: calls whose work overlaps
 * on the GPU (different streams, or different host threads) race and give
 * wrong results -- serialize them.  Device-detected errors (out-of-range
 * positions, an in-kernel wait that timed out) accumulate in one word of the
 * array until cf_noalloc_get_status reads and clears it; out-of-range rows
 * are left as described for cf_decode_attn_block.  Arguments, layouts and
 * other return codes are those of cf_create + cf_decode_attn_block. */
int cf_decode_attn_block_noalloc(const cf_config* cfg, int32_t batch, const void* hidden_states,
                                 const void* ln_weight, const void* w_qkv, const void* w_o,
                                 void* k_cache, void* v_cache, const int32_t* positions,
                                 void* out, void* stream);

/* Read and clear the device-side error word that the allocation-free calls
 * on the current device share (synchronize their stream first).  Allocates
 * nothing.  Returns CF_OK (also when no such call has run on this device),
 * CF_ERR_DEVICE_POS_RANGE, CF_ERR_DEVICE_TIMEOUT, CF_ERR_UNSUPPORTED (device
 * index beyond the library's table) or CF_ERR_CUDA.  Like the calls whose
 * errors it reports, it has no counterpart on the pages. */
int cf_noalloc_get_status(void);

#ifdef __cplusplus
}
#endif

#endif /* CF_H */
