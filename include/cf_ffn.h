/*
 * cf_ffn.h -- the rest of the decoder block after the attention residual:
 * second RMSNorm, gated FFN, residual.  One kernel per call, decode batches.
 *
 * Page cited by title and section:
 *   [LNA] "大模型推理中的算子融合优化：LayerNorm + Attention 的 CUDA Kernel
 *         手写与验证" (asdsk.com), §一: the LLaMA block is RMS Norm, QKV,
 *         RoPE, attention, O projection, residual, then a second RMS Norm and
 *         the FFN.  The page names the FFN but not its inner form; the LLaMA
 *         FFN is the gated one, computed here per batch row b as
 *           n   = h_b * g2 / sqrt(mean(h_b^2) + eps)
 *           a_i = silu(Wg[i,:] . n) * (Wu[i,:] . n),   silu(z) = z/(1+e^-z)
 *           out_b[j] = h_b[j] + sum_i a_i Wd[i, j]
 *         with all products accumulated in fp32.  Batches of 1-2 rows run
 *         one CUDA-core kernel; batches of 3-64 rows run a tensor-core pair
 *         (tcgen05): gate/up, with a = silu(gate)*up kept as 16-bit hi + lo
 *         values in the handle's workspace, then the down projection and the
 *         residual (launched as a programmatic dependent of the first).
 *
 * Layouts (row-major, contiguous, device memory, every pointer 16-byte
 * aligned):
 *   hidden, out         [batch, H]   storage dtype T
 *   ln_weight (g2)      [H]          T
 *   w_gate, w_up, w_down [I, H]      T; row i holds intermediate unit i's
 *                                    weights (gate and up rows are dotted
 *                                    with n, down row i is scaled by a_i)
 *
 * Ownership: the caller owns every tensor; the handle owns its fp32
 * accumulator [max_batch, H], a completion counter and an error flag.
 *
 * Errors: every function returns CF_OK or a negative CF_ERR_* code of cf.h.
 * cf_ffn_forward is asynchronous on `stream`, never allocates, synchronizes
 * or copies to the host, and may be captured in a CUDA graph; it may start
 * streaming weights while the previous kernel on the stream drains
 * (programmatic dependent launch) and reads `hidden` only after that kernel
 * has completed.  Device-side errors (a bounded wait that expired) are
 * reported by cf_ffn_get_status.  Not thread-safe per handle.
 */
#ifndef CF_FFN_H
#define CF_FFN_H

#include <stdint.h>

#include "cf.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cf_ffn_config {
  int32_t hidden;        /* H: multiple of 8, at most 4096                  */
  int32_t intermediate;  /* I >= 1, at most 128 units per SM (19456 on a
                            152-SM part)                                    */
  int32_t max_batch;     /* upper bound on `batch`: 1..64; above 2 the
                            storage dtype is 16-bit and hidden a multiple
                            of 128                                          */
  float rms_eps;         /* eps of the second RMSNorm (inside the sqrt)     */
  int32_t dtype;         /* cf_dtype of every tensor                        */
  int32_t stage_bytes;   /* 0 = default, else bytes of weight rows per
                            shared-memory stage (>= one row)                */
} cf_ffn_config;

typedef struct cf_ffn_handle cf_ffn_handle; /* opaque */

/* Validate cfg, prepare the kernel and allocate the workspace on the current
 * device.  Errors: CF_ERR_INVALID_ARG (bad field), CF_ERR_UNSUPPORTED (H, I
 * or max_batch outside the compiled range; max_batch above 2 with fp32
 * storage or H not a multiple of 128), CF_ERR_CUDA.  Nothing is left
 * allocated on failure.  The workspace holds the fp32 accumulator
 * [max_batch, H] and, for max_batch above 2, a as 16-bit hi and lo arrays
 * [max_batch, I rounded up to 8]. */
int cf_ffn_create(const cf_ffn_config* cfg, cf_ffn_handle** out);

/* out = hidden + FFN(RMSNorm(hidden; ln_weight)) for `batch` rows (0 <= batch
 * <= max_batch; 0 does nothing).  `out` must not overlap any input
 * (CF_ERR_ALIAS).  Errors: CF_ERR_INVALID_ARG (NULL or misaligned pointer,
 * bad batch), CF_ERR_ALIAS, CF_ERR_CUDA (launch failure). */
int cf_ffn_forward(cf_ffn_handle* h, int32_t batch, const void* hidden, const void* ln_weight,
                   const void* w_gate, const void* w_up, const void* w_down, void* out,
                   void* stream);

/* Device-side error of earlier calls (after the caller synchronized the
 * stream); clears it.  CF_OK or CF_ERR_DEVICE_TIMEOUT. */
int cf_ffn_get_status(cf_ffn_handle* h);

/* Blocks per launch and rows per weight stage the handle's one- and two-row
 * kernel uses (for tests and the bench); any pointer may be NULL. */
int cf_ffn_launch_info(const cf_ffn_handle* h, int32_t* blocks, int32_t* rows_per_stage,
                       int32_t* stages);

/* Optional timeline of the tensor-core pair (diagnostics): stamps is a device
 * array of (blocks1 + blocks2) x 56 unsigned 64-bit globaltimer values (ns),
 * one row per block of the gate/up kernel, then one per block of the down
 * kernel.  Gate/up rows: [0] start, [1] the dependency wait done, [2] its
 * share of the normalized rows written, [3] the grid barrier passed, [4 + st]
 * stage st (< 48) landed at the MMA issuer, [52] every MMA complete, [53]
 * epilogue done.  Down rows: [0] start, [1] the dependency wait done,
 * [4 + st] stage st landed at the MMA issuer, [52] every MMA complete, [53]
 * the partial tile reduced into the accumulator, [54] done.  NULL turns it
 * off (the default).  Other slots stay untouched. */
int cf_ffn_set_timeline(cf_ffn_handle* h, unsigned long long* stamps);

/* Kernels a call of `batch` rows launches: returns 1 (the one- and two-row
 * kernel, *blocks1 its grid, *blocks2 = 0) or 2 (the tensor-core pair, their
 * grids), or CF_ERR_INVALID_ARG.  Either pointer may be NULL. */
int cf_ffn_kernels(const cf_ffn_handle* h, int32_t batch, int32_t* blocks1, int32_t* blocks2);

void cf_ffn_destroy(cf_ffn_handle* h); /* NULL-safe */

#ifdef __cplusplus
}
#endif

#endif
