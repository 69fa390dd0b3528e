/*
 * cf_mla.h -- C ABI of the DeepSeek multi-head latent attention (MLA) variant
 * of the fused decode attention block.
 *
 * Page cited by title and section:
 *   [CF] "ClusterFusion框架深度解析：LLM推理优化的集群级通信革命"
 *        (devpress.csdn.net), §5.2 DeepSeek-MLA特殊处理: the latent key/value
 *        cache is partitioned across clusters and ClusterReduce gets a sparse
 *        form.
 *
 * The page gives only that adaptation; the projections are read as
 * DeepSeek's published MLA with an uncompressed query.  For every batch row b
 * with position p = positions[b]:
 *   n    = RMSNorm(x_b; ln_weight)                    (eps inside the root)
 *   q    = n . w_q           w_q  [H, nh*(dn+dr)]; head h = [nope (dn) | rope (dr)]
 *   a    = n . w_dkv         w_dkv [H, dc+dr];     a = [c (dc) | kr (dr)]
 *   c'   = RMSNorm(c; kv_norm_weight)
 *   RoPE (rotate-half, theta^(-2i/dr)) on every q rope part and on kr
 *   latent_cache[b, p, :] = [c' | kr]                 (rounded to the storage type)
 *   head h, positions t in 0..p, w_ukv [dc, nh*(dn+dv)] (head h's columns
 *   [k part (dn) | v part (dv)]):
 *     k_{t,h} = [L[t,:dc] . w_ukv[:, k part of h] | L[t, dc:]],
 *     v_{t,h} =  L[t,:dc] . w_ukv[:, v part of h],
 *     o_h = softmax_t(q_h . k_{t,h} / sqrt(dn+dr)) . v_{t,h}
 *   out_b = x_b + concat_h(o_h) . w_o                 w_o [nh*dv, H]
 * Built head dimensions: dn = 128, dr = 64, dv = 128, dc = 512 (DeepSeek's).
 *
 * The kernel computes the same result in the weight-absorbed order (the
 * query's no-position part is taken into the latent space once, q_lat_h =
 * w_uk_h q_nope_h, and the attention output stays latent until one w_uv_h
 * product per head), which reads the latent cache once instead of forming
 * per-head keys and values.  One launch per call: a persistent grid of
 * 8-block clusters, one block per SM, in four phases separated by grid-wide
 * barriers (bounded waits):
 *   1. the merged projection n . [w_q | w_dkv] in 192-column x 64-row tiles
 *      spread over all blocks (fp32 atomics into a workspace);
 *   2. the absorption q_lat_h and the latent row (its norm, RoPE, the cache
 *      append);
 *   3. attention over the latent cache, whose positions are partitioned
 *      across the clusters (and inside a cluster across its blocks); each
 *      block keeps online-softmax states for every head and a sparse
 *      ClusterReduce sends each head's state only to the block that owns it
 *      (one DSMEM push per head, no all-reduce), which merges the cluster's
 *      states and writes one partial per (cluster, head);
 *   4. per head (one cluster each): the merge of the clusters' partials, the
 *      w_uv product (reduced over the cluster by DSMEM all-reduce), the w_o
 *      product of the cluster's column bands, fp32 atomics, and the residual
 *      by the last head to finish a band.
 * A producer warp per block streams, by TMA, every byte the block reads in
 * the four phases, ahead of the consumers and across the barriers.
 *
 * Conventions: every function returns CF_OK (0) or a negative CF_ERR_* code
 * of cf.h; "device" pointers are on the device current at cf_mla_create; the
 * caller owns every tensor; tensors are dense, row-major, in the handle's
 * storage type, 16-byte aligned.
 */
#ifndef CF_MLA_H
#define CF_MLA_H

#include <stdint.h>

#include "cf.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cf_mla_config {
  int32_t hidden;     /* H: a multiple of 512                                 */
  int32_t n_heads;    /* nh: 8 or 16 (and at most the resident clusters)     */
  int32_t d_nope;     /* dn: 128                                              */
  int32_t d_rope;     /* dr: 64                                               */
  int32_t d_v;        /* dv: 128                                              */
  int32_t d_latent;   /* dc: 512                                              */
  int32_t max_batch;  /* 1..4, and at most the number of resident clusters    */
  int32_t s_max;      /* S: latent cache capacity per row                     */
  float rope_theta;
  float rms_eps;      /* both RMSNorms                                        */
  int32_t dtype;      /* CF_F16 or CF_BF16 (storage); arithmetic is fp32      */
} cf_mla_config;

typedef struct cf_mla_handle cf_mla_handle; /* opaque */

/* Validate cfg, plan the launch (one 8-block cluster per group of SMs, as
 * many clusters as can be resident at once with one block per SM) and
 * allocate the handle's device workspace on the current device.  On failure
 * nothing stays allocated and *out is NULL.  Errors: INVALID_ARG (NULL,
 * sizes), UNSUPPORTED (head dimensions, dtype, n_heads or hidden outside the
 * built set), CLUSTER (too few clusters resident), CUDA. */
int cf_mla_create(const cf_mla_config* cfg, cf_mla_handle** out);

/* Enqueue one MLA decode step for `batch` rows on `stream` (a cudaStream_t,
 * NULL = the legacy default stream).  Asynchronous: no allocation, host
 * synchronization or host copy, so it can be captured in a CUDA graph.
 *   hidden_states  [batch, H]                 read
 *   ln_weight      [H]                        read
 *   w_q            [H, nh*(dn+dr)]            read
 *   w_dkv          [H, dc+dr]                 read
 *   kv_norm_weight [dc]                       read
 *   w_ukv          [dc, nh*(dn+dv)]           read
 *   w_o            [nh*dv, H]                 read
 *   latent_cache   [batch, S, dc+dr]          slot [b, positions[b]] written with
 *                                             the new latent row, nothing else
 *   positions      [batch] int32              the new token's slot and RoPE
 *                                             position; attention covers 0..p
 *   out            [batch, H]                 written; must not overlap an input
 * A positions[b] outside [0, S) is reported by cf_mla_get_status as
 * CF_ERR_DEVICE_POS_RANGE; that row's cache is untouched and its out row
 * equals its hidden row.  batch == 0 is a no-op.  Errors: INVALID_ARG,
 * ALIAS, CUDA.  Not thread-safe per handle: one handle per stream. */
int cf_mla_decode(cf_mla_handle* h, int32_t batch, const void* hidden_states,
                  const void* ln_weight, const void* w_q, const void* w_dkv,
                  const void* kv_norm_weight, const void* w_ukv, const void* w_o,
                  void* latent_cache, const int32_t* positions, void* out, void* stream);

/* Read and clear the handle's device error flag (synchronize first):
 * CF_OK, CF_ERR_DEVICE_POS_RANGE, CF_ERR_DEVICE_TIMEOUT or CF_ERR_CUDA. */
int cf_mla_get_status(cf_mla_handle* h);

/* The launch shape: clusters, blocks per cluster, ring stages, bytes per
 * stage and shared memory per block. */
int cf_mla_launch_info(const cf_mla_handle* h, int32_t* clusters, int32_t* cluster_size,
                       int32_t* stages, int32_t* stage_bytes, int32_t* smem_bytes);

/* Free the handle and its workspace.  NULL is a no-op. */
void cf_mla_destroy(cf_mla_handle* h);

#ifdef __cplusplus
}
#endif

#endif /* CF_MLA_H */
