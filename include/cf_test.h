/*
 * cf_test.h -- test and measurement exports of the cluster collectives used
 * inside the fused decode kernel.  Not part of the decode API.
 *
 * ClusterReduce [CF §3.1.1, Alg. 1] and ClusterGather [CF §3.1.2, Alg. 2] of
 * "ClusterFusion框架深度解析：LLM推理优化的集群级通信革命" (devpress.csdn.net):
 * butterfly rounds with partner = rank ^ stride over distributed shared
 * memory.  Every call launches ONE thread-block cluster of `cluster_size`
 * blocks (1, 2, 4, 8 or 16) on `stream` and returns without waiting.
 *
 * All buffers are device float arrays, row r belonging to cluster block r;
 * n is a positive multiple of 4; errflag is a device int that receives bit 2
 * if an in-kernel wait timed out (it is only ever OR-ed).
 * Errors: CF_ERR_INVALID_ARG (sizes, NULLs, shared memory over 200 KB),
 * CF_ERR_CLUSTER, CF_ERR_CUDA.
 */
#ifndef CF_TEST_H
#define CF_TEST_H

#ifdef __cplusplus
extern "C" {
#endif

/* All-reduce: in, out [cluster_size][n]; every out row = op over in rows
 * (op 0 = sum, 1 = max).  All rows of out are bitwise identical. */
int cf_test_cluster_allreduce(int cluster_size, int op, int n, const float* in, float* out,
                              int* errflag, void* stream);

/* Reduce-scatter: in [cluster_size][cluster_size*n] (row r holds block r's N
 * slices of n floats); out [cluster_size][n]: out row r = sum over blocks of
 * slice r. */
int cf_test_cluster_reduce_scatter(int cluster_size, int n, const float* in, float* out,
                                   int* errflag, void* stream);

/* All-gather: in [cluster_size][n] (block r's slice); out
 * [cluster_size][cluster_size*n]: every row = concatenation of all slices. */
int cf_test_cluster_gather(int cluster_size, int n, const float* in, float* out, int* errflag,
                           void* stream);

/* Same collectives (kind 0 sum all-reduce, 1 max all-reduce, 2 reduce-scatter,
 * 3 gather) with the SM cycles each block spent inside the collective written
 * to cycles[cluster_size] (device long long).  Buffer shapes as above. */
int cf_bench_cluster_collective(int kind, int cluster_size, int n, const float* in, float* out,
                                int* errflag, long long* cycles, void* stream);

/* Bare TMA streaming rate of the decode kernel's W_qkv access pattern: one
 * launch of cluster_size * n_kv_heads blocks (no cluster attribute; any
 * cluster_size dividing hidden), each streaming its K band of the three
 * head_dim-wide column slices of head g of the fp16 matrix w [hidden,
 * (nq+2nkv)*head_dim] in tiles of rows_per_tile rows through `stages`
 * shared-memory stages, with shared memory padded so that ctas_per_sm blocks
 * fit per SM.  No compute.  Errors: CF_ERR_INVALID_ARG, CF_ERR_CUDA. */
int cf_bench_tma_stream(int hidden, int n_q_heads, int n_kv_heads, int head_dim,
                        int cluster_size, int rows_per_tile, int stages, int ctas_per_sm,
                        const void* w, int* errflag, void* stream);

/* Bare TMA streaming rate of the batched kernel's K/V access pattern: one
 * launch of n_kv_heads * batch / rows_per_block blocks; block i streams, for
 * KV head i % n_kv_heads and each of its rows_per_block batch rows, positions
 * [0, len) of the fp16 caches k_cache, v_cache [batch, s_max, n_kv_heads,
 * head_dim] in tiles of pos_per_tile positions (one K and one V box per
 * stage) through `stages` stages, shared memory padded so that ctas_per_sm
 * blocks fit per SM.  No compute.  Errors: CF_ERR_INVALID_ARG, CF_ERR_CUDA. */
int cf_bench_kv_stream(int batch, int s_max, int n_kv_heads, int head_dim, int elem_bytes,
                       int len, int rows_per_block, int pos_per_tile, int stages,
                       int ctas_per_sm, const void* k_cache, const void* v_cache, int* errflag,
                       void* stream);

/* Bare TMA streaming rate of weight-band tile shapes: `blocks` blocks, block i
 * streaming band_rows x band_cols of the row-major fp16 [rows, cols] matrix w
 * (band i mod cols/band_cols, row block i / (cols/band_cols) mod
 * rows/band_rows) as tiles of `bps` boxes {box_cols, box_rows} side by side,
 * through `stages` stages.  No compute.  flags: bit 0 the 128-byte swizzle;
 * bits 1-2 the L2 promotion (0: 256 B, 1: 128 B, 2: none, 3: 64 B); bit 3
 * launch with only the shared memory the ring needs (several blocks per SM),
 * else with the full opt-in amount (one block per SM); bit 4 walk the band's
 * tiles down its rows first (column groups outer).  Errors:
 * CF_ERR_INVALID_ARG, CF_ERR_CUDA. */
int cf_bench_box_stream(const void* w, int rows, int cols, int box_cols, int box_rows,
                        int flags, int bps, int band_rows, int band_cols, int stages,
                        int blocks, int* errflag, void* stream);

/* Bare streaming rate of contiguous per-block regions: `blocks` blocks, block
 * i streaming bytes [(i mod n) * region_bytes, +region_bytes) of w (n =
 * min(blocks, total_bytes / region_bytes)) in stages of stage_bytes (a
 * multiple of 1024), each filled by `pieces` equal bulk copies, through
 * `stages` stages; shared_sm != 0 launches with only the shared memory the
 * ring needs.  No compute.  Errors: CF_ERR_INVALID_ARG, CF_ERR_CUDA. */
int cf_bench_contig_stream(const void* w, long long total_bytes, long long region_bytes,
                           int stage_bytes, int pieces, int stages, int blocks, int shared_sm,
                           int* errflag, void* stream);

/* Phase timeline of later cf_decode_attn_block calls of handle h (a tuning
 * aid): when `stamps` is a zeroed device buffer of grid_blocks * 32 unsigned
 * 64-bit values, every block writes %globaltimer (ns) at its phase
 * boundaries into its row of 32 slots (slot meanings: the TimelineSlot enum
 * of the kernel sources, listed in order by the Python binding).  The grid
 * has cluster_size * n_kv_heads * ceil(batch / batch_tile) blocks.  NULL
 * turns it off.  Returns CF_OK or CF_ERR_INVALID_ARG. */
struct cf_handle;
int cf_set_timeline(struct cf_handle* h, unsigned long long* stamps);

/* One fifth-generation tensor-core product by one block:
 * d[128, n] = A . b[n, k]^T with fp32 accumulation, where A = a as a [128, k]
 * row-major array (a_mn = 0, K-major operand) or A = a^T with a a [k, 128]
 * row-major array (a_mn = 1, M-major operand staged as two 64-column boxes).
 * a and b are fp16 (dtype CF_F16) or bf16 (CF_BF16) device arrays (16-byte
 * aligned), d a row-major fp32 device array.  n a multiple of 16 in
 * [16, 256], k a multiple of 64 with the staged operands inside the block's
 * shared memory.  Errors: CF_ERR_INVALID_ARG, CF_ERR_CUDA. */
int cf_test_tc05_gemm(int dtype, int a_mn, int n, int k, const void* a, const void* b, float* d,
                      int* errflag, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CF_TEST_H */
