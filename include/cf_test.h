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

#include <stdint.h>

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

/* Failure detection of the bounded in-kernel waits [CF §4.3 典型性能问题排查]:
 * one exchange of the sum all-reduce between the two blocks of a 2-block
 * cluster in which block drop_rank (0 or 1; -1 = none) does not send, as if
 * its transfer were lost.  The partner's wait gives up after limit_cycles SM
 * cycles (the decode kernels use about one second) and ORs bit 2 (timeout)
 * into *errflag; the launch then finishes normally and the context stays
 * usable.  in, out [2][n] (n a multiple of 4, <= 16384): out row r = in row
 * r + the row block r received (zeros when nothing arrived).
 * Errors: CF_ERR_INVALID_ARG, CF_ERR_CUDA. */
int cf_test_lost_transfer(int n, int drop_rank, long long limit_cycles, const float* in,
                          float* out, int* errflag, void* stream);

/* Same collectives (kind 0 sum all-reduce, 1 max all-reduce, 2 reduce-scatter,
 * 3 gather) with the SM cycles each block spent inside the collective written
 * to cycles[cluster_size] (device long long).  Buffer shapes as above. */
int cf_bench_cluster_collective(int kind, int cluster_size, int n, const float* in, float* out,
                                int* errflag, long long* cycles, void* stream);

/* Phase timeline of later cf_decode_attn_block calls of handle h (a tuning
 * aid): when `stamps` is a zeroed device buffer of grid_blocks * 32 unsigned
 * 64-bit values, every block writes %globaltimer (ns) at its phase
 * boundaries into its row of 32 slots (slot meanings: the TimelineSlot enum
 * of the kernel sources, listed in order by the Python binding).  The grid
 * has cluster_size * n_kv_heads * ceil(batch / batch_tile) blocks.  NULL
 * turns it off.  Returns CF_OK or CF_ERR_INVALID_ARG. */
struct cf_handle;
int cf_set_timeline(struct cf_handle* h, unsigned long long* stamps);

/* Phase timeline of later cf_mla_decode calls of handle h (a tuning aid):
 * when `stamps` is a zeroed device buffer of clusters * 4 * 32 unsigned
 * 64-bit values, every block writes %globaltimer (ns) at its phase boundaries
 * into its row of 32 slots (slot meanings: the MlaTimelineSlot enum of the
 * kernel source, listed in order by the Python binding).  NULL turns it off.
 * Returns CF_OK or CF_ERR_INVALID_ARG. */
struct cf_mla_handle;
int cf_mla_set_timeline(struct cf_mla_handle* h, unsigned long long* stamps);

/* The intermediate activations a = silu(gate) * up of the last
 * cf_ffn_forward call of handle h with `batch` rows on the tensor-core pair
 * (batches of 3 or more rows): the kernel keeps a as 16-bit hi + lo pairs,
 * which this reads back (synchronously) and writes summed into the host
 * array a_out [batch, intermediate].  A test aid.  Errors:
 * CF_ERR_INVALID_ARG, CF_ERR_UNSUPPORTED (a handle without the pair),
 * CF_ERR_CUDA. */
struct cf_ffn_handle;
int cf_ffn_debug_a(const struct cf_ffn_handle* h, int32_t batch, float* a_out);

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
