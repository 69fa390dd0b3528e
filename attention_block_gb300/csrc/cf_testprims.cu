// cf_testprims.cu -- test-only exports that run the cluster collectives of
// cf_cluster.cuh on caller data (declared in include/cf_test.h).
//
// Each launch is one cluster of N blocks; block r copies its row in[r] into
// shared memory, runs one collective with the 256 threads that the fused
// kernel also uses for them, and writes the result row to out[r].  A second
// entry point times one collective in SM cycles (the GB300 counterpart of the
// primitive latencies in [CF §3.1.2, Table 1], page "ClusterFusion框架深度解析"
// (devpress.csdn.net)).
#include <cuda_runtime.h>

#include "cf.h"
#include "cf_cluster.cuh"
#include "cf_test.h"

using namespace cf;

namespace {

constexpr int kNT = kConsumers;
constexpr int kBar = 1;

enum { kAllSum = 0, kAllMax = 1, kReduceScatter = 2, kGather = 3 };

// Floats of receive area a collective needs (see cf_cluster.cuh).
__host__ __device__ int recv_floats(int kind, int N, int n) {
  int nr = 0;
  while ((1 << nr) < N) ++nr;
  return kind == kReduceScatter ? (N - 1) * n : (kind == kGather ? 0 : nr * n);
}

// Shared-memory layout: data [len] | receive area | kMaxRounds barriers.
__global__ void __launch_bounds__(kNT) prim_kernel(int kind, int n, const float* __restrict__ in,
                                                   float* __restrict__ out, int* errflag,
                                                   long long* cycles) {
  extern __shared__ __align__(16) float smem[];
  const int N = (int)gridDim.x;  // one cluster spans the grid
  const int rank = (int)cluster_ctarank();
  const int tid = threadIdx.x;
  // data length per block: all-reduce n; reduce-scatter and gather N*n
  const int len = (kind == kReduceScatter || kind == kGather) ? N * n : n;
  float* data = smem;
  float* rbuf = smem + len;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + len + recv_floats(kind, N, n));
  const int nrounds = __ffs(N) - 1;
  if (tid == 0) {
    for (int r = 0; r < nrounds; ++r) mbar_init(&bars[r], 1);
    fence_mbar_init_cluster();
    for (int r = 0; r < nrounds; ++r) {
      int bytes = kind == kReduceScatter ? reduce_scatter_round_bytes(N, r, n)
                  : kind == kGather      ? gather_round_bytes(r, n)
                                         : allreduce_round_bytes(n);
      mbar_arrive_expect_tx(&bars[r], bytes);
    }
  }
  for (int i = tid; i < len; i += kNT) {
    if (kind == kGather)
      data[i] = (i >= rank * n && i < (rank + 1) * n) ? in[(size_t)rank * n + (i - rank * n)] : 0.f;
    else
      data[i] = in[(size_t)rank * len + i];
  }
  __syncthreads();
  cluster_sync_all();
  const long long t0 = clock64();
  switch (kind) {
    case kAllSum:
      cluster_allreduce<OpSum, kNT, kBar>(data, n, rbuf, bars, rank, N, tid, errflag);
      break;
    case kAllMax:
      cluster_allreduce<OpMax, kNT, kBar>(data, n, rbuf, bars, rank, N, tid, errflag);
      break;
    case kReduceScatter:
      cluster_reduce_scatter<kNT, kBar>(data, n, rbuf, bars, rank, N, tid, errflag);
      break;
    default:
      cluster_gather<kNT, kBar>(data, n, bars, rank, N, tid, errflag);
      break;
  }
  const long long t1 = clock64();
  if (tid == 0 && cycles != nullptr) cycles[rank] = t1 - t0;
  if (kind == kReduceScatter) {
    for (int i = tid; i < n; i += kNT) out[(size_t)rank * n + i] = data[rank * n + i];
  } else {
    for (int i = tid; i < len; i += kNT) out[(size_t)rank * len + i] = data[i];
  }
  cluster_sync_all();
}

// A lost transfer and the bounded wait that catches it: one exchange of the
// all-reduce between the two blocks of a 2-block cluster in which block
// `drop_rank` (0 or 1; -1 for none) does not send.  Its partner's wait gives
// up after `limit` SM cycles and records kDevErrTimeout; the dropping block
// still receives, so no remote write is in flight when the blocks leave.
// out[r] = in[r] + whatever block r received (nothing: zeros).
__global__ void __launch_bounds__(kNT) lost_send_kernel(int n, int drop_rank, long long limit,
                                                        const float* __restrict__ in,
                                                        float* __restrict__ out, int* errflag) {
  extern __shared__ __align__(16) float smem[];
  const int rank = (int)cluster_ctarank();
  const int tid = threadIdx.x;
  float* data = smem;
  float* rb = smem + n;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 2 * n);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init_cluster();
    mbar_arrive_expect_tx(bar, allreduce_round_bytes(n));
  }
  for (int i = tid; i < n; i += kNT) {
    data[i] = in[(size_t)rank * n + i];
    rb[i] = 0.f;
  }
  __syncthreads();
  cluster_sync_all();
  if (rank != drop_rank) push_to_peer<kNT>(data, rb, n, bar, (uint32_t)(rank ^ 1), tid);
  mbar_wait_cluster(bar, 0, errflag, limit);
  for (int i = tid; i < n; i += kNT) out[(size_t)rank * n + i] = data[i] + rb[i];
  cluster_sync_all();
}

int run(int kind, int N, int n, const float* in, float* out, int* errflag, long long* cycles,
        void* stream) {
  if (!(N == 1 || N == 2 || N == 4 || N == 8 || N == 16)) return CF_ERR_INVALID_ARG;
  if (n <= 0 || n % 4 != 0 || in == nullptr || out == nullptr || errflag == nullptr)
    return CF_ERR_INVALID_ARG;
  const int len = (kind == kReduceScatter || kind == kGather) ? N * n : n;
  const size_t smem = (size_t)(len + recv_floats(kind, N, n)) * 4 + kMaxRounds * 8;
  if (smem > 200 * 1024) return CF_ERR_INVALID_ARG;
  if (cudaFuncSetAttribute(prim_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return CF_ERR_CUDA;
  if (N > 8 &&
      cudaFuncSetAttribute(prim_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
          cudaSuccess)
    return CF_ERR_CLUSTER;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = N;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(N, 1, 1);
  lc.blockDim = dim3(kNT, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = static_cast<cudaStream_t>(stream);
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, prim_kernel, kind, n, in, out, errflag, cycles) != cudaSuccess) {
    cudaGetLastError();
    return CF_ERR_CUDA;
  }
  return CF_OK;
}

}  // namespace

extern "C" {

int cf_test_cluster_allreduce(int cluster_size, int op, int n, const float* in, float* out,
                              int* errflag, void* stream) {
  if (op != 0 && op != 1) return CF_ERR_INVALID_ARG;
  return run(op == 0 ? kAllSum : kAllMax, cluster_size, n, in, out, errflag, nullptr, stream);
}

int cf_test_cluster_reduce_scatter(int cluster_size, int n, const float* in, float* out,
                                   int* errflag, void* stream) {
  return run(kReduceScatter, cluster_size, n, in, out, errflag, nullptr, stream);
}

int cf_test_cluster_gather(int cluster_size, int n, const float* in, float* out, int* errflag,
                           void* stream) {
  return run(kGather, cluster_size, n, in, out, errflag, nullptr, stream);
}

int cf_test_lost_transfer(int n, int drop_rank, long long limit_cycles, const float* in,
                          float* out, int* errflag, void* stream) {
  if (n <= 0 || n % 4 != 0 || n > 16384 || drop_rank < -1 || drop_rank > 1 ||
      limit_cycles <= 0 || in == nullptr || out == nullptr || errflag == nullptr)
    return CF_ERR_INVALID_ARG;
  const size_t smem = (size_t)2 * n * 4 + 16;
  if (cudaFuncSetAttribute(lost_send_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return CF_ERR_CUDA;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(2, 1, 1);
  lc.blockDim = dim3(kNT, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = static_cast<cudaStream_t>(stream);
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, lost_send_kernel, n, drop_rank, limit_cycles, in, out, errflag) !=
      cudaSuccess) {
    cudaGetLastError();
    return CF_ERR_CUDA;
  }
  return CF_OK;
}

int cf_bench_cluster_collective(int kind, int cluster_size, int n, const float* in, float* out,
                                int* errflag, long long* cycles, void* stream) {
  if (kind < 0 || kind > 3 || cycles == nullptr) return CF_ERR_INVALID_ARG;
  return run(kind, cluster_size, n, in, out, errflag, cycles, stream);
}

}  // extern "C"
