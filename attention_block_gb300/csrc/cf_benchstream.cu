// cf_benchstream.cu -- test/measurement export: the bare TMA streaming rate of
// the fused kernel's W_qkv access pattern, without any compute.
//
// Every block plays the role of one block of the decode kernel at B = 1: it
// streams rows [rank*H/N, (rank+1)*H/N) of the three d-column slices (q, k, v
// of one head) of a row-major [H, C] matrix through a ring of shared-memory
// stages with the same TMA boxes, one producer lane and one consumer warp
// that only waits on each stage and releases it.  The achieved bandwidth of
// this skeleton bounds what the projection phase can reach for a given
// launch shape (blocks per SM, stages, stage size).
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "cf.h"
#include "cf_ptx.cuh"
#include "cf_test.h"

using namespace cf;

namespace {

struct StreamParams {
  CUtensorMap tm;  // 2D {C, H}, box {d, rw}
  int H, nq, nkv, d, N, rw, stages, stage_bytes;
  int* errflag;
};

__global__ void __launch_bounds__(64) stream_kernel(const __grid_constant__ StreamParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)p.stages * p.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = blockIdx.x % p.N;
  const int g = (blockIdx.x / p.N) % p.nkv;
  const int Hc = p.H / p.N, nkt = Hc / p.rw, k0 = rank * Hc;
  const uint32_t seg = (uint32_t)(p.rw * p.d * 2);
  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int kt = 0; kt < nkt; ++kt) {
        const int s = kt % p.stages;
        if (kt >= p.stages) mbar_wait(&empty[s], ((kt / p.stages) + 1) & 1, p.errflag);
        mbar_arrive_expect_tx(&full[s], 3 * seg);
        uint8_t* dst = sm + (size_t)s * p.stage_bytes;
        const int y = k0 + kt * p.rw;
        tma_load_2d(dst, &p.tm, g * p.d, y, &full[s], pol);
        tma_load_2d(dst + seg, &p.tm, (p.nq + g) * p.d, y, &full[s], pol);
        tma_load_2d(dst + 2 * seg, &p.tm, (p.nq + p.nkv + g) * p.d, y, &full[s], pol);
      }
    }
    __syncwarp();
  } else {
    for (int kt = 0; kt < nkt; ++kt) {
      const int s = kt % p.stages;
      mbar_wait(&full[s], (kt / p.stages) & 1, p.errflag);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}


// K/V cache streaming skeleton of the batched kernel's attention phase: block
// i serves KV head i % nkv and batch rows [(i / nkv) * rpb, +rpb), streaming
// positions [0, len) of each row's K and V in tiles of rt positions (one
// {d, 1, rt, 1} box of each per stage).
struct KvStreamParams {
  CUtensorMap tk, tv;  // 4D {d, nkv, S, B}, box {d, 1, rt, 1}
  int nkv, d, len, rpb, rt, stages, stage_bytes, esz;
  int* errflag;
};

__global__ void __launch_bounds__(64) kv_stream_kernel(const __grid_constant__ KvStreamParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)p.stages * p.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x % p.nkv;
  const int b0 = (blockIdx.x / p.nkv) * p.rpb;
  const int ntile = (p.len + p.rt - 1) / p.rt;
  const int total = ntile * p.rpb;
  const uint32_t half = (uint32_t)(p.rt * p.d * p.esz);
  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int it = 0; it < total; ++it) {
        const int s = it % p.stages;
        if (it >= p.stages) mbar_wait(&empty[s], ((it / p.stages) + 1) & 1, p.errflag);
        mbar_arrive_expect_tx(&full[s], 2 * half);
        uint8_t* dst = sm + (size_t)s * p.stage_bytes;
        const int r = it / ntile, t = it % ntile;
        tma_load_4d(dst, &p.tk, 0, g, t * p.rt, b0 + r, &full[s], pol);
        tma_load_4d(dst + half, &p.tv, 0, g, t * p.rt, b0 + r, &full[s], pol);
      }
    }
    __syncwarp();
  } else {
    for (int it = 0; it < total; ++it) {
      const int s = it % p.stages;
      mbar_wait(&full[s], (it / p.stages) & 1, p.errflag);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
}

}  // namespace

extern "C" int cf_bench_tma_stream(int hidden, int n_q_heads, int n_kv_heads, int head_dim,
                                   int cluster_size, int rows_per_tile, int stages,
                                   int ctas_per_sm, const void* w, int* errflag, void* stream) {
  if (w == nullptr || errflag == nullptr || ((uintptr_t)w & 15u)) return CF_ERR_INVALID_ARG;
  if (hidden <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads) return CF_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return CF_ERR_INVALID_ARG;
  if (cluster_size <= 0 || hidden % cluster_size) return CF_ERR_INVALID_ARG;
  if (rows_per_tile <= 0 || rows_per_tile > 256 || (hidden / cluster_size) % rows_per_tile)
    return CF_ERR_INVALID_ARG;
  if (stages < 1 || stages > kMaxStages || ctas_per_sm < 1 || ctas_per_sm > 8)
    return CF_ERR_INVALID_ARG;
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (enc == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return CF_ERR_CUDA;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  StreamParams p;
  const int C = (n_q_heads + 2 * n_kv_heads) * head_dim;
  const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)hidden};
  const cuuint64_t str[1] = {(cuuint64_t)C * 2};
  const cuuint32_t box[2] = {(cuuint32_t)head_dim, (cuuint32_t)rows_per_tile};
  const cuuint32_t es[2] = {1, 1};
  if (enc(&p.tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(w), dims, str, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CF_ERR_CUDA;
  p.H = hidden;
  p.nq = n_q_heads;
  p.nkv = n_kv_heads;
  p.d = head_dim;
  p.N = cluster_size;
  p.rw = rows_per_tile;
  p.stages = stages;
  p.stage_bytes = (3 * rows_per_tile * head_dim * 2 + 1023) / 1024 * 1024;
  p.errflag = errflag;
  cudaDeviceProp prop;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
    return CF_ERR_CUDA;
  // Pad the dynamic shared memory so exactly ctas_per_sm blocks fit per SM.
  const int ring = stages * p.stage_bytes + 2 * kMaxStages * 8 + 1024;
  const int per_block = (int)prop.sharedMemPerMultiprocessor / ctas_per_sm -
                        (int)prop.reservedSharedMemPerBlock - 64;
  if (ring > per_block || ring > (int)prop.sharedMemPerBlockOptin) return CF_ERR_INVALID_ARG;
  if (cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, per_block) !=
      cudaSuccess)
    return CF_ERR_CUDA;
  const int grid = cluster_size * n_kv_heads;
  stream_kernel<<<grid, 64, per_block, static_cast<cudaStream_t>(stream)>>>(p);
  if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
  return CF_OK;
}

extern "C" int cf_bench_kv_stream(int batch, int s_max, int n_kv_heads, int head_dim, int elem_bytes,
                                  int len, int rows_per_block, int pos_per_tile, int stages,
                                  int ctas_per_sm, const void* k_cache, const void* v_cache,
                                  int* errflag, void* stream) {
  if (k_cache == nullptr || v_cache == nullptr || errflag == nullptr ||
      ((uintptr_t)k_cache & 15u) || ((uintptr_t)v_cache & 15u))
    return CF_ERR_INVALID_ARG;
  if (batch <= 0 || s_max <= 0 || n_kv_heads <= 0 || (head_dim != 64 && head_dim != 128))
    return CF_ERR_INVALID_ARG;
  if (elem_bytes != 2 || len <= 0 || len > s_max || rows_per_block <= 0 ||
      batch % rows_per_block != 0)
    return CF_ERR_INVALID_ARG;
  if (pos_per_tile <= 0 || pos_per_tile > 256 || stages < 1 || stages > kMaxStages ||
      ctas_per_sm < 1 || ctas_per_sm > 8)
    return CF_ERR_INVALID_ARG;
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (enc == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return CF_ERR_CUDA;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  KvStreamParams p;
  const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)n_kv_heads, (cuuint64_t)s_max,
                              (cuuint64_t)batch};
  const cuuint64_t str[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_kv_heads * head_dim * 2,
                             (cuuint64_t)s_max * n_kv_heads * head_dim * 2};
  const cuuint32_t box[4] = {(cuuint32_t)head_dim, 1u, (cuuint32_t)pos_per_tile, 1u};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  for (int which = 0; which < 2; ++which)
    if (enc(which == 0 ? &p.tk : &p.tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
            const_cast<void*>(which == 0 ? k_cache : v_cache), dims, str, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return CF_ERR_CUDA;
  p.nkv = n_kv_heads;
  p.d = head_dim;
  p.len = len;
  p.rpb = rows_per_block;
  p.rt = pos_per_tile;
  p.stages = stages;
  p.esz = elem_bytes;
  p.stage_bytes = (2 * pos_per_tile * head_dim * elem_bytes + 1023) / 1024 * 1024;
  p.errflag = errflag;
  cudaDeviceProp prop;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
    return CF_ERR_CUDA;
  const int ring = stages * p.stage_bytes + 2 * kMaxStages * 8 + 1024;
  const int per_block = (int)prop.sharedMemPerMultiprocessor / ctas_per_sm -
                        (int)prop.reservedSharedMemPerBlock - 64;
  if (ring > per_block || ring > (int)prop.sharedMemPerBlockOptin) return CF_ERR_INVALID_ARG;
  if (cudaFuncSetAttribute(kv_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           per_block) != cudaSuccess)
    return CF_ERR_CUDA;
  const int grid = n_kv_heads * (batch / rows_per_block);
  kv_stream_kernel<<<grid, 64, per_block, static_cast<cudaStream_t>(stream)>>>(p);
  if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
  return CF_OK;
}
