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


// Generic weight-band streaming skeleton: block i streams rows
// [r_i, r_i + band_rows) x columns [c_i, c_i + band_cols) of a row-major
// 16-bit [rows, cols] matrix as tiles of `bps` boxes {box_cols, box_rows} side
// by side (one stage per tile), no compute.
struct BoxStreamParams {
  CUtensorMap tm;
  int rows, cols, box_cols, box_rows, bps, band_rows, band_cols, stages, stage_bytes;
  int col_major;  // tiles walk the band's rows first (columns outer)
  int* errflag;
};

__global__ void __launch_bounds__(64) box_stream_kernel(const __grid_constant__ BoxStreamParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)p.stages * p.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb_c = p.cols / p.band_cols;
  const int c_i = (blockIdx.x % nb_c) * p.band_cols;
  const int r_i = ((blockIdx.x / nb_c) * p.band_rows) % p.rows;
  const int tc = p.bps * p.box_cols;  // columns per tile
  const int n_r = p.band_rows / p.box_rows, n_c = p.band_cols / tc, total = n_r * n_c;
  const uint32_t box_bytes = (uint32_t)(p.box_cols * p.box_rows * 2);
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
        mbar_arrive_expect_tx(&full[s], p.bps * box_bytes);
        uint8_t* dst = sm + (size_t)s * p.stage_bytes;
        const int ti = p.col_major ? (it % n_r) : (it / n_c);
        const int tj = p.col_major ? (it / n_r) : (it % n_c);
        const int rr = r_i + ti * p.box_rows, cc = c_i + tj * tc;
        for (int j = 0; j < p.bps; ++j)
          tma_load_2d(dst + j * box_bytes, &p.tm, cc + j * p.box_cols, rr, &full[s], pol);
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


// Contiguous streaming skeleton: block i streams bytes [r_i, r_i + region) of
// w, r_i = (i mod nregions) * region, in stages of stage_bytes made of
// `pieces` equal bulk copies.  No compute.
struct ContigStreamParams {
  const uint8_t* w;
  long long region;
  int nregions, stage_bytes, pieces, stages;
  int* errflag;
};

__global__ void __launch_bounds__(64) contig_stream_kernel(const __grid_constant__ ContigStreamParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + (size_t)p.stages * p.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint8_t* src = p.w + (long long)(blockIdx.x % p.nregions) * p.region;
  const int total = (int)(p.region / p.stage_bytes);
  const uint32_t piece = (uint32_t)(p.stage_bytes / p.pieces);
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
        mbar_arrive_expect_tx(&full[s], (uint32_t)p.stage_bytes);
        uint8_t* dst = sm + (size_t)s * p.stage_bytes;
        for (int j = 0; j < p.pieces; ++j)
          bulk_load_1d(dst + j * piece, src + (long long)it * p.stage_bytes + j * piece, piece,
                       &full[s], pol);
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

extern "C" int cf_bench_box_stream(const void* w, int rows, int cols, int box_cols, int box_rows,
                                   int flags, int bps, int band_rows, int band_cols,
                                   int stages, int blocks, int* errflag, void* stream) {
  if (w == nullptr || errflag == nullptr || ((uintptr_t)w & 15u)) return CF_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || box_cols <= 0 || box_cols > 256 || box_rows <= 0 ||
      box_rows > 256 || (box_cols * 2) % 16 != 0 || bps <= 0 || blocks <= 0)
    return CF_ERR_INVALID_ARG;
  const bool swizzle128 = flags & 1;
  const int promo = (flags >> 1) & 3;  // 0: 256 B, 1: 128 B, 2: none, 3: 64 B
  const bool shared_sm = (flags >> 3) & 1;
  if (swizzle128 && box_cols * 2 > 128) return CF_ERR_INVALID_ARG;
  if (band_rows % box_rows || band_cols % (bps * box_cols) || cols % band_cols ||
      rows % band_rows || stages < 1 || stages > kMaxStages)
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
  BoxStreamParams p;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t str[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  if (enc(&p.tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(w), dims, str, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE,
          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
          promo == 0   ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
          : promo == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
          : promo == 2 ? CU_TENSOR_MAP_L2_PROMOTION_NONE
                       : CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CF_ERR_CUDA;
  p.rows = rows;
  p.cols = cols;
  p.box_cols = box_cols;
  p.box_rows = box_rows;
  p.bps = bps;
  p.band_rows = band_rows;
  p.band_cols = band_cols;
  p.stages = stages;
  p.col_major = (flags >> 4) & 1;
  p.stage_bytes = (bps * box_cols * box_rows * 2 + 1023) / 1024 * 1024;
  p.errflag = errflag;
  cudaDeviceProp prop;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
    return CF_ERR_CUDA;
  const int need = stages * p.stage_bytes + 2 * kMaxStages * 8 + 1024;
  const int per_block = (int)prop.sharedMemPerBlockOptin;
  if (need > per_block) return CF_ERR_INVALID_ARG;
  const int smem = shared_sm ? need : per_block;
  if (cudaFuncSetAttribute(box_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           per_block) != cudaSuccess)
    return CF_ERR_CUDA;
  box_stream_kernel<<<blocks, 64, smem, static_cast<cudaStream_t>(stream)>>>(p);
  if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
  return CF_OK;
}

extern "C" int cf_bench_contig_stream(const void* w, long long total_bytes, long long region_bytes,
                                      int stage_bytes, int pieces, int stages, int blocks,
                                      int shared_sm, int* errflag, void* stream) {
  if (w == nullptr || errflag == nullptr || ((uintptr_t)w & 15u)) return CF_ERR_INVALID_ARG;
  if (blocks <= 0 || stages < 1 || stages > kMaxStages || pieces < 1 || stage_bytes <= 0 ||
      stage_bytes % (16 * pieces) != 0 || region_bytes <= 0 || region_bytes % stage_bytes != 0 ||
      region_bytes > total_bytes)
    return CF_ERR_INVALID_ARG;
  ContigStreamParams p;
  p.w = static_cast<const uint8_t*>(w);
  p.region = region_bytes;
  const long long nr = total_bytes / region_bytes;
  p.nregions = (int)(nr < blocks ? nr : blocks);
  p.stage_bytes = stage_bytes;
  p.pieces = pieces;
  p.stages = stages;
  p.errflag = errflag;
  cudaDeviceProp prop;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
    return CF_ERR_CUDA;
  const int need = stages * ((stage_bytes + 1023) / 1024 * 1024) + 2 * kMaxStages * 8 + 1024;
  const int per_block = (int)prop.sharedMemPerBlockOptin;
  if (need > per_block || stage_bytes % 1024 != 0) return CF_ERR_INVALID_ARG;
  if (cudaFuncSetAttribute(contig_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           per_block) != cudaSuccess)
    return CF_ERR_CUDA;
  contig_stream_kernel<<<blocks, 64, shared_sm ? need : per_block,
                         static_cast<cudaStream_t>(stream)>>>(p);
  if (cudaGetLastError() != cudaSuccess) return CF_ERR_CUDA;
  return CF_OK;
}
