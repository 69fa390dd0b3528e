// cf_testtc05.cu -- test-only export of one tcgen05 product (declared in
// include/cf_test.h): D[128, N] = A[128, K] . B[N, K]^T in fp32 from fp16 or
// bf16 operands, by one CTA, through the helpers of cf_tc05.cuh.  A is either
// K-major (given as [128, K]) or M-major (given as [K, 128], staged as two
// 64-column boxes of K rows, the layout of a weight tile read by TMA); B is
// K-major.  It checks the descriptor encodings and the TMEM data path
// against a host matmul.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "cf.h"
#include "cf_ptx.cuh"
#include "cf_tc05.cuh"
#include "cf_test.h"

using namespace cf;

namespace {

constexpr int kM = 128;

// Bytes between the two 64-column boxes of an M-major A: the box plus a gap,
// so that the descriptor's leading byte offset is exercised.
__host__ __device__ constexpr int mn_box_stride(int K) { return K * 128 + 1024; }

// Shared memory: A (K-major slabs [K/64][128 rows][128 B], or M-major boxes
// [2][K rows][128 B] at mn_box_stride), B slabs [K/64][N rows][128 B], the
// mbarrier and the TMEM address word.
template <typename T, bool kBf16>
__global__ void __launch_bounds__(128, 1) tc05_test_kernel(const T* __restrict__ A,
                                                           const T* __restrict__ B,
                                                           float* __restrict__ D, int a_mn, int N,
                                                           int K, int* errflag) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int nslab = K / 64;
  uint8_t* sa = sm;
  uint8_t* sb = sa + (a_mn ? 2 * (size_t)mn_box_stride(K) : (size_t)nslab * kM * 128);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sb + (size_t)nslab * N * 128);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // stage A and B with the 128-byte swizzle, 8 elements (16 bytes) at a time
  auto stage = [&](const T* src, uint8_t* dst, int rows) {
    for (int c = tid; c < rows * (K / 8); c += blockDim.x) {
      const int r = c / (K / 8), k8 = c % (K / 8);  // 16-byte chunk k8 of row r
      const int slab = k8 / 8, j = k8 % 8;
      const uint4 v = *reinterpret_cast<const uint4*>(src + (size_t)r * K + k8 * 8);
      *reinterpret_cast<uint4*>(dst + (size_t)slab * rows * 128 + r * 128 + ((j ^ (r & 7)) << 4)) =
          v;
    }
  };
  if (a_mn) {
    // A given as [K][128]: box bx holds columns 64bx..64bx+63 of every k row,
    // row k at k*128, 16-byte chunk j at j ^ (k & 7)
    for (int c = tid; c < K * 16; c += blockDim.x) {
      const int k = c / 16, m8 = c % 16, bx = m8 / 8, j = m8 % 8;
      const uint4 v = *reinterpret_cast<const uint4*>(A + (size_t)k * kM + m8 * 8);
      *reinterpret_cast<uint4*>(sa + (size_t)bx * mn_box_stride(K) + k * 128 +
                                ((j ^ (k & 7)) << 4)) = v;
    }
  } else {
    stage(A, sa, kM);
  }
  stage(B, sb, N);
  fence_proxy_async_smem();  // generic-proxy stores before the tensor core reads
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init_cluster();
  }
  const uint32_t ncols = N <= 32 ? 32u : (N <= 64 ? 64u : (N <= 128 ? 128u : 256u));
  if (warp == 0) {
    tmem_alloc(tslot, ncols);
    tmem_relinquish();
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  const uint32_t taddr = *tslot;

  if (tid == 0) {
    const uint32_t idesc = idesc_kind_f16(kBf16, kM, N, a_mn != 0);
    for (int ks = 0; ks < K / 16; ++ks) {
      const int slab = ks / 4;
      const uint32_t koff = (uint32_t)(ks % 4) * 32u;
      const uint64_t ad =
          a_mn ? smem_desc_mn_sw128(smem_u32(sa) + (uint32_t)ks * 2048u,
                                    (uint32_t)mn_box_stride(K), 1024)
               : smem_desc_k_sw128(smem_u32(sa + (size_t)slab * kM * 128) + koff, 1024);
      const uint64_t bd = smem_desc_k_sw128(smem_u32(sb + (size_t)slab * N * 128) + koff, 1024);
      tc05_mma_f16(taddr, ad, bd, idesc, ks > 0);
    }
    tc05_commit(bar);
  }
  mbar_wait(bar, 0, errflag);
  tc05_fence_after();
  for (int c0 = 0; c0 < N; c0 += 8) {
    float v[8];
    tmem_ld_32x32b_x8(taddr + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
    float* row = D + (size_t)(32 * warp + lane) * N + c0;
#pragma unroll
    for (int i = 0; i < 8; ++i) row[i] = v[i];
  }
  tc05_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, ncols);
}

}  // namespace

extern "C" int cf_test_tc05_gemm(int dtype, int a_mn, int n, int k, const void* a, const void* b,
                                 float* d, int* errflag, void* stream) {
  if ((dtype != CF_F16 && dtype != CF_BF16) || (a_mn != 0 && a_mn != 1) || n < 16 || n > 256 ||
      n % 16 != 0 || k < 64 || k % 64 != 0 || a == nullptr || b == nullptr || d == nullptr || errflag == nullptr ||
      ((uintptr_t)a & 15u) || ((uintptr_t)b & 15u))
    return CF_ERR_INVALID_ARG;
  const size_t need = (a_mn ? 2 * (size_t)mn_box_stride(k) : (size_t)(k / 64) * kM * 128) +
                      (size_t)(k / 64) * n * 128 + 64 + 1024;
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
    return CF_ERR_CUDA;
  const int smem = (int)prop.sharedMemPerBlockOptin;  // the whole window: every address is valid
  if (need > (size_t)smem) return CF_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == CF_F16) {
    if (cudaFuncSetAttribute(tc05_test_kernel<__half, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return CF_ERR_CUDA;
    tc05_test_kernel<__half, false><<<1, 128, smem, st>>>(static_cast<const __half*>(a),
                                                   static_cast<const __half*>(b), d, a_mn, n,
                                                   k, errflag);
  } else {
    if (cudaFuncSetAttribute(tc05_test_kernel<__nv_bfloat16, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return CF_ERR_CUDA;
    tc05_test_kernel<__nv_bfloat16, true><<<1, 128, smem, st>>>(
        static_cast<const __nv_bfloat16*>(a), static_cast<const __nv_bfloat16*>(b), d, a_mn, n, k,
        errflag);
  }
  return cudaGetLastError() == cudaSuccess ? CF_OK : CF_ERR_CUDA;
}
