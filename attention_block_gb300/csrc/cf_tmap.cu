// cf_tmap.cu -- 2D TMA tensor-map encoding for the FFN's host code (the
// declaration and its contract are in cf_tmap.h).  The driver's encoder is
// looked up once through the runtime's entry-point query.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "cf.h"
#include "cf_tmap.h"

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode2d = nullptr;
std::once_flag g_encode2d_once;

bool have_encoder() {
  std::call_once(g_encode2d_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode2d = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode2d != nullptr;
}

}  // namespace

bool cf::encode_tmap_2d(CUtensorMap* m, int dtype, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                        uint32_t box_outer, bool swizzle128) {
  if (!have_encoder()) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t str[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType t = dtype == CF_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                : dtype == CF_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return g_encode2d(m, t, 2, const_cast<void*>(base), dims, str, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
