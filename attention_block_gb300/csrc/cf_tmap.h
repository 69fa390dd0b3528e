// cf_tmap.h -- internal: 2D TMA tensor-map encoding for the FFN's host code
// (implemented in cf_tmap.cu).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace cf {

// Encode a 2D tiled tensor map over a row-major [outer, inner] array of
// 16-bit (dtype CF_F16 / CF_BF16) or fp32 elements with rows `row_bytes`
// apart, boxes of box_inner x box_outer elements, optionally with the
// 128-byte swizzle; out-of-range elements read as zero.  False on failure.
bool encode_tmap_2d(CUtensorMap* m, int dtype, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128);

}  // namespace cf
