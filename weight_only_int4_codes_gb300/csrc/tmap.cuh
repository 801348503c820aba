// tmap.cuh -- host helpers: TMA tensor maps (see tmap.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

// A row-major 2-D tensor of `outer` rows x `inner` elements (row pitch
// `row_stride_bytes`, a multiple of 16), loaded in boxes of
// box_outer x box_inner elements.  Out-of-bounds box elements read as zero.
// Returns false if the driver rejects the description.
bool make_tmap_2d(CUtensorMap *out, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                  uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swizzle);

// General form, rank 1..3: dims[0] is the contiguous dimension, strides_bytes[i]
// the byte stride of dimension i + 1 (any order, multiples of 16), box[i] the
// box extent in dimension i.
bool make_tmap(CUtensorMap *out, CUtensorMapDataType dtype, int rank, const void *base,
               const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
               CUtensorMapSwizzle swizzle);

}  // namespace w4a16
