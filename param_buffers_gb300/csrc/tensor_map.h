// Host-side encoding of TMA tensor maps (2-D, row-major) through the driver entry point
// looked up at run time, so the library does not link libcuda directly.
#pragma once
#include <cuda.h>

#include <cstdint>

#include "gtp.h"

namespace gtp {

// A 2-D row-major tensor: `inner` contiguous elements per row, `outer` rows,
// `row_stride_bytes` between rows (a multiple of 16).  The box is box_inner x box_outer
// elements; `swizzle` is a CU_TENSOR_MAP_SWIZZLE_* value.  Out-of-bounds loads read zeros.
gtp_status encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                          uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle);

}  // namespace gtp
