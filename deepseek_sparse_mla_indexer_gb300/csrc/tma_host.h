// Host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled), fetched
// from the driver at run time so the library needs no link-time libcuda.
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace nsa {

// 2D row-major tensor [rows, cols] of `dtype` with rows `row_pitch_bytes`
// apart; boxes of box_cols x box_rows elements.  Returns false on failure.
bool make_tma_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t cols, uint64_t rows,
                 uint64_t row_pitch_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle);

}  // namespace nsa
