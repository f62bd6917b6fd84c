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

// 3D tensor [d2, d1, d0] (d0 innermost, contiguous) with byte strides
// stride1 (between d1 steps) and stride2 (between d2 steps); boxes b0 x b1 x b2.
bool make_tma_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t d0, uint64_t d1,
                 uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                 CUtensorMapSwizzle swizzle);

}  // namespace nsa
