// t2s_tmap.h -- TMA tensor-map encoding for row-major FP32 matrices.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace t2s {

// Encodes a 2-D tiled tensor map over a row-major FP32 matrix of `rows` rows of
// `cols` elements (row stride = cols * 4 bytes), with a box of box_cols x box_rows
// elements, the given swizzle, and zero fill outside the matrix.
// Requirements checked by the driver: base 16-byte aligned, row stride a multiple of
// 16 bytes, box extents <= 256, box_cols * 4 a multiple of 16 bytes (and <= the
// swizzle span when swizzled). Returns cudaErrorInvalidValue if the driver rejects
// the map, or the error from looking up the driver entry point.
cudaError_t encode_tmap_f32_2d(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                               uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle);

// The same for a row-major matrix of 16-bit BF16 elements (row stride = cols * 2 bytes).
cudaError_t encode_tmap_bf16_2d(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                                uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle);

}  // namespace t2s
