// tq_tmap.h -- host-side construction of the 2D TMA descriptors (tensor maps)
// the kernels' producer warp uses to move [16 rows x segment] boxes of packed
// weight codes and scales.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tq {

// Describe `rows` rows of `inner` elements (elem_bytes each, row stride
// row_stride_bytes, a multiple of 16) as a 2D tensor with box
// [box_inner x box_rows]; out-of-range parts of a box read as zero.
cudaError_t make_tmap_2d(CUtensorMap *out, CUtensorMapDataType dtype, const void *base,
                         uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                         uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);

// The 2-bit codes of `rows` rows of row_bytes (a multiple of 128) as a 3D
// uint8 tensor {128, row_bytes/128 planes, rows} with box {128, 2, 16} and the
// 128-byte swizzle: one copy brings 16 rows x 256 bytes, each row's two
// 128-byte planes adjacent.
cudaError_t make_codes_tmap_3d(CUtensorMap *out, const void *base, uint64_t row_bytes, uint64_t rows);

}  // namespace tq
