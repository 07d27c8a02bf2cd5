// tq_tmap.h -- host-side construction of the 2D TMA descriptors (tensor maps)
// the GEMV producer uses to move [rows x bytes] boxes of packed weight codes.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tq {

// Describe codes (n rows of row_bytes) as a 2D uint8 tensor with box
// [box_bytes x box_rows]; out-of-range parts of a box read as zero.
cudaError_t make_codes_tmap(CUtensorMap *out, const uint8_t *codes, int n, size_t row_bytes,
                            uint32_t box_bytes, uint32_t box_rows);

}  // namespace tq
