// tq_misc.cuh -- weight packing (a load-time step).
#pragma once

#include "tq_device.cuh"

namespace tq {

// codes [n][k] (one code per byte) -> packed bytes.  One thread per output
// byte; each reads 4 (2-bit) or 8 (1-bit) consecutive codes.
template <int FMT>
__global__ void pack_kernel(const uint8_t *__restrict__ codes, int64_t out_bytes,
                            uint8_t *__restrict__ packed) {
    constexpr int per = FMT == 0 ? 4 : 8;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < out_bytes;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint8_t *c = codes + i * per;
        uint32_t byte = 0;
#pragma unroll
        for (int t = 0; t < per; ++t)
            byte |= FMT == 0 ? (static_cast<uint32_t>(c[t] & 3u) << (2 * t))
                             : (static_cast<uint32_t>(c[t] & 1u) << t);
        packed[i] = static_cast<uint8_t>(byte);
    }
}

}  // namespace tq
