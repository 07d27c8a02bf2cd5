// tq_misc.cuh -- weight packing (load time) and the RMS-normalise used between
// stacked FFN layers.
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

// One CTA of 256 threads per row.  Thread t sums y[i]^2 for i = t, t+256, ...
// in ascending order; the 256 partials combine at distance 1, 2, ..., 128
// (xor shuffles inside each warp, then the 8 warp sums as a fixed tree).
constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_bf16_kernel(const float *__restrict__ y,
                                                                    int n, float eps,
                                                                    uint16_t *__restrict__ x) {
    __shared__ float warp_sum[kNormThreads / 32];
    __shared__ float inv_s;
    const float *yr = y + static_cast<size_t>(blockIdx.x) * n;
    uint16_t *xr = x + static_cast<size_t>(blockIdx.x) * n;
    const int t = threadIdx.x;
    float acc = 0.0f;
    for (int i = t; i < n; i += kNormThreads) acc = __fadd_rn(acc, __fmul_rn(yr[i], yr[i]));
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    if ((t & 31) == 0) warp_sum[t >> 5] = acc;
    __syncthreads();
    if (t == 0) {
        const float w01 = __fadd_rn(warp_sum[0], warp_sum[1]);
        const float w23 = __fadd_rn(warp_sum[2], warp_sum[3]);
        const float w45 = __fadd_rn(warp_sum[4], warp_sum[5]);
        const float w67 = __fadd_rn(warp_sum[6], warp_sum[7]);
        const float ss = __fadd_rn(__fadd_rn(w01, w23), __fadd_rn(w45, w67));
        const float ms = __fdiv_rn(ss, static_cast<float>(n));
        inv_s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    }
    __syncthreads();
    const float inv = inv_s;
    for (int i = t; i < n; i += kNormThreads) xr[i] = f32_to_bf16_bits(__fmul_rn(yr[i], inv));
}

}  // namespace tq
