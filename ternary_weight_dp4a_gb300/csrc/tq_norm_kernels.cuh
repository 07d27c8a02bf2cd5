// tq_norm_kernels.cuh -- the standalone rotation / RMS-normalise kernels.
// Included by exactly one translation unit (tq_api.cu).
#pragma once

#include "tq_rotq.cuh"

namespace tq {

// x: bf16 bits [m][k] -> q int8 [m][k], s fp32 [m][k/128].  One warp per
// (row, block); blockDim.x = 256.  Launched as a programmatic dependent: it
// reads x only after its predecessor in the stream has completed.
__global__ void __launch_bounds__(256) rotate_quant_kernel(const uint16_t *__restrict__ x,
                                                           int64_t nblocks_total, int k,
                                                           int8_t *__restrict__ q,
                                                           float *__restrict__ s) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t gb = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gb >= nblocks_total) return;
    const int nb = k / kBlock;
    const int64_t row = gb / nb;
    const int b = static_cast<int>(gb % nb);
    const uint16_t *xb = x + row * k + static_cast<int64_t>(b) * kBlock;
    float v[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = bf16_bits_to_f32(xb[lane + 32 * c]);
    rotq_block_store(v, lane, q + row * k + static_cast<int64_t>(b) * kBlock, s + gb);
}

// RMS-normalise then rotate + quantise, one CTA of 256 threads per row:
// x = bf16_rn(y * (1 / sqrt(sum(y^2)/n + eps))) with sum(y^2) as 256 partial
// sums (thread t adds y[t], y[t+256], ... in order) combined pairwise at
// distance 1, 2, ..., 128; then each warp rotates and quantises blocks
// w, w+8, ... of the row.  Optionally also writes the bf16 row to x_out.
constexpr int kNormThreads = 256;

__device__ __forceinline__ float row_inv_rms(const float *__restrict__ yr, int n, float eps,
                                             float *warp_sum) {
    const int t = threadIdx.x;
    float acc = 0.0f;
    for (int i = t; i < n; i += kNormThreads) acc = __fadd_rn(acc, __fmul_rn(yr[i], yr[i]));
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    if ((t & 31) == 0) warp_sum[t >> 5] = acc;
    __syncthreads();
    const float w01 = __fadd_rn(warp_sum[0], warp_sum[1]);
    const float w23 = __fadd_rn(warp_sum[2], warp_sum[3]);
    const float w45 = __fadd_rn(warp_sum[4], warp_sum[5]);
    const float w67 = __fadd_rn(warp_sum[6], warp_sum[7]);
    const float ss = __fadd_rn(__fadd_rn(w01, w23), __fadd_rn(w45, w67));
    const float ms = __fdiv_rn(ss, static_cast<float>(n));
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

__global__ void __launch_bounds__(kNormThreads) rmsnorm_rotq_kernel(
    const float *__restrict__ y, int n, float eps, int8_t *__restrict__ q, float *__restrict__ s,
    uint16_t *__restrict__ x_out) {
    __shared__ float warp_sum[kNormThreads / 32];
    pdl_launch_dependents();
    pdl_wait();
    const float *yr = y + static_cast<size_t>(blockIdx.x) * n;
    const float inv = row_inv_rms(yr, n, eps, warp_sum);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = n / kBlock;
    for (int b = warp; b < nb; b += kNormThreads / 32) {
        float v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int i = b * kBlock + lane + 32 * c;
            const uint16_t xb = f32_to_bf16_bits(__fmul_rn(yr[i], inv));
            if (x_out != nullptr) x_out[static_cast<size_t>(blockIdx.x) * n + i] = xb;
            v[c] = bf16_bits_to_f32(xb);
        }
        rotq_block_store(v, lane, q + static_cast<size_t>(blockIdx.x) * n + b * kBlock,
                         s + static_cast<size_t>(blockIdx.x) * nb + b);
    }
}

// Plain RMS-normalise to bf16 (one CTA of 256 threads per row).
__global__ void __launch_bounds__(kNormThreads) rmsnorm_bf16_kernel(const float *__restrict__ y,
                                                                    int n, float eps,
                                                                    uint16_t *__restrict__ x) {
    __shared__ float warp_sum[kNormThreads / 32];
    pdl_launch_dependents();
    pdl_wait();
    const float *yr = y + static_cast<size_t>(blockIdx.x) * n;
    uint16_t *xr = x + static_cast<size_t>(blockIdx.x) * n;
    const float inv = row_inv_rms(yr, n, eps, warp_sum);
    for (int i = threadIdx.x; i < n; i += kNormThreads) xr[i] = f32_to_bf16_bits(__fmul_rn(yr[i], inv));
}

}  // namespace tq
