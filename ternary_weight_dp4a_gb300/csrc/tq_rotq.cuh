// tq_rotq.cuh -- blockwise 128-point Walsh-Hadamard rotation + int8 absmax
// quantisation, one warp per 128-element block.
//
// "the Hadamard rotation emits that int8 copy for gate and up to share"
// (sparkinfer PR #1154, "decode and small packed batches read the FFN from a
// ternary copy through a dp4a GEMV", Summary).  The transform is the fast
// butterfly network in natural order, span 1, 2, 4, ..., 64; each stage is an
// elementwise IEEE add/sub, so spreading it over lanes and registers gives the
// same bits as any sequential evaluation of the same stages.
#pragma once

#include "tq_device.cuh"

namespace tq {

// Lane l holds elements l, l+32, l+64, l+96 of one block in v[0..3]; the block
// is rotated in place.  All 32 lanes must call.
__device__ __forceinline__ void wht128_warp(float v[4], int lane) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
        const bool upper = (lane & h) != 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float other = __shfl_xor_sync(0xffffffffu, v[c], h);
            // lower index keeps a+b, upper index keeps a-b (a = lower, b = upper)
            v[c] = upper ? __fsub_rn(other, v[c]) : __fadd_rn(v[c], other);
        }
    }
    // span 32: element pairs (c=0,c=1) and (c=2,c=3); span 64: (0,2), (1,3)
    {
        const float a0 = v[0], b0 = v[1], a1 = v[2], b1 = v[3];
        v[0] = __fadd_rn(a0, b0); v[1] = __fsub_rn(a0, b0);
        v[2] = __fadd_rn(a1, b1); v[3] = __fsub_rn(a1, b1);
    }
    {
        const float a0 = v[0], b0 = v[2], a1 = v[1], b1 = v[3];
        v[0] = __fadd_rn(a0, b0); v[2] = __fsub_rn(a0, b0);
        v[1] = __fadd_rn(a1, b1); v[3] = __fsub_rn(a1, b1);
    }
    const float c = __uint_as_float(0x3db504f3u);  // (float)(1/sqrt(128))
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __fmul_rn(v[i], c);
}

// Quantise a rotated block held as in wht128_warp: returns s, writes this
// lane's four int8 codes to q[4].
__device__ __forceinline__ float quant_block_warp(const float v[4], int8_t q[4]) {
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (amax == 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = 0;
        return 0.0f;
    }
    const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int t = __float2int_rn(__fdiv_rn(v[i], s));
        t = t > 127 ? 127 : (t < -127 ? -127 : t);
        q[i] = static_cast<int8_t>(t);
    }
    return s;
}

// Rotate + quantise one block whose four per-lane values are already loaded;
// writes q (global layout) and s.
__device__ __forceinline__ void rotq_block_store(float v[4], int lane, int8_t *qb, float *sb) {
    wht128_warp(v, lane);
    int8_t qq[4];
    const float sc = quant_block_warp(v, qq);
#pragma unroll
    for (int c = 0; c < 4; ++c) qb[lane + 32 * c] = qq[c];
    if (lane == 0) *sb = sc;
}

}  // namespace tq
