// tq_stage.cuh -- pieces shared by the dp4a kernel (tq_kernel.cuh) and the
// tensor-core kernel (tq_tc_kernel.cuh): gpu-scope release / acquire
// primitives, the staged element order of a 128-block, the blockwise
// Walsh-Hadamard rotation + int8 quantisation of values held in that order,
// and the pairwise tree of the fold order.
//
// Staged order: the weight decode (tq_dp4a.cuh) produces the weights of a
// block in a fixed permutation (staged_pos); activations are laid out in the
// same permutation so that each 32-bit operand word meets its weights.
#pragma once

#include "tq_dp4a.cuh"

namespace tq {

// Add with release semantics at gpu scope (fire-and-forget): the writes that
// precede it (cumulatively) are visible to whoever observes the sum.
__device__ __forceinline__ void red_add_release_gpu(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Fetch-and-add with acquire-release semantics at gpu scope.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Element of a block at staged position p (the inverse of staged_pos).
template <int FMT>
__device__ __forceinline__ int staged_elem(int p) {
    if (FMT == 0) {
        const int q = p & 15, g = q >> 2;
        return (p & ~15) + (((g & 1) << 3) | ((q & 3) << 1) | (g >> 1));
    }
    return (p & ~31) + 8 * (p & 3) + ((p >> 2) & 7);
}

// One butterfly stage of the 128-point transform on values held in staged
// order (lane l holds staged positions 4l..4l+3 in v[0..3]).  The stage's
// element span maps to a lane bit (xor mask lm) or to a bit of the register
// index (rm); the element with the bit clear keeps a + b, the other a - b.
__device__ __forceinline__ void wht_stage(float (&v)[4], int lane, int lm, int rm) {
    if (lm != 0) {
        const bool upper = (lane & lm) != 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float other = __shfl_xor_sync(0xffffffffu, v[c], lm);
            v[c] = upper ? __fsub_rn(other, v[c]) : __fadd_rn(v[c], other);
        }
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if ((c & rm) == 0) {
                const float x = v[c], y = v[c | rm];
                v[c] = __fadd_rn(x, y);
                v[c | rm] = __fsub_rn(x, y);
            }
    }
}

// The transform's final scale by (float)(1/sqrt(128)), then s = absmax / 127
// and q = round-half-even(v / s) clamped to [-127, 127] (all q = 0 and s = 0
// for an all-zero block) over the warp's 128 values, 4 per lane.  Returns s;
// sum gets the block's sum of codes (every lane).
__device__ __forceinline__ float scale_quant4(float (&v)[4], int8_t (&q)[4], int &sum) {
    const float cs = __uint_as_float(0x3db504f3u);  // (float)(1/sqrt(128))
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = __fmul_rn(v[c], cs);
    // absmax: the order of non-negative floats is that of their bit patterns
    const float lmax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(lmax)));
    const float sc = amax == 0.0f ? 0.0f : __fdiv_rn(amax, 127.0f);
    int lsum = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        int t = 0;
        if (amax != 0.0f) {
            // the clamp matters only when absmax / 127 underflows to zero
            t = __float2int_rn(__fdiv_rn(v[c], sc));
            t = t > 127 ? 127 : (t < -127 ? -127 : t);
        }
        q[c] = static_cast<int8_t>(t);
        lsum += t;
    }
    sum = __reduce_add_sync(0xffffffffu, lsum);
    return sc;
}

// Rotate and quantise one block held in staged order (lane l holds staged
// positions 4l..4l+3 in v): the transform's stages in element-span order,
// then scale_quant4.  word gets the lane's four codes as four consecutive
// staged bytes.
template <int FMT>
__device__ __forceinline__ float rotq_staged(float (&v)[4], int lane, int8_t (&q)[4], uint32_t &word, int &sum) {
    // element span 1, 2, ..., 64 -> (lane xor mask, register bit)
    constexpr int kLm[2][7] = {{2, 0, 0, 1, 4, 8, 16}, {1, 2, 4, 0, 0, 8, 16}};
    constexpr int kRm[2][7] = {{0, 1, 2, 0, 0, 0, 0}, {0, 0, 0, 1, 2, 0, 0}};
#pragma unroll
    for (int st = 0; st < 7; ++st) wht_stage(v, lane, kLm[FMT][st], kRm[FMT][st]);
    const float sc = scale_quant4(v, q, sum);
    word = 0u;
#pragma unroll
    for (int c = 0; c < 4; ++c) word |= (static_cast<uint32_t>(static_cast<uint8_t>(q[c]))) << (8 * c);
    return sc;
}

// Load, in staged order, the four bf16 values of block row `row` (bf16
// [.][n]) lane l rotates: 2-bit staged positions 4l..4l+3 are elements b,
// b+2, b+4, b+6 of the 16-group l/4 (b in {0, 8, 1, 9}), the low or high
// halves of one aligned 16-byte word; 1-bit ones are strided by 8.
template <int FMT>
__device__ __forceinline__ void load_staged_bf16(const uint16_t *blk, int lane, float (&v)[4], bool cached) {
    if (FMT == 0) {
        const int g = lane & 3, b = ((g & 1) << 3) | (g >> 1);
        const uint4 *src = reinterpret_cast<const uint4 *>(blk + (lane >> 2) * 16 + (b & 8));
        const uint4 w = cached ? __ldg(src) : __ldcg(src);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
            v[c] = bf16_bits_to_f32(static_cast<uint16_t>((b & 1) ? (ws[c] >> 16) : (ws[c] & 0xffffu)));
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            v[c] = bf16_bits_to_f32(cached ? __ldg(blk + staged_elem<FMT>(4 * lane + c)) : __ldcg(blk + staged_elem<FMT>(4 * lane + c)));
    }
}

// Pairwise tree over V[0..cnt) (stride `stride` floats), in place: each level
// adds (0,1), (2,3), ... and passes an odd last node up.
__device__ __forceinline__ float fold_tree(float *V, int cnt, int stride) {
    while (cnt > 1) {
        int nxt = 0;
        for (int i = 0; i + 1 < cnt; i += 2, ++nxt)
            V[nxt * stride] = __fadd_rn(V[i * stride], V[(i + 1) * stride]);
        if (cnt & 1) {
            V[nxt * stride] = V[(cnt - 1) * stride];
            ++nxt;
        }
        cnt = nxt;
    }
    return V[0];
}

}  // namespace tq
