// tq_dp4a.cuh -- the compute core of the ternary GEMV: packed codes decode
// with prmt into bytes that dp4a multiplies with the int8 activation.
//
// Exactness is by construction: every block dot is an int32 sum of int8
// products, converted to fp32 exactly (|d| < 2^22).
//
// 2-bit: codes 0, 1, 2 (weights 0, +1, -1) decode to the biased bytes
// w + 1 = 1, 2, 0, one prmt per four codes.  A selector nibble holding two
// codes (c_hi at bits 2-3, c_lo at bits 0-1) picks byte 4 * (c_hi & 1) + c_lo
// of the pool {kTableB : kTableA} = {2 2 2 2 : 1 1 1 1}, or, for c_hi = 2 (bit
// 3), that byte's sign replicated: 0.  Every byte of a table half is the
// same, so c_lo does not matter and the nibble decodes c_hi: w itself decodes
// the odd codes of its low half, w >> 16 those of its high half, w << 2 and
// w >> 14 (each even code moved to the top of a nibble) the even ones.  The
// bias leaves the block exactly: d = sum((w+1)*q) - sum(q).  A word of codes
// 0..15 gives the dp4a operands of weights [0 2 4 6], [8 10 12 14],
// [1 3 5 7], [9 11 13 15].
// 1-bit: bit e of a row's block is weight e (1 -> +1, 0 -> -1); register s
// (0..7) of a word holds bits s, 8+s, 16+s, 24+s as bytes 0/1 and
// d = 2*sum(b*q) - sum(q).
// The activation is staged in shared memory in these orders, so each operand
// register meets one 32-bit word of it.
#pragma once

#include "tq_device.cuh"

namespace tq {

constexpr int kTileRows = 16;       // weight rows per unit
constexpr int kSegBlocks = 8;       // 128-blocks per segment (fold order)

constexpr uint32_t kTableA = 0x01010101u;
constexpr uint32_t kTableB = 0x02020202u;

__device__ __forceinline__ void decode_t2(uint32_t w, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    r0 = prmt(kTableA, kTableB, w << 2);
    r1 = prmt(kTableA, kTableB, w >> 14);
    r2 = prmt(kTableA, kTableB, w);
    r3 = prmt(kTableA, kTableB, w >> 16);
}

// Position of element e (0..127) of a block in its staged 128 bytes.
template <int FMT>
__host__ __device__ __forceinline__ int staged_pos(int e) {
    if (FMT == 0) {
        // per 16 weights: [0 2 4 6 | 8 10 12 14 | 1 3 5 7 | 9 11 13 15]
        const int r = e & 15;
        return (e & ~15) + 4 * (2 * (r & 1) + (r >> 3)) + ((r >> 1) & 3);
    }
    // per 32 weights: byte 4s + k holds weight 8k + s
    return (e & ~31) + 4 * (e & 7) + ((e >> 3) & 3);
}

// Exact int -> float for |i| < 2^22 through the fp32 bit pattern of 2^23 + 2^22:
// (float)(i + bias) where `magic_minus_bias` = 0x4b400000 - bias.
constexpr int kMagic = 0x4b400000;

}  // namespace tq
