// tq_gemv.cuh -- ternary (2-bit) / binary (1-bit) weight-streaming GEMV for a
// packed decode step of M <= 8 activation rows.
//
// Design ("dp4a GEMV with its int8 activation staged in shared memory", "each
// row's lane walk, per-block fold and shuffle tree unchanged" -- sparkinfer PR
// #1154, "decode and small packed batches read the FFN from a ternary copy
// through a dp4a GEMV", Summary and commit message), re-derived for sm_103a:
//
//  * A group of 8 lanes owns one output (NW weight rows at once: NW = 2 reads
//    the gate and the up row of the same output).  Lane p of the group walks
//    blocks b = p, p+8, p+16, ...; per block it loads the row's 32 code bytes
//    (2-bit) or 16 (1-bit) with one 256-/128-bit streaming load, so the 8 lanes
//    read 256 (128) contiguous bytes per step and every byte is used once.
//  * The int8 activation of all M rows is staged once per CTA in shared
//    memory, 144 bytes per 128-block (16 bytes of padding put the 8 lanes'
//    blocks in 8 different bank quads), with its bytes permuted so that a
//    prmt-decoded weight word lines up with one 16-byte shared load.
//  * 2-bit decode: the code word w is masked into nibble selectors
//    (w & 0x33333333, (w >> 2) & 0x33333333) and prmt maps each code through
//    the byte table {0, +1, -1, 0}: 4 signed bytes per prmt, one dp4a each.
//  * 1-bit decode: (w >> s) & 0x01010101 gives 0/1 bytes; the block dot is
//    2 * sum(bit * q) - sum(q), with sum(q) per block precomputed at staging.
//  * Per block the exact int32 dot is folded as t = (float)d * (sw * s) and
//    added to the lane's partial; the 8 partials meet in a xor-shuffle tree
//    (distance 1, 2, 4).  Nothing here depends on M, so a packed row's bits
//    equal its single-row bits.
#pragma once

#include "tq_device.cuh"

namespace tq {

struct GemvArgs {
    const uint8_t *codes[2];
    const uint16_t *scales[2];
    int n;            // outputs (tiles)
    int k;
    const int8_t *q;  // [M][k]
    const float *s;   // [M][k/128]
    float *y;         // [M][n]        (plain GEMV)
    uint16_t *h;      // [M][n] bf16   (gate/up: h = bf16(silu(g) * u))
    int32_t *dots;    // [M][n][k/128] or nullptr
};

template <int FMT> struct FmtTraits;
template <> struct FmtTraits<0> { static constexpr int kBlockBytes = 32; };
template <> struct FmtTraits<1> { static constexpr int kBlockBytes = 16; };

constexpr int kGemvThreads = 256;
constexpr int kTilesPerCta = kGemvThreads / kLanesPerRow;

__host__ __device__ constexpr size_t gemv_smem_bytes(int fmt, int m, int nb) {
    return static_cast<size_t>(m) * nb * kActStride + static_cast<size_t>(m) * nb * 4 +
           (fmt == 1 ? static_cast<size_t>(m) * nb * 4 : 0);
}

// Stage q [M][k] into shared memory in the permuted, padded layout.
template <int FMT, int M>
__device__ __forceinline__ void stage_activation(const int8_t *__restrict__ q,
                                                 const float *__restrict__ s, int k,
                                                 uint8_t *act, float *sact, int *qsum) {
    const int nb = k / kBlock;
    for (int i = threadIdx.x; i < M * nb; i += blockDim.x) {
        sact[i] = s[i];
        if (FMT == 1) qsum[i] = 0;
    }
    if (FMT == 1) __syncthreads();
    if (FMT == 0) {
        // 16-byte chunks: bytes x0..x15 -> [x0 x2 x4 x6][x8 .. x14][x1 .. x7][x9 .. x15]
        const int per_row = k / 16;
        for (int c = threadIdx.x; c < M * per_row; c += blockDim.x) {
            const int mm = c / per_row, off = (c % per_row) * 16;
            const uint4 x = *reinterpret_cast<const uint4 *>(q + static_cast<size_t>(mm) * k + off);
            uint4 o;
            o.x = prmt(x.x, x.y, 0x6420u);
            o.y = prmt(x.z, x.w, 0x6420u);
            o.z = prmt(x.x, x.y, 0x7531u);
            o.w = prmt(x.z, x.w, 0x7531u);
            const int b = off / kBlock, w = (off % kBlock) / 16;
            *reinterpret_cast<uint4 *>(act + (mm * nb + b) * kActStride + 16 * w) = o;
        }
    } else {
        // 32-byte groups: staged word s (s = 0..7) = bytes [x_s, x_{8+s}, x_{16+s}, x_{24+s}]
        const int per_row = k / 32;
        for (int c = threadIdx.x; c < M * per_row; c += blockDim.x) {
            const int mm = c / per_row, off = (c % per_row) * 32;
            const uint4 *src = reinterpret_cast<const uint4 *>(q + static_cast<size_t>(mm) * k + off);
            const uint4 lo = src[0], hi = src[1];
            const uint32_t X[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
            uint32_t o[8];
#pragma unroll
            for (int sl = 0; sl < 8; ++sl) {
                const int j = sl >> 2, by = sl & 3;
                const uint32_t sel = static_cast<uint32_t>(by) | (static_cast<uint32_t>(by + 4) << 4);
                const uint32_t t1 = prmt(X[j], X[j + 2], sel);
                const uint32_t t2 = prmt(X[j + 4], X[j + 6], sel);
                o[sl] = prmt(t1, t2, 0x5410u);
            }
            const int b = off / kBlock, w = (off % kBlock) / 32;
            uint4 *dst = reinterpret_cast<uint4 *>(act + (mm * nb + b) * kActStride + 32 * w);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            int part = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) part = __dp4a(static_cast<int>(X[j]), 0x01010101, part);
            atomicAdd(&qsum[mm * nb + b], part);
        }
    }
    __syncthreads();
}

// 2-bit: exact dot of one 32-byte block with M staged activation rows.
template <int M>
__device__ __forceinline__ void block_dots_t2(const u32x8 &w, const uint8_t *act_b, int nb,
                                              int dot[M]) {
    constexpr uint32_t kTable = 0x00ff0100u;  // code 0 -> 0, 1 -> +1, 2 -> -1, 3 -> 0
#pragma unroll
    for (int mm = 0; mm < M; ++mm) dot[mm] = 0;
#pragma unroll
    for (int wd = 0; wd < 8; ++wd) {
        const uint32_t e = w.v[wd] & 0x33333333u;
        const uint32_t o = (w.v[wd] >> 2) & 0x33333333u;
        const uint32_t p0 = prmt(kTable, kTable, e);
        const uint32_t p1 = prmt(kTable, kTable, e >> 16);
        const uint32_t p2 = prmt(kTable, kTable, o);
        const uint32_t p3 = prmt(kTable, kTable, o >> 16);
#pragma unroll
        for (int mm = 0; mm < M; ++mm) {
            const uint4 a = *reinterpret_cast<const uint4 *>(act_b + mm * nb * kActStride + 16 * wd);
            int d = dot[mm];
            d = dp4a(p0, a.x, d);
            d = dp4a(p1, a.y, d);
            d = dp4a(p2, a.z, d);
            d = dp4a(p3, a.w, d);
            dot[mm] = d;
        }
    }
}

// 1-bit: exact dot of one 16-byte block with M staged activation rows.
template <int M>
__device__ __forceinline__ void block_dots_b1(const uint4 &w4, const uint8_t *act_b, int nb,
                                              const int *qsum_b, int dot[M]) {
    const uint32_t W[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int mm = 0; mm < M; ++mm) dot[mm] = 0;
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
        uint32_t bits[8];
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) bits[sl] = (W[wd] >> sl) & 0x01010101u;
#pragma unroll
        for (int mm = 0; mm < M; ++mm) {
            const uint4 *a = reinterpret_cast<const uint4 *>(act_b + mm * nb * kActStride + 32 * wd);
            const uint4 lo = a[0], hi = a[1];
            int d = dot[mm];
            d = dp4a(bits[0], lo.x, d);
            d = dp4a(bits[1], lo.y, d);
            d = dp4a(bits[2], lo.z, d);
            d = dp4a(bits[3], lo.w, d);
            d = dp4a(bits[4], hi.x, d);
            d = dp4a(bits[5], hi.y, d);
            d = dp4a(bits[6], hi.z, d);
            d = dp4a(bits[7], hi.w, d);
            dot[mm] = d;
        }
    }
#pragma unroll
    for (int mm = 0; mm < M; ++mm) dot[mm] = 2 * dot[mm] - qsum_b[mm * nb];
}

// NW = 1: y[mm][n] = GEMV.  NW = 2 (gate/up): h[mm][n] = bf16(silu(g) * u).
template <int FMT, int M, int NW>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int k = a.k, nb = k / kBlock;
    uint8_t *act = smem;
    float *sact = reinterpret_cast<float *>(smem + static_cast<size_t>(M) * nb * kActStride);
    int *qsum = reinterpret_cast<int *>(sact + M * nb);

    stage_activation<FMT, M>(a.q, a.s, k, act, sact, qsum);

    const int lane = threadIdx.x & 31;
    const int p = lane & (kLanesPerRow - 1);
    const int tile = blockIdx.x * kTilesPerCta + (threadIdx.x >> 3);
    const bool active = tile < a.n;

    float acc[NW][M];
#pragma unroll
    for (int r = 0; r < NW; ++r)
#pragma unroll
        for (int mm = 0; mm < M; ++mm) acc[r][mm] = 0.0f;

    if (active) {
        constexpr int BB = FmtTraits<FMT>::kBlockBytes;
        const size_t row_bytes = static_cast<size_t>(nb) * BB;
        const uint8_t *wrow[NW];
        const uint16_t *srow[NW];
#pragma unroll
        for (int r = 0; r < NW; ++r) {
            wrow[r] = a.codes[r] + static_cast<size_t>(tile) * row_bytes;
            srow[r] = a.scales[r] + static_cast<size_t>(tile) * nb;
        }
        for (int b = p; b < nb; b += kLanesPerRow) {
            const uint8_t *act_b = act + b * kActStride;
#pragma unroll
            for (int r = 0; r < NW; ++r) {
                int dot[M];
                if (FMT == 0) {
                    const u32x8 w = ldg_stream_32B(wrow[r] + static_cast<size_t>(b) * BB);
                    block_dots_t2<M>(w, act_b, nb, dot);
                } else {
                    const uint4 w = ldg_stream_16B(wrow[r] + static_cast<size_t>(b) * BB);
                    block_dots_b1<M>(w, act_b, nb, qsum + b, dot);
                }
                const float swf = f16_bits_to_f32(ldg_u16(srow[r] + b));
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    const float t = __fmul_rn(__int2float_rn(dot[mm]),
                                              __fmul_rn(swf, sact[mm * nb + b]));
                    acc[r][mm] = __fadd_rn(acc[r][mm], t);
                }
                if (NW == 1 && a.dots != nullptr) {
#pragma unroll
                    for (int mm = 0; mm < M; ++mm)
                        a.dots[(static_cast<size_t>(mm) * a.n + tile) * nb + b] = dot[mm];
                }
            }
        }
    }
    // fixed tree over the 8 partials: distance 1, 2, 4 (fp32 add commutes, so
    // both partners of each exchange hold the same sum)
#pragma unroll
    for (int r = 0; r < NW; ++r)
#pragma unroll
        for (int mm = 0; mm < M; ++mm) {
            float v = acc[r][mm];
            v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
            v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
            v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
            acc[r][mm] = v;
        }
    if (active && p == 0) {
#pragma unroll
        for (int mm = 0; mm < M; ++mm) {
            if (NW == 1) {
                a.y[static_cast<size_t>(mm) * a.n + tile] = acc[0][mm];
            } else {
                const float hv = __fmul_rn(tq_silu(acc[0][mm]), acc[NW - 1][mm]);
                a.h[static_cast<size_t>(mm) * a.n + tile] = f32_to_bf16_bits(hv);
            }
        }
    }
}

}  // namespace tq
