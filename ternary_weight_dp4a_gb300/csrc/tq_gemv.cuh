// tq_gemv.cuh -- ternary (2-bit) / binary (1-bit) weight-streaming GEMV for a
// packed decode step of M <= 8 activation rows, and the fused gate/up variant.
//
// Design ("dp4a GEMV with its int8 activation staged in shared memory", "each
// row's lane walk, per-block fold and shuffle tree unchanged" -- sparkinfer PR
// #1154, "decode and small packed batches read the FFN from a ternary copy
// through a dp4a GEMV", Summary and commit message), re-derived for sm_103a:
//
//  * A CTA owns a tile of T = 4 * NCW consecutive outputs and has NCW consumer
//    warps plus one producer warp.  The producer streams the tile's weight
//    rows through an S-stage shared-memory ring with bulk copies (the TMA
//    engine, cp.async.bulk + mbarrier): stage k holds, for every row of the
//    tile, the 8 consecutive 128-weight blocks 8k .. 8k+7.  It starts before
//    the kernel waits on its predecessor in the stream (programmatic
//    dependent launch), so HBM keeps streaming across kernel boundaries.
//  * Each output is owned by a group of 8 consumer lanes.  Lane p walks blocks
//    b = p, p+8, p+16, ... -- in stage k it handles block 8k + p -- so one
//    stage gives every lane exactly one block per row.
//  * The int8 activation of all M rows is staged once per CTA in shared
//    memory, 144 bytes per 128-block (16 bytes of padding put the 8 lanes'
//    blocks in 8 different bank quads), permuted so each decoded weight word
//    meets one 16-byte shared load, plus per block its scale and sum(q).
//  * 2-bit decode: prmt maps codes to value+1 (see decode_t2); 1-bit decode:
//    (w >> s) & 0x01010101 gives 0/1 bytes.  The exact block dot is
//    sum(dec * q) - sum(q) (2-bit) or 2 * sum(bit * q) - sum(q) (1-bit).
//  * Per block, t = (float)d * (sw * s) is added to the lane's partial; the 8
//    partials meet in a xor-shuffle tree (distance 1, 2, 4).  Nothing here
//    depends on M, so a packed row's bits equal its single-row bits.
//  * Gate/up epilogue: h = bf16(silu(g) * u) is stored; the last CTA to
//    finish each 128-block of h (atomic counter, no waiting) rotates and
//    quantises that block for the down GEMV and resets the counter.
#pragma once

#include <cuda.h>

#include "tq_device.cuh"
#include "tq_rotq.cuh"

namespace tq {

struct GemvArgs {
    CUtensorMap tmap[2];       // codes of [0] / [1] as 2D uint8 tensors, box [seg x T]
    const uint8_t *codes[2];   // [0]: the matrix (or gate), [1]: up
    const uint16_t *scales[2];
    int n;                     // outputs
    int k;
    const int8_t *q;           // [M][k] activation
    const float *s;            // [M][k/128]
    float *y;                  // plain GEMV: [M][n]
    uint16_t *h;               // gate/up: [M][n] bf16
    int8_t *qh;                // gate/up with h rotation: [M][n]
    float *sh;                 // [M][n/128]
    unsigned *counters;        // [n/128], zero on entry and on exit
    int32_t *dots;             // [M][n][k/128] or nullptr
    unsigned *err;             // error word (a bounded wait ran out), or nullptr
};

template <int FMT> struct FmtTraits;
template <> struct FmtTraits<0> { static constexpr int kBlockBytes = 32; };
template <> struct FmtTraits<1> { static constexpr int kBlockBytes = 16; };

constexpr int kBlocksPerBox = 8;        // one block per lane per box
constexpr int kBoxesPerStage = 2;       // two blocks per lane per stage
constexpr int kBlocksPerStage = kBlocksPerBox * kBoxesPerStage;

// Shared-memory bytes of one CTA (dynamic part).
__host__ __device__ constexpr size_t gemv_ring_bytes(int fmt, int mats, int ncw, int stages) {
    // + 1024 to align the ring start for the tensor copies
    return static_cast<size_t>(stages) * mats * (4 * ncw) * kBlocksPerStage *
               (fmt == 0 ? 32 : 16) + 1024;
}
// stage layout: [matrix][box][tile row][box width]
__host__ __device__ constexpr size_t gemv_act_bytes(int m, int nb) {
    // staged activation + per-block fp32 scale + per-block int (magic - sum q),
    // rounded up to 16 bytes
    return (static_cast<size_t>(m) * nb * (kActStride + 4 + 4) + 15) / 16 * 16;
}
// per matrix: the CTA's fp16 scales plus up to 16 bytes of alignment slack on
// each side, rounded to 16 bytes
__host__ __device__ constexpr size_t gemv_scale_region(int outs, int nb) {
    return (static_cast<size_t>(outs) * nb * 2 + 32 + 15) / 16 * 16;
}
__host__ __device__ constexpr size_t gemv_scale_bytes(int mats, int outs, int nb) {
    return static_cast<size_t>(mats) * gemv_scale_region(outs, nb);
}

// Stage q [M][k] into shared memory in the permuted, padded layout, with
// sact[mm][b] = s and cmag[mm][b] = 0x4b400000 - sum(q of the block).  Run by
// the first `nthr` threads of the CTA, which synchronise on named barrier 1.
template <int FMT, int M>
__device__ __forceinline__ void stage_activation(const int8_t *__restrict__ q,
                                                 const float *__restrict__ s, int k,
                                                 uint8_t *act, float *sact, int *cmag, int nthr) {
    const int nb = k / kBlock;
    for (int i = threadIdx.x; i < M * nb; i += nthr) {
        sact[i] = s[i];
        cmag[i] = 0x4b400000;
    }
    named_barrier(1, nthr);
    const int per_row = k / 32;
    for (int c = threadIdx.x; c < M * per_row; c += nthr) {
        const int mm = c / per_row, off = (c % per_row) * 32;
        const uint4 *src = reinterpret_cast<const uint4 *>(q + static_cast<size_t>(mm) * k + off);
        const uint4 lo = src[0], hi = src[1];
        const uint32_t X[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        const int b = off / kBlock;
        uint8_t *dst = act + (mm * nb + b) * kActStride + (off % kBlock);
        if (FMT == 0) {
            // per 16 bytes x0..x15 -> [x0 x2 x4 x6][x8 .. x14][x1 .. x7][x9 .. x15]
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint4 o;
                o.x = prmt(X[4 * h + 0], X[4 * h + 1], 0x6420u);
                o.y = prmt(X[4 * h + 2], X[4 * h + 3], 0x6420u);
                o.z = prmt(X[4 * h + 0], X[4 * h + 1], 0x7531u);
                o.w = prmt(X[4 * h + 2], X[4 * h + 3], 0x7531u);
                *reinterpret_cast<uint4 *>(dst + 16 * h) = o;
            }
        } else {
            // per 32 bytes: staged word s (s = 0..7) = [x_s, x_{8+s}, x_{16+s}, x_{24+s}]
            uint32_t o[8];
#pragma unroll
            for (int sl = 0; sl < 8; ++sl) {
                const int j = sl >> 2, by = sl & 3;
                const uint32_t sel = static_cast<uint32_t>(by) | (static_cast<uint32_t>(by + 4) << 4);
                const uint32_t t1 = prmt(X[j], X[j + 2], sel);
                const uint32_t t2 = prmt(X[j + 4], X[j + 6], sel);
                o[sl] = prmt(t1, t2, 0x5410u);
            }
            reinterpret_cast<uint4 *>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<uint4 *>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
        int part = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) part = __dp4a(static_cast<int>(X[j]), 0x01010101, part);
        atomicSub(&cmag[mm * nb + b], part);
    }
    named_barrier(1, nthr);
}

// Raw (biased) dots of NBLK blocks x R weight rows (code words in
// w[blk][r][8] (2-bit) or w[blk][r][4] (1-bit)); block blk meets the staged
// activation block at act_b[blk], for M activation rows.
// 2-bit: sum((w+1) * q); 1-bit: sum(bit * q).
template <int FMT, int M, int NBLK, int R>
__device__ __forceinline__ void block_dots(const uint32_t (&w)[NBLK][R][8],
                                           const uint8_t *const (&act_b)[NBLK], int nb,
                                           int (&dot)[NBLK][R][M]) {
#pragma unroll
    for (int x = 0; x < NBLK; ++x)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int mm = 0; mm < M; ++mm) dot[x][r][mm] = 0;
    if constexpr (FMT == 0) {
        int dot2[NBLK][R][M];   // a second chain: words 4..7 (exact ints, summed at the end)
#pragma unroll
        for (int x = 0; x < NBLK; ++x)
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int mm = 0; mm < M; ++mm) dot2[x][r][mm] = 0;
#pragma unroll
        for (int wd = 0; wd < 8; ++wd) {
#pragma unroll
            for (int x = 0; x < NBLK; ++x) {
                Decoded4 d[R];
#pragma unroll
                for (int r = 0; r < R; ++r) d[r] = decode_t2(w[x][r][wd]);
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    const uint4 a = *reinterpret_cast<const uint4 *>(act_b[x] + mm * nb * kActStride + 16 * wd);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        int v = wd < 4 ? dot[x][r][mm] : dot2[x][r][mm];
                        v = dp4a(d[r].p[0], a.x, v);
                        v = dp4a(d[r].p[1], a.y, v);
                        v = dp4a(d[r].p[2], a.z, v);
                        v = dp4a(d[r].p[3], a.w, v);
                        if (wd < 4) dot[x][r][mm] = v; else dot2[x][r][mm] = v;
                    }
                }
            }
        }
#pragma unroll
        for (int x = 0; x < NBLK; ++x)
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int mm = 0; mm < M; ++mm) dot[x][r][mm] += dot2[x][r][mm];
    } else {
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
            for (int x = 0; x < NBLK; ++x) {
                uint32_t bits[R][8];
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int sl = 0; sl < 8; ++sl) bits[r][sl] = (w[x][r][wd] >> sl) & 0x01010101u;
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    const uint4 *ap = reinterpret_cast<const uint4 *>(act_b[x] + mm * nb * kActStride + 32 * wd);
                    const uint4 lo = ap[0], hi = ap[1];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        int v = dot[x][r][mm];
                        v = dp4a(bits[r][0], lo.x, v);
                        v = dp4a(bits[r][1], lo.y, v);
                        v = dp4a(bits[r][2], lo.z, v);
                        v = dp4a(bits[r][3], lo.w, v);
                        v = dp4a(bits[r][4], hi.x, v);
                        v = dp4a(bits[r][5], hi.y, v);
                        v = dp4a(bits[r][6], hi.z, v);
                        v = dp4a(bits[r][7], hi.w, v);
                        dot[x][r][mm] = v;
                    }
                }
            }
        }
    }
}

// Dots of NBLK consecutive-in-chain blocks (b0, b0 + 8, ...) of this lane's R
// rows from the stage, folded into acc in chain order.
template <int FMT, int M, int NBLK, int R, bool DOTS>
__device__ __forceinline__ void stage_blocks(const uint8_t *stage, int T, int rs, int g, int p,
                                             int b0, const uint8_t *act, const float *sact,
                                             const int *cmag, const __half *sw0,
                                             const __half *sw1, int nb, float (&acc)[R][M],
                                             int32_t *dots_out, size_t dots_row_stride) {
    constexpr int BB = FmtTraits<FMT>::kBlockBytes;
    uint32_t w[NBLK][R][8];
    const uint8_t *act_b[NBLK];
#pragma unroll
    for (int x = 0; x < NBLK; ++x) {
        act_b[x] = act + (b0 + x * kBlocksPerBox) * kActStride;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t *seg = stage + ((r * kBoxesPerStage + x) * T + g) * rs + p * BB;
            const uint4 x0 = *reinterpret_cast<const uint4 *>(seg);
            w[x][r][0] = x0.x; w[x][r][1] = x0.y; w[x][r][2] = x0.z; w[x][r][3] = x0.w;
            if constexpr (FMT == 0) {
                const uint4 x1 = *reinterpret_cast<const uint4 *>(seg + 16);
                w[x][r][4] = x1.x; w[x][r][5] = x1.y; w[x][r][6] = x1.z; w[x][r][7] = x1.w;
            } else {
                w[x][r][4] = w[x][r][5] = w[x][r][6] = w[x][r][7] = 0u;
            }
        }
    }
    int dot[NBLK][R][M];
    block_dots<FMT, M, NBLK, R>(w, act_b, nb, dot);
#pragma unroll
    for (int x = 0; x < NBLK; ++x) {
        const int b = b0 + x * kBlocksPerBox;
#pragma unroll
        for (int mm = 0; mm < M; ++mm) {
            const float sa = sact[mm * nb + b];
            const int cm = cmag[mm * nb + b];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                // exact (float)(block dot): remove the decode bias
                const int raw = FMT == 0 ? dot[x][r][mm] : 2 * dot[x][r][mm];
                const float df = int_to_float_exact(raw, cm);
                const float ws = __half2float((r == 0 ? sw0 : sw1)[b]);
                acc[r][mm] = __fadd_rn(acc[r][mm], __fmul_rn(df, __fmul_rn(ws, sa)));
                if (DOTS) dots_out[mm * dots_row_stride + b] = raw - (0x4b400000 - cm);
            }
        }
    }
}

// CTA c of G owns outputs [c*n/G, (c+1)*n/G), processed in tiles of up to
// T = 4 * NCW outputs (one per 8-lane group).  Dynamic shared memory:
//   ring [S][R][T][8 blocks] | activation | sact | cmag | scales f32 [R][outs][nb]
__host__ __device__ constexpr int gemv_cta_outputs_max(int n, int grid) {
    return (n + grid - 1) / grid;
}

// FMT: 0 = 2-bit, 1 = 1-bit.  M: activation rows.  GATEUP: two matrices (gate,
// up) and the SiLU*up epilogue.  NCW: consumer warps.  S: ring stages.
template <int FMT, int M, bool GATEUP, int NCW, int S>
__global__ void __launch_bounds__(32 * (NCW + 1)) gemv_kernel(const __grid_constant__ GemvArgs a) {
    constexpr int R = GATEUP ? 2 : 1;                 // weight rows per output
    constexpr int T = 4 * NCW;                        // outputs per tile
    constexpr int BB = FmtTraits<FMT>::kBlockBytes;
    constexpr int kBoxW = kBlocksPerBox * BB;         // box width in bytes
    constexpr int kStageBytes = R * kBoxesPerStage * T * kBoxW;
    constexpr int kConsumers = 32 * NCW;

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[S];
    __shared__ __align__(8) uint64_t empty_bar[S];
    __shared__ __align__(8) uint64_t scale_bar;
    __shared__ int s_last[2];

    const int k = a.k, nb = k / kBlock;
    const int spt = (nb + kBlocksPerStage - 1) / kBlocksPerStage;   // stages per tile
    const size_t row_bytes = static_cast<size_t>(nb) * BB;
    const int rs = nb < kBlocksPerBox ? nb * BB : kBoxW;              // box width in bytes
    const int box_rows = a.n < T ? a.n : T;
    const int n_beg = static_cast<int>((static_cast<long long>(a.n) * blockIdx.x) / gridDim.x);
    const int n_end = static_cast<int>((static_cast<long long>(a.n) * (blockIdx.x + 1)) / gridDim.x);
    const int outs = n_end - n_beg;
    const int tiles = (outs + T - 1) / T;
    const int nst = tiles * spt;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // tensor copies land at 1024-byte-aligned stage bases
    uint8_t *ring = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
    // (the scale regions below start 16-byte aligned: every size before is a
    // multiple of 16)
    uint8_t *act = ring + static_cast<size_t>(S) * kStageBytes;
    float *sact = reinterpret_cast<float *>(act + static_cast<size_t>(M) * nb * kActStride);
    int *cmag = reinterpret_cast<int *>(sact + M * nb);
    // per matrix: fp16 scales of outputs [n_beg, n_end); element i at sw_base[r] + i
    uint8_t *swreg = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(cmag + M * nb) + 15) & ~static_cast<uintptr_t>(15));
    const size_t sreg = gemv_scale_region(outs, nb);
    const size_t sbyte0 = static_cast<size_t>(n_beg) * nb * 2;          // global byte offset
    const int shead = static_cast<int>(sbyte0 & 15);                     // its misalignment

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), NCW);
        }
        mbar_init(smem_u32(&scale_bar), 1);
        mbar_init_fence();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        // Weights are never written by earlier work in the stream, so the ring
        // fills before (and while) the kernel waits on its predecessor.
        if (lane == 0) {
            // the CTA's weight scales: the 16-byte-aligned span around
            // [sbyte0, sbyte0 + 2*outs*nb); a span that would run past the end of
            // the scale array stops short and the consumers fetch the rest
            const size_t total = static_cast<size_t>(a.n) * nb * 2;
            const size_t g0 = sbyte0 - shead;
            size_t g1 = (sbyte0 + static_cast<size_t>(outs) * nb * 2 + 15) & ~static_cast<size_t>(15);
            if (g1 > total) g1 = total & ~static_cast<size_t>(15);
            const uint32_t bytes = g1 > g0 ? static_cast<uint32_t>(g1 - g0) : 0u;
            mbar_arrive_expect_tx(smem_u32(&scale_bar), bytes * R);
            if (bytes)
#pragma unroll
                for (int r = 0; r < R; ++r)
                    bulk_copy_g2s(smem_u32(swreg + r * sreg),
                                  reinterpret_cast<const uint8_t *>(a.scales[r]) + g0, bytes,
                                  smem_u32(&scale_bar));
        }
        bool ok = true;
        int issued = 0;
        for (int st = 0; st < nst && ok; ++st) {
            const int slot = st % S;
            if (st >= S) {
                if (lane == 0) ok = mbar_wait(smem_u32(&empty_bar[slot]), ((st / S) - 1) & 1);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            const int tile = st / spt, ks = st % spt;
            const int t0 = n_beg + tile * T;
            const uint32_t full = smem_u32(&full_bar[slot]);
            if (lane == 0) {
                // per matrix and box: a [rs bytes x box_rows] box; boxes that start
                // past the row's end are skipped; rows or bytes past the tensor's
                // end arrive as zeros and count toward the bytes
                const int nbox = min(kBoxesPerStage, (nb - ks * kBlocksPerStage + kBlocksPerBox - 1) / kBlocksPerBox);
                mbar_arrive_expect_tx(full, static_cast<uint32_t>(R * nbox * box_rows * rs));
#pragma unroll
                for (int r = 0; r < R; ++r)
                    for (int bx = 0; bx < nbox; ++bx)
                        tma_load_2d(smem_u32(ring + static_cast<size_t>(slot) * kStageBytes +
                                             (r * kBoxesPerStage + bx) * T * rs),
                                    &a.tmap[r], (ks * kBlocksPerStage + bx * kBlocksPerBox) * BB, t0, full);
            }
            __syncwarp();
            issued = st + 1;
        }
        if (lane == 0) {
            if (!ok && a.err != nullptr) atomicOr(a.err, 1u);
            // every issued copy lands before this thread exits
            for (int st = issued > S ? issued - S : 0; st < issued; ++st)
                if (!mbar_wait(smem_u32(&full_bar[st % S]), (st / S) & 1) && a.err != nullptr)
                    atomicOr(a.err, 2u);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    pdl_wait();
    {
        // scale elements the bulk copy could not cover (at the array's end)
        const size_t total = static_cast<size_t>(a.n) * nb * 2;
        const size_t g0 = sbyte0 - shead;
        const size_t covered_end = min((sbyte0 + static_cast<size_t>(outs) * nb * 2 + 15) & ~static_cast<size_t>(15),
                                       total & ~static_cast<size_t>(15));
        const size_t want_end = sbyte0 + static_cast<size_t>(outs) * nb * 2;
        if (covered_end < want_end) {
            const int first = static_cast<int>((covered_end - sbyte0) / 2);
            const int cnt = static_cast<int>((want_end - covered_end) / 2);
            for (int i = threadIdx.x; i < R * cnt; i += kConsumers) {
                const int r = i / cnt, e = first + i % cnt;
                reinterpret_cast<uint16_t *>(swreg + r * sreg + shead)[e] =
                    ldg_u16(a.scales[r] + static_cast<size_t>(n_beg) * nb + e);
            }
        }
        (void)g0;
    }
    stage_activation<FMT, M>(a.q, a.s, k, act, sact, cmag, kConsumers);
    if (!mbar_wait(smem_u32(&scale_bar), 0) && lane == 0 && a.err != nullptr) atomicOr(a.err, 8u);

    const int p = lane & (kLanesPerRow - 1);
    const int g = threadIdx.x >> 3;                  // output within a tile
    bool ok = true;
    int st = 0;
    for (int tile = 0; tile < tiles; ++tile) {
        const int o = tile * T + g;                  // output offset within the CTA
        const bool valid = o < outs;
        float acc[R][M];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int mm = 0; mm < M; ++mm) acc[r][mm] = 0.0f;
        for (int ks = 0; ks < spt; ++ks, ++st) {
            const int slot = st % S;
            if (ok && !mbar_wait(smem_u32(&full_bar[slot]), (st / S) & 1)) ok = false;
            // this lane's blocks of the stage: j = 2ks and 2ks + 1 of its chain
            const int b0 = ks * kBlocksPerStage + p;
            if (ok && valid && b0 < nb) {
                const uint8_t *stage = ring + static_cast<size_t>(slot) * kStageBytes;
                const __half *sw0 = reinterpret_cast<const __half *>(swreg + shead) + o * nb;
                const __half *sw1 = reinterpret_cast<const __half *>(swreg + sreg + shead) + o * nb;
                int32_t *dptr = (!GATEUP && a.dots != nullptr)
                                    ? a.dots + static_cast<size_t>(n_beg + o) * nb : nullptr;
                const size_t dstride = static_cast<size_t>(a.n) * nb;
                if (b0 + kBlocksPerBox < nb) {
                    if (dptr) stage_blocks<FMT, M, 2, R, true>(stage, T, rs, g, p, b0, act, sact, cmag, sw0, sw1, nb, acc, dptr, dstride);
                    else stage_blocks<FMT, M, 2, R, false>(stage, T, rs, g, p, b0, act, sact, cmag, sw0, sw1, nb, acc, dptr, dstride);
                } else {
                    if (dptr) stage_blocks<FMT, M, 1, R, true>(stage, T, rs, g, p, b0, act, sact, cmag, sw0, sw1, nb, acc, dptr, dstride);
                    else stage_blocks<FMT, M, 1, R, false>(stage, T, rs, g, p, b0, act, sact, cmag, sw0, sw1, nb, acc, dptr, dstride);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
        }
        if (!ok) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int mm = 0; mm < M; ++mm) acc[r][mm] = __int_as_float(0x7fc00000);   // NaN marks it
        }
        // fixed tree over the 8 partials: distance 1, 2, 4 (fp32 add commutes,
        // so both partners of each exchange hold the same sum)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int mm = 0; mm < M; ++mm) {
                float v = acc[r][mm];
                v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
                v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
                v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 4));
                acc[r][mm] = v;
            }
        if (valid && p == 0) {
            const size_t out = static_cast<size_t>(n_beg + o);
#pragma unroll
            for (int mm = 0; mm < M; ++mm) {
                if constexpr (!GATEUP) {
                    a.y[static_cast<size_t>(mm) * a.n + out] = acc[0][mm];
                } else {
                    const float hv = __fmul_rn(tq_silu(acc[0][mm]), acc[1][mm]);
                    a.h[static_cast<size_t>(mm) * a.n + out] = f32_to_bf16_bits(hv);
                }
            }
        }
    }
    if (!ok && lane == 0 && a.err != nullptr) atomicOr(a.err, 4u);

    if constexpr (GATEUP) {
        if (a.counters != nullptr) {
            // the last CTA to finish a 128-block of h rotates + quantises it;
            // this CTA's outputs touch at most two such blocks
            named_barrier(1, kConsumers);
            const int hb0 = n_beg / kBlock, hb1 = (n_end - 1) / kBlock;
            if (threadIdx.x == 0) {
                __threadfence();
                for (int j = 0; j < 2; ++j) {
                    const int hb = hb0 + j;
                    s_last[j] = 0;
                    if (hb > hb1) continue;
                    const int lo = max(n_beg, hb * kBlock), hi = min(n_end, (hb + 1) * kBlock);
                    const unsigned add = static_cast<unsigned>(hi - lo);
                    const unsigned before = atomicAdd(&a.counters[hb], add);
                    if (before + add == static_cast<unsigned>(kBlock)) {
                        a.counters[hb] = 0u;
                        s_last[j] = 1;
                    }
                }
                __threadfence();
            }
            named_barrier(1, kConsumers);
            for (int j = 0; j < 2; ++j) {
                if (!s_last[j]) continue;
                const int hb = hb0 + j;
                for (int mm = warp; mm < M; mm += NCW) {
                    const uint16_t *hrow = a.h + static_cast<size_t>(mm) * a.n + hb * kBlock;
                    float v[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) v[c] = bf16_bits_to_f32(__ldcg(hrow + lane + 32 * c));
                    rotq_block_store(v, lane, a.qh + static_cast<size_t>(mm) * a.n + hb * kBlock,
                                     a.sh + static_cast<size_t>(mm) * (a.n / kBlock) + hb);
                }
            }
        }
    }
}

}  // namespace tq
