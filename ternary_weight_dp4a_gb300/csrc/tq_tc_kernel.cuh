// tq_tc_kernel.cuh -- the tensor-core GEMV / FFN kernel: the ternary (or
// binary) weights are decoded by the CUDA cores into e4m3 and written to
// tensor memory, and the 5th-generation tensor core (tcgen05.mma
// kind::f8f6f4, M = 128, N = 16) forms the exact block dots against the int8
// activation split into two e4m3 parts.
//
// Exactness.  2-bit weights decode (prmt, as in tq_dp4a.cuh) to w + 1 in
// {0, 1, 2}; 1-bit weights to b * 2^-6 with b in {0, 1}.  An int8 code q is
// split as q = 16 hi + lo with hi in [-8, 8], lo in [-8, 7]; every one of
// these values is an e4m3 number, every product is exact, and every partial
// sum is an integer (a multiple of 2^-6 for 1-bit) far below 2^24 in
// magnitude, so the f32 accumulation in tensor memory is exact.  The block
// dot then follows exactly: 2-bit d = 16 D_hi + D_lo - sum(q); 1-bit
// d = 128 (16 D_hi + D_lo) - sum(q) (w = 2b - 1).  Activation row r of a pass
// occupies MMA columns 2r (hi) and 2r + 1 (lo).
//
// Work.  A unit is 128 weight rows (one MMA M) x one segment (8 consecutive
// 128-blocks) of one matrix: one or two 16 KB planes of codes (128 rows x
// 128 bytes: four 2-bit blocks or eight 1-bit blocks) and 2 KB of scales.
// Units are dealt to CTAs round-robin over a fixed order: phase A (gate, up)
// tile-major (tile, matrix, segment), then phase B (down or a plain GEMV)
// segment-major (segment, tile).  Every CTA streams its units through one
// pipeline:
//   producer warp   TMA of the code planes and scales into shared-memory rings
//   8 decoder warps prmt decode -> e4m3 -> tcgen05.st into TMEM A stages
//                   (128 lanes x 32 columns = one block each; two slots of a
//                   group of 4 blocks)
//   MMA thread      per group, 4 x tcgen05.mma (K = 32 each) per block into
//                   the block's own TMEM accumulator (32 columns apart),
//                   interleaved across the group's blocks, then two commits
//   4 epilogue warps tcgen05.ld of a group's accumulators (one wait), the
//                   exact block dot, t_b = d * (sw * sa), the segment sums in
//                   ascending block order -> global partials
//   counter warp    counts each finished unit for its tile in global memory;
//                   the count that completes a tile queues its fold here
//   4 fold warps    pairwise tree over a tile's segment sums from every CTA;
//                   phase A: h = bf16(silu(g) u), and with rotate_h the
//                   128-point rotation + quantisation of that block of h,
//                   written in the layout phase B's MMA reads and released
//                   per 8-block segment; phase B: y
//   stager warp     phase B: waits until a segment of its input is ready and
//                   bulk-copies it into a shared-memory slot.
// A step (phase A and B in one launch) needs every CTA resident (phase B
// waits for blocks of h other CTAs fold): one CTA per SM, cooperative launch.
//
// Every wait is bounded; one that runs out sets a bit in the error word and a
// CTA-wide abort flag, and the CTA winds down without hanging.
#pragma once

#include <cuda.h>

#include "tq_stage.cuh"
#include "tq_tcgen05.cuh"

namespace tq {
namespace tc {

constexpr int kTile = 128;                    // weight rows per unit (MMA M)
constexpr int kSeg = kSegBlocks;              // 128-blocks per segment
constexpr int kPlane = 16384;                 // ring slot: 128 rows x 128 bytes of codes
constexpr int kScBytes = kTile * kSeg * 2;    // scales of one unit (fp16 [128][8])
constexpr int kN = 16;                        // MMA N: hi / lo columns of up to 8 rows

// warp roles
constexpr int kWProducer = 0, kWMma = 1, kWStager = 2, kWAlloc = 3;
constexpr int kWDec0 = 4, kNumDec = 8;
constexpr int kWEpi0 = 12, kNumEpi = 4;
constexpr int kWFold0 = 16, kNumFold = 4;
constexpr int kWarps = 20;
constexpr int kThreads = 32 * kWarps;
constexpr int kPrologueThreads = 32 * (kNumDec + kNumEpi + kNumFold);   // decoder, epilogue and fold warps

// named barriers (0 is __syncthreads)
constexpr int kBarPrologue = 1, kBarEpi = 2, kBarFold = 3;

// tensor memory: A stages [0, 256), accumulators [256, 512)
constexpr int kAStages = 8, kDStages = 8;
constexpr int kEpiGroup = 4;                  // blocks per group (one MMA batch, one epilogue read)
constexpr int kGroupSlots = kAStages / kEpiGroup;   // groups in flight (A stages and accumulators)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol0 = 0, kDCol0 = 32 * kAStages;

constexpr int kMaxRing = 16, kMaxSc = 8, kMaxB = 4;
constexpr int kQueue = 64;                    // fold jobs per CTA per launch (host-checked: units + 1)
constexpr int kMaxSegs = 32;                  // segments per output of a fold (k <= 32768)
constexpr int kMaxSegsA = 8;                  // phase A (gate / up): hidden <= 8192
constexpr int kJobEnd = -1, kJobEmpty = -2;

// Bytes of one 128-block of the B operand (activation rows, hi / lo) in
// shared memory, its K-direction core-matrix stride (LBO) and 8-row-group
// stride (SBO).  Up to 4 rows use 8 B rows (1 KB per block); the MMA still
// reads N = 16 rows, the upper 8 from the next core matrices (their
// accumulator columns are never read).  5..8 rows use 16 B rows.
template <int M> constexpr int kBBlk = M <= 4 ? 1024 : 2048;
template <int M> constexpr uint32_t kLbo = M <= 4 ? 128u : 256u;
constexpr uint32_t kSbo = 128u;

// Byte offset of (B row n, staged position p) inside a block.
template <int M>
__device__ __forceinline__ int b_off(int n, int p) {
    return M <= 4 ? (p >> 4) * 128 + n * 16 + (p & 15)
                  : (p >> 4) * 256 + (n >> 3) * 128 + (n & 7) * 16 + (p & 15);
}

struct TcMat {
    CUtensorMap tm_codes;     // uint8 {row bytes, n}, box {128, 128}, 128-byte swizzle
    CUtensorMap tm_scales;    // uint16 {nb, n}, box {8, 128} (valid when scales_tma)
    const uint16_t *scales;
    int n, k, nb, nseg, ntiles, scales_tma;
};

enum : int { kInRotX = 0, kInNormY = 1, kInPlain = 2 };

struct TcArgs {
    TcMat mat[3];             // phase A: gate, up; phase B: mat[2]
    int do_a, do_b, m;        // m: rows of this pass (<= M)
    int ua, ub;               // units of phase A and of phase B
    int ring, sc_slots, b_slots;
    // dynamic shared memory: ring | scales ring | phase A operand | its
    // (scale, sum q) pairs | phase B slots | their pairs | fold scratch
    uint32_t off_sc, off_ba, off_bap, off_bb, off_bbp, off_fold;
    // phase A input
    int in_mode;
    const uint16_t *x;        // bf16 [m][hidden]                    (kInRotX)
    const float *y_in;        // fp32 [m][hidden]                    (kInNormY)
    float eps;
    const int8_t *qa;         // int8 [m][hidden], fp32 [m][hidden/128] (kInPlain)
    const float *sa;
    int8_t *qx;               // CTA 0 writes the quantised input here (may be null)
    float *sx;
    // phase A output
    uint16_t *h;              // bf16 [m][inter]
    int rotate_h;
    int8_t *qh;               // [m][inter], [m][inter/128]
    float *sh;
    uint8_t *hst;             // h as phase B's operand: [inter/128] blocks of kBBlk bytes
    float2 *hsn;              // [inter/128][M] (scale, sum q)
    // phase B input (operand blocks + pairs, laid out as hst / hsn) and output
    const uint8_t *bst;
    const float2 *bsn;
    float *y;                 // fp32 [m][n]
    int32_t *dots;            // int32 [m][n][nb] or null
    // workspace: segment sums of every unit, per-tile unit counts (zero
    // between launches), per-segment ready counts of h and the launch ticket
    float *part_a, *part_b;
    unsigned *cnt_a, *cnt_b;
    unsigned *segready;
    unsigned long long *ticket;
    unsigned *err;            // bit 0 producer (slot free), 1 producer drain, 2 decoder (codes),
                              // 3 MMA (operands), 5 epilogue (accumulator / scales),
                              // 6 stager (segment of h), 7 fold queue, 8 stager drain
};

struct Unit {
    int phase, mi, tile, seg, bcount;
};

__device__ __forceinline__ Unit unit_of(const TcArgs &a, int u) {
    Unit r;
    if (u < a.ua) {
        const TcMat &g = a.mat[0];
        const int per_tile = 2 * g.nseg;
        r.phase = 0;
        r.tile = u / per_tile;
        const int rem = u - r.tile * per_tile;
        r.mi = rem / g.nseg;
        r.seg = rem - r.mi * g.nseg;
        r.bcount = min(kSeg, g.nb - r.seg * kSeg);
    } else {
        const TcMat &d = a.mat[2];
        const int v = u - a.ua;
        r.phase = 1;
        r.mi = 2;
        r.seg = v / d.ntiles;
        r.tile = v - r.seg * d.ntiles;
        r.bcount = min(kSeg, d.nb - r.seg * kSeg);
    }
    return r;
}

// e4m3 bits of a small integer (|v| <= 16): from the binary32 pattern of |v|
// (exponent rebased from 127 to 7, top three fraction bits kept).
__device__ __forceinline__ uint32_t e4m3_int(int v) {
    if (v == 0) return 0u;
    const uint32_t f = __float_as_uint(static_cast<float>(v < 0 ? -v : v));
    return (v < 0 ? 0x80u : 0u) | (((f >> 20) - 960u) & 0x7fu);
}

// q = 16 hi + lo, hi in [-8, 8], lo in [-8, 7]; four codes -> the e4m3 words
// of their hi and lo parts (byte j from code j).
__device__ __forceinline__ void hilo_words(const int (&q)[4], uint32_t &whi, uint32_t &wlo) {
    whi = 0u;
    wlo = 0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int hi = (q[j] + 8) >> 4;
        const int lo = q[j] - 16 * hi;
        whi |= e4m3_int(hi) << (8 * j);
        wlo |= e4m3_int(lo) << (8 * j);
    }
}

// ---------------------------------------------------------------------------
// Bounded waits.  A wait gives up after ~0.5 s of clock cycles (or at once
// when another role of the CTA has given up): it records its error bit in
// *bad and raises the CTA's abort flag.  Waits that only follow other waits
// (the counter's and the fold warps' waits for finished work) get twice the
// budget, so the wait that names the cause runs out first.
// ---------------------------------------------------------------------------
constexpr long long kFollowerBudgetCycles = 2 * kWaitBudgetCycles;

__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned bit,
                                        unsigned &bad, long long budget = kWaitBudgetCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > budget) {
            bad |= bit;
            *abort_flag = 1;
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// Phase A's operand: every CTA stages the input rows, rotated (or plain) and
// quantised, as hi / lo e4m3 rows of the B operand, in staged order, with
// one (scale, sum q) pair per block and row.  Run by the decoder, epilogue
// and fold warps (pw = 0..15 of them) before their own work; rows m..M-1 are
// zero.
// ---------------------------------------------------------------------------
template <int FMT, int M>
__device__ __forceinline__ void store_b_words(uint8_t *blk, float2 *pairs, int b, int r, int lane, const int (&q)[4],
                                              float sc, int sum) {
    uint32_t whi, wlo;
    hilo_words(q, whi, wlo);
    const int p = 4 * lane;
    *reinterpret_cast<uint32_t *>(blk + b_off<M>(2 * r, p)) = whi;
    *reinterpret_cast<uint32_t *>(blk + b_off<M>(2 * r + 1, p)) = wlo;
    if (lane == 0) pairs[b * M + r] = make_float2(sc, static_cast<float>(sum));
}

template <int FMT, int M, typename LoadFn>
__device__ __forceinline__ void stage_rotated_tc(const TcArgs &a, LoadFn load, int k, uint8_t *ba, float2 *bap,
                                                 int pw, int lane, bool write_plain, int r_only) {
    const int nb = k / kBlock;
    const int rows = r_only >= 0 ? 1 : M;
    constexpr int kGroup = 4;                 // blocks a warp has in flight (their loads overlap)
    constexpr int kPW = kPrologueThreads / 32;
    for (int blk0 = pw; blk0 < rows * nb; blk0 += kGroup * kPW) {
        float v[kGroup][4];
        int rr[kGroup], bb[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int blk = blk0 + u * kPW;
            rr[u] = r_only >= 0 ? r_only : blk / nb;
            bb[u] = r_only >= 0 ? blk : blk - rr[u] * nb;
            if (blk < rows * nb && rr[u] < a.m) load(rr[u], bb[u], v[u]);
            else v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0.0f;
        }
        int8_t q8[kGroup][4];
        uint32_t word[kGroup];
        int sum[kGroup];
        float sc[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) sc[u] = rotq_staged<FMT>(v[u], lane, q8[u], word[u], sum[u]);
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int blk = blk0 + u * kPW;
            if (blk >= rows * nb) break;
            const int r = rr[u], b = bb[u];
            const int q[4] = {q8[u][0], q8[u][1], q8[u][2], q8[u][3]};
            store_b_words<FMT, M>(ba + static_cast<size_t>(b) * kBBlk<M>, bap, b, r, lane, q, sc[u], sum[u]);
            if (write_plain && r < a.m) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    a.qx[static_cast<size_t>(r) * k + b * kBlock + staged_elem<FMT>(4 * lane + c)] = q8[u][c];
                if (lane == 0) a.sx[static_cast<size_t>(r) * nb + b] = sc[u];
            }
        }
    }
}

// Plain int8 input (already quantised, natural order) -> staged hi / lo rows.
template <int FMT, int M>
__device__ __forceinline__ void stage_plain_tc(const TcArgs &a, int k, uint8_t *ba, float2 *bap, int pw, int lane) {
    const int nb = k / kBlock;
    constexpr int kPW = kPrologueThreads / 32;
    for (int blk = pw; blk < M * nb; blk += kPW) {
        const int r = blk / nb, b = blk - r * nb;
        int q[4] = {0, 0, 0, 0};
        float sc = 0.0f;
        if (r < a.m) {
            const int8_t *src = a.qa + static_cast<size_t>(r) * k + b * kBlock;
#pragma unroll
            for (int c = 0; c < 4; ++c) q[c] = __ldcg(reinterpret_cast<const signed char *>(src) + staged_elem<FMT>(4 * lane + c));
            sc = __ldcg(a.sa + static_cast<size_t>(r) * nb + b);
        }
        const int sum = __reduce_add_sync(0xffffffffu, q[0] + q[1] + q[2] + q[3]);
        store_b_words<FMT, M>(ba + static_cast<size_t>(b) * kBBlk<M>, bap, b, r, lane, q, sc, sum);
    }
}

// ---------------------------------------------------------------------------
// Decode one block row of codes (this thread's weight row) from the ring's
// swizzled plane into 32 e4m3 words in staged order.
// ---------------------------------------------------------------------------
template <int FMT>
__device__ __forceinline__ void decode_block(const uint8_t *plane, int row, int bl, uint32_t (&w)[32]) {
    if constexpr (FMT == 0) {
        // block bl (0..3 within the plane) is 32 bytes: 16-byte chunks 2 bl, 2 bl + 1
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = (2 * bl + h) ^ (row & 7);
            const uint4 cw = *reinterpret_cast<const uint4 *>(plane + row * 128 + c * 16);
            const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // w + 1 in {0, 1, 2} as e4m3 {0, 1.0, 2.0}: pool {2.0 x4 : 1.0 x4}
                const uint32_t wd = words[i];
                const int o = 16 * h + 4 * i;
                w[o + 0] = prmt(0x38383838u, 0x40404040u, wd << 2);
                w[o + 1] = prmt(0x38383838u, 0x40404040u, wd >> 14);
                w[o + 2] = prmt(0x38383838u, 0x40404040u, wd);
                w[o + 3] = prmt(0x38383838u, 0x40404040u, wd >> 16);
            }
        }
    } else {
        // block bl (0..7) is one 16-byte chunk; bit s of byte j of word i is
        // weight 32 i + 8 j + s; register 8 i + s holds weights 32 i + 8 j + s
        // (j = 0..3) as e4m3 2^-6 (bit set) or 0, at bit 3 of each byte
        const int c = bl ^ (row & 7);
        const uint4 cw = *reinterpret_cast<const uint4 *>(plane + row * 128 + c * 16);
        const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t wd = words[i];
            w[8 * i + 0] = (wd << 3) & 0x08080808u;
            w[8 * i + 1] = (wd << 2) & 0x08080808u;
            w[8 * i + 2] = (wd << 1) & 0x08080808u;
            w[8 * i + 3] = wd & 0x08080808u;
            w[8 * i + 4] = (wd >> 1) & 0x08080808u;
            w[8 * i + 5] = (wd >> 2) & 0x08080808u;
            w[8 * i + 6] = (wd >> 3) & 0x08080808u;
            w[8 * i + 7] = (wd >> 4) & 0x08080808u;
        }
    }
}

// Pairwise tree over n values V[0..n) (n <= N): each level adds (0,1),
// (2,3), ... and passes an odd last node up.  Written as in-place levels over
// the fixed array (node i of the next level from nodes 2i, 2i + 1, ascending,
// so no node is overwritten before it is read) with every index static, so V
// stays in registers; the combination order is that of the tree.
template <int N>
__device__ __forceinline__ float fold_tree_fixed(float (&V)[N], int n) {
#pragma unroll
    for (int level = 0; (1 << level) < N; ++level) {
        if (n > 1) {
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                if (2 * i + 1 < n) V[i] = __fadd_rn(V[2 * i], V[2 * i + 1]);
                else if (2 * i < n) V[i] = V[2 * i];
            }
            n = (n + 1) >> 1;
        }
    }
    return V[0];
}

// Load the segment sums of one output (n <= N of them, stride floats apart)
// with every load in flight together.
template <int N>
__device__ __forceinline__ void load_segs(float (&V)[N], const float *p, int n, size_t stride) {
#pragma unroll
    for (int i = 0; i < N; ++i) V[i] = i < n ? __ldcg(p + static_cast<size_t>(i) * stride) : 0.0f;
}

template <int FMT, int M>
__global__ void __launch_bounds__(kThreads, 1) tc_kernel(const __grid_constant__ TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t ring_full[kMaxRing], ring_empty[kMaxRing];
    __shared__ __align__(8) uint64_t sc_full[kMaxSc], sc_empty[kMaxSc];
    // per group slot (kEpiGroup consecutive blocks of a unit): A stages
    // written by every decoder warp / released by the MMA commit; accumulators
    // committed by the MMA / released by the four epilogue warps
    __shared__ __align__(8) uint64_t a_full[kGroupSlots], a_empty[kGroupSlots];
    __shared__ __align__(8) uint64_t d_full[kGroupSlots], d_empty[kGroupSlots];
    __shared__ __align__(8) uint64_t b_full[kMaxB], b_empty[kMaxB];
    __shared__ __align__(8) uint64_t ba_ready, mma_done;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ __align__(8) uint64_t unit_done[kQueue];   // per unit: the 4 epilogue warps stored its sums
    __shared__ int s_jobs[kQueue];
    __shared__ int s_job;
    __shared__ float s_warp[8];
    __shared__ float s_red[kNumFold][M];
    __shared__ int s_redi[kNumFold][M];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *ring = base;
    uint8_t *scring = base + a.off_sc;
    uint8_t *ba = base + a.off_ba;
    float2 *bap = reinterpret_cast<float2 *>(base + a.off_bap);
    uint8_t *bb = base + a.off_bb;
    float2 *bbp = reinterpret_cast<float2 *>(base + a.off_bbp);
    float *fold_x = reinterpret_cast<float *>(base + a.off_fold);                 // [M][128]
    uint8_t *fold_b = base + a.off_fold + M * kTile * 4;                           // one operand block
    volatile int *abort_flag = &s_abort;
    const int total = a.ua + a.ub;
    const int nunits = cta < total ? (total - 1 - cta) / G + 1 : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.ring; ++i) {
            mbar_init(smem_u32(&ring_full[i]), 1);
            mbar_init(smem_u32(&ring_empty[i]), kNumDec);
        }
        for (int i = 0; i < a.sc_slots; ++i) {
            mbar_init(smem_u32(&sc_full[i]), 1);
            mbar_init(smem_u32(&sc_empty[i]), kNumEpi);
        }
        for (int i = 0; i < kGroupSlots; ++i) {
            mbar_init(smem_u32(&a_full[i]), kNumDec);
            mbar_init(smem_u32(&a_empty[i]), 1);
            mbar_init(smem_u32(&d_full[i]), 1);
            mbar_init(smem_u32(&d_empty[i]), kNumEpi);
        }
        for (int i = 0; i < a.b_slots; ++i) {
            mbar_init(smem_u32(&b_full[i]), 1);
            mbar_init(smem_u32(&b_empty[i]), 1 + kNumEpi);
        }
        mbar_init(smem_u32(&ba_ready), 1);
        mbar_init(smem_u32(&mma_done), 1);
        for (int i = 0; i < kQueue; ++i) mbar_init(smem_u32(&unit_done[i]), kNumEpi);
        mbar_init_fence();
        s_abort = 0;
    }
    for (int i = threadIdx.x; i < kQueue; i += kThreads) s_jobs[i] = kJobEmpty;
    if (warp == kWAlloc) {
        tmem_alloc(smem_u32(&s_tmem), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s_tmem;
    pdl_launch_dependents();
    unsigned bad = 0u;

    if (warp >= kWDec0) {
        // ---- phase A's operand, by the decoder, epilogue and fold warps
        const int pw = warp - kWDec0;                 // 0..15
        pdl_wait();
        if (a.do_a && a.ua > 0) {
            const TcMat &gm = a.mat[0];
            const int hidden = gm.k;
            const bool plain_out = cta == 0 && a.qx != nullptr;
            if (a.in_mode == kInRotX) {
                const uint16_t *x = a.x;
                stage_rotated_tc<FMT, M>(a, [&](int r, int b, float (&v)[4]) {
                    load_staged_bf16<FMT>(x + static_cast<size_t>(r) * hidden + b * kBlock, lane, v, false);
                }, hidden, ba, bap, pw, lane, plain_out, -1);
            } else if (a.in_mode == kInNormY) {
                const int t = pw * 32 + lane;
                for (int r = 0; r < M; ++r) {
                    if (r >= a.m) {
                        stage_rotated_tc<FMT, M>(a, [&](int, int, float (&v)[4]) { v[0] = v[1] = v[2] = v[3] = 0.0f; },
                                                 hidden, ba, bap, pw, lane, false, r);
                        continue;
                    }
                    // 1/rms: 256 partial sums (thread t adds y[t], y[t+256], ...),
                    // each warp's 32 combined at distance 1, 2, ..., 16, then
                    // ((w0+w1)+(w2+w3)) + ((w4+w5)+(w6+w7))
                    const float *yr = a.y_in + static_cast<size_t>(r) * hidden;
                    // (the first 8 warps of the group hold the 256 partials)
                    float acc = 0.0f;
                    if (t < 256)
                        for (int i = t; i < hidden; i += 256) {
                            const float v = __ldcg(yr + i);
                            acc = __fadd_rn(acc, __fmul_rn(v, v));
                        }
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
                    if (lane == 0 && pw < 8) s_warp[pw] = acc;
                    named_barrier(kBarPrologue, kPrologueThreads);
                    const float w01 = __fadd_rn(s_warp[0], s_warp[1]), w23 = __fadd_rn(s_warp[2], s_warp[3]);
                    const float w45 = __fadd_rn(s_warp[4], s_warp[5]), w67 = __fadd_rn(s_warp[6], s_warp[7]);
                    const float ss = __fadd_rn(__fadd_rn(w01, w23), __fadd_rn(w45, w67));
                    const float inv =
                        __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(hidden)), a.eps)));
                    named_barrier(kBarPrologue, kPrologueThreads);
                    stage_rotated_tc<FMT, M>(a, [&](int, int b, float (&v)[4]) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            v[c] = bf16_bits_to_f32(f32_to_bf16_bits(
                                __fmul_rn(__ldcg(yr + b * kBlock + staged_elem<FMT>(4 * lane + c)), inv)));
                    }, hidden, ba, bap, pw, lane, plain_out, r);
                }
            } else {
                stage_plain_tc<FMT, M>(a, hidden, ba, bap, pw, lane);
            }
            fence_proxy_async_smem();
            named_barrier(kBarPrologue, kPrologueThreads);
            if (pw == 0 && lane == 0) mbar_arrive(smem_u32(&ba_ready));
        }

    }

    if (warp == kWProducer) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int slot = 0, sround = 0;         // ring position of the next plane
            int issued_planes = 0, ks = 0;     // planes issued, scales-ring uses
            bool ok = true;
            for (int k = 0; k < nunits && ok; ++k) {
                const Unit U = unit_of(a, cta + k * G);
                const TcMat &md = a.mat[U.mi];
                const int planes = FMT == 0 ? (U.bcount > 4 ? 2 : 1) : 1;
                for (int p = 0; p < planes && ok; ++p) {
                    if (sround > 0 && !(ok = tc_wait(smem_u32(&ring_empty[slot]), (sround - 1) & 1, abort_flag, 1u, bad)))
                        break;
                    const uint32_t fb = smem_u32(&ring_full[slot]);
                    mbar_arrive_expect_tx(fb, kPlane);
                    const int x0 = FMT == 0 ? U.seg * 256 + p * 128 : U.seg * 128;
                    tma_load_2d(smem_u32(ring + static_cast<size_t>(slot) * kPlane), &md.tm_codes, x0, U.tile * kTile,
                                fb, pol);
                    ++issued_planes;
                    if (++slot == a.ring) {
                        slot = 0;
                        ++sround;
                    }
                }
                if (ok && md.scales_tma) {
                    const int ss = ks % a.sc_slots, sr = ks / a.sc_slots;
                    ++ks;
                    if (sr > 0 && !(ok = tc_wait(smem_u32(&sc_empty[ss]), (sr - 1) & 1, abort_flag, 1u, bad))) break;
                    const uint32_t fb = smem_u32(&sc_full[ss]);
                    mbar_arrive_expect_tx(fb, kScBytes);
                    tma_load_2d(smem_u32(scring + static_cast<size_t>(ss) * kScBytes), &md.tm_scales, U.seg * kSeg,
                                U.tile * kTile, fb, pol);
                }
            }
            // nothing may still be landing in shared memory at exit: wait for
            // the last fill of every slot (after a normal run each has been
            // consumed and the check returns at once)
            for (int sl = 0; sl < a.ring && sl < issued_planes; ++sl) {
                const int last = sl + a.ring * ((issued_planes - 1 - sl) / a.ring);
                if (!mbar_wait(smem_u32(&ring_full[sl]), (last / a.ring) & 1)) {
                    bad |= 2u;
                    break;
                }
            }
            for (int i = max(0, ks - a.sc_slots); i < ks; ++i)
                if (!mbar_wait(smem_u32(&sc_full[i % a.sc_slots]), (i / a.sc_slots) & 1)) {
                    bad |= 2u;
                    break;
                }
        }
        __syncwarp();
    } else if (warp == kWMma) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3(kTile, kN);
            bool ok = true;
            if (a.do_a && a.ua > 0) ok = tc_wait(smem_u32(&ba_ready), 0, abort_flag, 8u, bad);
            int G = 0, kb = 0;                     // groups issued, phase-B units
            for (int k = 0; k < nunits && ok; ++k) {
                const Unit U = unit_of(a, cta + k * gridDim.x);
                const uint8_t *bsrc;
                int bs = 0;
                if (U.phase == 0) {
                    bsrc = ba + static_cast<size_t>(U.seg) * kSeg * kBBlk<M>;
                } else {
                    bs = kb % a.b_slots;
                    if (!(ok = tc_wait(smem_u32(&b_full[bs]), (kb / a.b_slots) & 1, abort_flag, 8u, bad))) break;
                    bsrc = bb + static_cast<size_t>(bs) * kSeg * kBBlk<M>;
                }
                // the unit's blocks in groups of up to kEpiGroup (group G uses
                // slot G mod kGroupSlots: A stages and accumulators kEpiGroup x
                // slot ..): the group's accumulators are independent, so its
                // MMAs go out interleaved (K step 0 of each block, then K step
                // 1, ...), followed by one commit per barrier
                for (int b0 = 0; b0 < U.bcount && ok; b0 += kEpiGroup, ++G) {
                    const int nb_g = min(kEpiGroup, U.bcount - b0);
                    const int gs = G % kGroupSlots, gr = G / kGroupSlots;
                    if (!(ok = tc_wait(smem_u32(&a_full[gs]), gr & 1, abort_flag, 8u, bad))) break;
                    if (gr > 0 && !(ok = tc_wait(smem_u32(&d_empty[gs]), (gr - 1) & 1, abort_flag, 8u, bad))) break;
                    tc_fence_after();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
#pragma unroll
                        for (int j = 0; j < kEpiGroup; ++j) {
                            if (j >= nb_g) break;
                            const uint32_t stage = static_cast<uint32_t>(gs * kEpiGroup + j);
                            const uint32_t baddr = smem_u32(bsrc + static_cast<size_t>(b0 + j) * kBBlk<M>);
                            tc_mma_e4m3_ts(tbase + kDCol0 + 32u * stage, tbase + kACol0 + 32u * stage + 8u * i,
                                           smem_desc_kmajor(baddr + 2u * i * kLbo<M>, kLbo<M>, kSbo), idesc, i > 0);
                        }
                    }
                    tc_commit(smem_u32(&a_empty[gs]));
                    tc_commit(smem_u32(&d_full[gs]));
                }
                if (U.phase == 1) {
                    tc_commit(smem_u32(&b_empty[bs]));
                    ++kb;
                }
            }
            // every MMA this thread issued has completed before TMEM is freed
            tc_commit(smem_u32(&mma_done));
            if (!mbar_wait(smem_u32(&mma_done), 0)) bad |= 8u;
        }
        __syncwarp();
    } else if (warp == kWStager) {
        // ------------------------------------------------------------ phase B input
        if (lane == 0 && a.ub > 0) {
            pdl_wait();
            const bool ticketed = a.do_a && a.rotate_h;
            unsigned epoch = 0;
            if (ticketed) epoch = static_cast<unsigned>(atomicAdd(a.ticket, 1ull) / static_cast<unsigned long long>(G));
            int kb = 0;
            bool ok = true;
            for (int k = 0; k < nunits && ok; ++k) {
                const Unit U = unit_of(a, cta + k * G);
                if (U.phase != 1) continue;
                const int bs = kb % a.b_slots, br = kb / a.b_slots;
                if (br > 0 && !(ok = tc_wait(smem_u32(&b_empty[bs]), (br - 1) & 1, abort_flag, 64u, bad))) break;
                if (ticketed) {
                    // the segment's blocks of h have been folded and rotated
                    // (by whichever CTAs completed them) in this launch
                    const unsigned target = (epoch + 1u) * static_cast<unsigned>(U.bcount);
                    const long long t0 = clock64();
                    while (static_cast<int>(ld_acquire_u32(a.segready + U.seg) - target) < 0) {
                        if (*abort_flag || clock64() - t0 > kWaitBudgetCycles) {
                            if (!*abort_flag) bad |= 64u;
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    if (!ok) break;
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                const uint32_t fb = smem_u32(&b_full[bs]);
                const uint32_t nbytes = static_cast<uint32_t>(U.bcount) * kBBlk<M>;
                const uint32_t pbytes = static_cast<uint32_t>(kSeg) * M * 8u;   // whole segment (16-byte multiple)
                mbar_arrive_expect_tx(fb, nbytes + pbytes);
                bulk_copy_g2s(smem_u32(bb + static_cast<size_t>(bs) * kSeg * kBBlk<M>),
                              a.bst + static_cast<size_t>(U.seg) * kSeg * kBBlk<M>, nbytes, fb);
                bulk_copy_g2s(smem_u32(bbp + static_cast<size_t>(bs) * kSeg * M),
                              a.bsn + static_cast<size_t>(U.seg) * kSeg * M, pbytes, fb);
                ++kb;
            }
            // the last fills of the slots have landed before exit
            for (int i = max(0, kb - a.b_slots); i < kb; ++i)
                if (!mbar_wait(smem_u32(&b_full[i % a.b_slots]), (i / a.b_slots) & 1)) {
                    bad |= 256u;
                    break;
                }
        }
        __syncwarp();
    } else if (warp == kWAlloc) {
        // ------------------------------------------------------------ counter
        // (the warp that allocated tensor memory; it frees it at the end).
        // Lane 0 takes the units in order as the epilogue finishes them and
        // counts each for its tile in global memory; the count that completes
        // a tile (every CTA's units of it have stored their segment sums)
        // queues the tile's fold for this CTA's fold warps.
        if (lane == 0) {
            pdl_wait();
            int nj = 0;
            for (int k = 0; k < nunits; ++k) {
                if (!tc_wait(smem_u32(&unit_done[k]), 0, abort_flag, 128u, bad, kFollowerBudgetCycles)) break;
                const Unit U = unit_of(a, cta + k * G);
                const TcMat &md = a.mat[U.mi];
                unsigned *cnt = U.phase == 0 ? a.cnt_a + U.tile : a.cnt_b + U.tile;
                const unsigned need = U.phase == 0 ? 2u * md.nseg : static_cast<unsigned>(md.nseg);
                // acquire-release at gpu scope: releases the sums this CTA's
                // epilogue stored (ordered before through the unit barrier),
                // acquires those of the CTAs that counted before
                const unsigned old = atom_add_acq_rel_gpu(cnt, 1u);
                if (old + 1u == need) {
                    *cnt = 0u;                                   // every unit of the tile has counted
                    __threadfence();
                    reinterpret_cast<volatile int *>(s_jobs)[nj++] = U.phase == 0 ? U.tile : (0x10000 | U.tile);
                }
            }
            __threadfence();
            reinterpret_cast<volatile int *>(s_jobs)[nj] = kJobEnd;
        }
        __syncwarp();
    } else if (warp >= kWDec0 && warp < kWDec0 + kNumDec) {
        // ------------------------------------------------------------ decoders
        const int q4 = warp & 3, grp = (warp - kWDec0) >> 2;
        const int row = 32 * q4 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        int slot = 0, sround = 0, Gi = 0;
        bool ok = true;
        for (int k = 0; k < nunits && ok; ++k) {
            const Unit U = unit_of(a, cta + k * G);
            // groups of kEpiGroup blocks; a 2-bit plane is one group, a 1-bit
            // plane the whole unit.  Decoder group grp takes blocks grp and
            // grp + 2 of each group; every decoder warp arrives once per group.
            for (int b0 = 0; b0 < U.bcount && ok; b0 += kEpiGroup, ++Gi) {
                if ((FMT == 0 || b0 == 0) &&
                    !(ok = __all_sync(0xffffffffu, tc_wait(smem_u32(&ring_full[slot]), sround & 1, abort_flag, 4u, bad))))
                    break;
                const uint8_t *plane = ring + static_cast<size_t>(slot) * kPlane;
                const int gs = Gi % kGroupSlots, gr = Gi / kGroupSlots;
                if (gr > 0 &&
                    !(ok = __all_sync(0xffffffffu, tc_wait(smem_u32(&a_empty[gs]), (gr - 1) & 1, abort_flag, 4u, bad))))
                    break;
                tc_fence_after();
                const int nb_g = min(kEpiGroup, U.bcount - b0);
                for (int j = grp; j < nb_g; j += 2) {
                    uint32_t w[32];
                    decode_block<FMT>(plane, row, FMT == 0 ? j : b0 + j, w);
                    tmem_st_x32(tbase + lane_base + kACol0 + 32u * static_cast<uint32_t>(gs * kEpiGroup + j), w);
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&a_full[gs]));
                // this warp's reads of the plane are done after its last group
                if (FMT == 0 || b0 + kEpiGroup >= U.bcount) {
                    if (lane == 0) mbar_arrive(smem_u32(&ring_empty[slot]));
                    if (++slot == a.ring) {
                        slot = 0;
                        ++sround;
                    }
                }
            }
        }
    } else {
        // ---------------------------------------------- epilogue + fold warps
        pdl_wait();
        if (warp < kWFold0) {
            // -------------------------------------------------------- epilogue
            const int q4 = warp & 3;
            const int row = 32 * q4 + lane;
            const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
            int Ge = 0, kb = 0, ks = 0;            // groups read, phase-B units, scales-ring uses
            bool ok = true;
            for (int k = 0; k < nunits && ok; ++k) {
                const Unit U = unit_of(a, cta + k * G);
                const TcMat &md = a.mat[U.mi];
                const int grow = U.tile * kTile + row;
                // this row's weight scales for the unit's blocks
                uint32_t wsr[4] = {0u, 0u, 0u, 0u};
                if (md.scales_tma) {
                    const int ss = ks % a.sc_slots;
                    if (!(ok = __all_sync(0xffffffffu, tc_wait(smem_u32(&sc_full[ss]), (ks / a.sc_slots) & 1, abort_flag, 32u, bad))))
                        break;
                    ++ks;
                    const uint4 s4 = *reinterpret_cast<const uint4 *>(scring + static_cast<size_t>(ss) * kScBytes + row * 16);
                    wsr[0] = s4.x; wsr[1] = s4.y; wsr[2] = s4.z; wsr[3] = s4.w;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sc_empty[ss]));
                } else if (grow < md.n) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int b0 = U.seg * kSeg + 2 * i;
                        const uint32_t lo = 2 * i < U.bcount ? ldg_u16(md.scales + static_cast<size_t>(grow) * md.nb + b0) : 0u;
                        const uint32_t hi = 2 * i + 1 < U.bcount ? ldg_u16(md.scales + static_cast<size_t>(grow) * md.nb + b0 + 1) : 0u;
                        wsr[i] = lo | (hi << 16);
                    }
                }
                const float2 *pairs;
                int bs = 0;
                if (U.phase == 0) {
                    pairs = bap + static_cast<size_t>(U.seg) * kSeg * M;
                } else {
                    bs = kb % a.b_slots;
                    if (!(ok = __all_sync(0xffffffffu, tc_wait(smem_u32(&b_full[bs]), (kb / a.b_slots) & 1, abort_flag, 32u, bad))))
                        break;
                    pairs = bbp + static_cast<size_t>(bs) * kSeg * M;
                }
                float acc[M];
#pragma unroll
                for (int r = 0; r < M; ++r) acc[r] = 0.0f;
                int32_t *dots = U.phase == 1 ? a.dots : nullptr;
                // the unit's blocks in groups of kEpiGroup (group G in slot G mod
                // kGroupSlots): one wait per group, the accumulators read kLd
                // blocks at a time with one wait for the loads, every index
                // static (the loops are unrolled with guards, so nothing moves
                // to local memory)
                constexpr int kLd = M <= 4 ? kEpiGroup : 2;
#pragma unroll
                for (int gi = 0; gi < kSeg / kEpiGroup; ++gi) {
                    const int b0 = gi * kEpiGroup;
                    if (ok && b0 < U.bcount) {
                        const int nb_g = min(kEpiGroup, U.bcount - b0);
                        const int gs = Ge % kGroupSlots, gr = Ge / kGroupSlots;
                        ok = __all_sync(0xffffffffu, tc_wait(smem_u32(&d_full[gs]), gr & 1, abort_flag, 32u, bad));
                        if (ok) {
                            tc_fence_after();
#pragma unroll
                            for (int j0 = 0; j0 < kEpiGroup; j0 += kLd) {
                                uint32_t d[kLd][2 * M];
#pragma unroll
                                for (int j = 0; j < kLd; ++j)
                                    if (j0 + j < nb_g)
                                        tmem_ld<2 * M>(tbase + lane_base + kDCol0 +
                                                           32u * static_cast<uint32_t>(gs * kEpiGroup + j0 + j),
                                                       d[j]);
                                tmem_wait_ld();
#pragma unroll
                                for (int j = 0; j < kLd; ++j) {
                                    if (j0 + j < nb_g) {
                                        const int bl = b0 + j0 + j;          // static after unrolling
                                        const uint32_t wsw = wsr[bl >> 1];
                                        const float ws = f16_bits_to_f32(
                                            static_cast<uint16_t>((bl & 1) ? (wsw >> 16) : (wsw & 0xffffu)));
#pragma unroll
                                        for (int r = 0; r < M; ++r) {
                                            const float2 pr = pairs[bl * M + r];    // (activation scale, sum q)
                                            const float x = __fmaf_rn(16.0f, __uint_as_float(d[j][2 * r]),
                                                                      __uint_as_float(d[j][2 * r + 1]));
                                            const float dv = FMT == 0 ? __fsub_rn(x, pr.y) : __fmaf_rn(128.0f, x, -pr.y);
                                            acc[r] = __fadd_rn(acc[r], __fmul_rn(dv, __fmul_rn(ws, pr.x)));
                                            if (dots != nullptr && r < a.m && grow < md.n)
                                                dots[(static_cast<size_t>(r) * md.n + grow) * md.nb + U.seg * kSeg + bl] =
                                                    __float2int_rn(dv);
                                        }
                                    }
                                }
                            }
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(smem_u32(&d_empty[gs]));
                        }
                        ++Ge;
                    }
                }
                if (!ok) break;
                if (U.phase == 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&b_empty[bs]));
                    ++kb;
                }
                // segment sums -> global; the counter warp counts the unit for
                // its tile once all four epilogue warps have stored theirs
                float *pp = U.phase == 0
                                ? a.part_a + ((static_cast<size_t>(U.mi) * md.ntiles + U.tile) * md.nseg + U.seg) * M * kTile
                                : a.part_b + (static_cast<size_t>(U.tile) * md.nseg + U.seg) * M * kTile;
#pragma unroll
                for (int r = 0; r < M; ++r)
                    if (r < a.m) __stcg(pp + r * kTile + row, acc[r]);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&unit_done[k]));
            }
        } else {
            // ------------------------------------------------------------ fold
            const int e = (warp - kWFold0) * 32 + lane;          // element / row within the tile
            const int fw = warp - kWFold0;
            int head = 0;
            for (;;) {
                if (e == 0) {
                    int job = kJobEnd;
                    const long long t0 = clock64();
                    for (;;) {
                        const int j = *reinterpret_cast<volatile int *>(&s_jobs[head]);
                        if (j != kJobEmpty) {
                            __threadfence();
                            job = j;
                            break;
                        }
                        if (*abort_flag) break;
                        if (clock64() - t0 > kFollowerBudgetCycles) {
                            bad |= 128u;
                            break;
                        }
                        __nanosleep(100);
                    }
                    s_job = job;
                }
                named_barrier(kBarFold, 32 * kNumFold);
                const int job = s_job;
                named_barrier(kBarFold, 32 * kNumFold);
                ++head;
                if (job == kJobEnd) break;
                __threadfence();               // acquire the other CTAs' segment sums
                if ((job & 0x10000) == 0) {
                    // ---- phase A tile t: h = bf16(silu(g) u), then its rotation
                    const int t = job;
                    const TcMat &gm = a.mat[0];
                    const int inter = gm.n, nseg = gm.nseg, nbh = inter / kBlock;
                    float hv[M];
#pragma unroll
                    for (int r = 0; r < M; ++r) {
                        hv[r] = 0.0f;
                        if (r >= a.m) continue;
                        float Vg[kMaxSegsA], Vu[kMaxSegsA];
                        const float *pg = a.part_a + (static_cast<size_t>(t) * nseg) * M * kTile + r * kTile + e;
                        const float *pu = a.part_a + ((static_cast<size_t>(gm.ntiles) + t) * nseg) * M * kTile + r * kTile + e;
                        load_segs(Vg, pg, nseg, static_cast<size_t>(M) * kTile);
                        load_segs(Vu, pu, nseg, static_cast<size_t>(M) * kTile);
                        const float gv = fold_tree_fixed(Vg, nseg);
                        const float uv = fold_tree_fixed(Vu, nseg);
                        const uint16_t hb = f32_to_bf16_bits(__fmul_rn(tq_silu(gv), uv));
                        if (t * kTile + e < inter) a.h[static_cast<size_t>(r) * inter + t * kTile + e] = hb;
                        hv[r] = bf16_bits_to_f32(hb);
                    }
                    if (a.rotate_h) {
                        // the operand block starts at zero (rows m..M-1 stay zero)
                        for (int i = e; i < kBBlk<M> / 16; i += kTile)
                            reinterpret_cast<uint4 *>(fold_b)[i] = make_uint4(0u, 0u, 0u, 0u);
                        // the 128-point transform on element e = this thread's row of
                        // the tile, every row r of the pass at once: spans 1..16 are
                        // lane shuffles, spans 32 and 64 go through shared memory
#pragma unroll
                        for (int sp = 1; sp < 32; sp <<= 1) {
#pragma unroll
                            for (int r = 0; r < M; ++r) {
                                const float o = __shfl_xor_sync(0xffffffffu, hv[r], sp);
                                hv[r] = (e & sp) ? __fsub_rn(o, hv[r]) : __fadd_rn(hv[r], o);
                            }
                        }
#pragma unroll
                        for (int sp = 32; sp < 128; sp <<= 1) {
#pragma unroll
                            for (int r = 0; r < M; ++r) fold_x[r * kTile + e] = hv[r];
                            named_barrier(kBarFold, 32 * kNumFold);
#pragma unroll
                            for (int r = 0; r < M; ++r) {
                                const float o = fold_x[r * kTile + (e ^ sp)];
                                hv[r] = (e & sp) ? __fsub_rn(o, hv[r]) : __fadd_rn(hv[r], o);
                            }
                            named_barrier(kBarFold, 32 * kNumFold);
                        }
#pragma unroll
                        for (int r = 0; r < M; ++r) {
                            hv[r] = __fmul_rn(hv[r], __uint_as_float(0x3db504f3u));        // (float)(1/sqrt(128))
                            const unsigned lmax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv[r])));
                            if (lane == 0) s_red[fw][r] = __uint_as_float(lmax);
                        }
                        named_barrier(kBarFold, 32 * kNumFold);
                        int qv[M];
                        float scv[M];
#pragma unroll
                        for (int r = 0; r < M; ++r) {
                            qv[r] = 0;
                            scv[r] = 0.0f;
                            const float amax = fmaxf(fmaxf(s_red[0][r], s_red[1][r]), fmaxf(s_red[2][r], s_red[3][r]));
                            if (r < a.m && amax != 0.0f) {
                                scv[r] = __fdiv_rn(amax, 127.0f);
                                const int qq = __float2int_rn(__fdiv_rn(hv[r], scv[r]));
                                qv[r] = qq > 127 ? 127 : (qq < -127 ? -127 : qq);
                            }
                            const int ls = __reduce_add_sync(0xffffffffu, qv[r]);
                            if (lane == 0) s_redi[fw][r] = ls;
                        }
                        named_barrier(kBarFold, 32 * kNumFold);
                        const int p = staged_pos<FMT>(e);
#pragma unroll
                        for (int r = 0; r < M; ++r) {
                            if (r >= a.m) continue;
                            const int hi = (qv[r] + 8) >> 4, lo = qv[r] - 16 * hi;
                            fold_b[b_off<M>(2 * r, p)] = static_cast<uint8_t>(e4m3_int(hi));
                            fold_b[b_off<M>(2 * r + 1, p)] = static_cast<uint8_t>(e4m3_int(lo));
                            a.qh[static_cast<size_t>(r) * inter + t * kTile + e] = static_cast<int8_t>(qv[r]);
                        }
                        if (e < M) {
                            const int r = e;
                            const int sum = (s_redi[0][r] + s_redi[1][r]) + (s_redi[2][r] + s_redi[3][r]);
                            if (r < a.m) a.sh[static_cast<size_t>(r) * nbh + t] = scv[r];
                            a.hsn[static_cast<size_t>(t) * M + r] =
                                r < a.m ? make_float2(scv[r], static_cast<float>(sum)) : make_float2(0.0f, 0.0f);
                        }
                        named_barrier(kBarFold, 32 * kNumFold);
                        for (int i = e; i < kBBlk<M> / 16; i += kTile)
                            __stcg(reinterpret_cast<uint4 *>(a.hst + static_cast<size_t>(t) * kBBlk<M>) + i,
                                   reinterpret_cast<const uint4 *>(fold_b)[i]);
                        named_barrier(kBarFold, 32 * kNumFold);
                        if (e == 0 && a.do_b) {
                            __threadfence();
                            red_add_release_gpu(a.segready + t / kSeg, 1u);
                        }
                    }
                } else {
                    // ---- phase B tile t: y
                    const int t = job & 0xffff;
                    const TcMat &dm = a.mat[2];
                    const int n = dm.n, nseg = dm.nseg;
                    if (t * kTile + e < n) {
#pragma unroll
                        for (int r = 0; r < M; ++r) {
                            if (r >= a.m) continue;
                            float V[kMaxSegs];
                            const float *pb = a.part_b + (static_cast<size_t>(t) * nseg) * M * kTile + r * kTile + e;
                            load_segs(V, pb, nseg, static_cast<size_t>(M) * kTile);
                            a.y[static_cast<size_t>(r) * n + t * kTile + e] = fold_tree_fixed(V, nseg);
                        }
                    }
                }
            }
        }
    }

    // ---- wind-down: every role has finished with TMEM and shared memory
    if (bad != 0u && a.err != nullptr) atomicOr(a.err, bad);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWAlloc) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace tc
}  // namespace tq
