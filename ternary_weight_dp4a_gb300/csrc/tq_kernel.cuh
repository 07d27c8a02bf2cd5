// tq_kernel.cuh -- the persistent kernel behind every GEMV and FFN entry
// point: one CTA per SM, a producer warp streaming weight tiles through a
// shared-memory ring with tensor-map copies, fifteen consumer warps turning
// them into exact block dots with prmt + dp4a (tq_dp4a.cuh).
//
// Work.  A phase multiplies m <= 4 activation rows by one or two weight
// matrices of n rows x k.  Its unit of work is 16 weight rows x one segment
// (8 consecutive 128-blocks) of one matrix: 4 KB of codes + 256 B of scales,
// one ring slot.  A CTA owns whole 16-row tiles (dealt in rounds, see Deal);
// its compute warps claim the units of its tiles as they come free.  Each unit
// yields the segment sums S_j (fold order: ascending blocks from +0) of its 16
// outputs; the warp that completes a tile's last unit folds the S_j with the
// pairwise tree and runs the tile's epilogue.
//
// Phase A (gate/up): input x rotated + quantised by every CTA (or read as
// int8), units of gate and up, epilogue h = bf16(silu(g) * u); the warp whose
// tile completes a 128-block of h rotates and quantises that block.
// Phase B (down, or a plain GEMV): input int8 rows staged from global memory
// (a segment at a time as h becomes ready, or all at once in a launch of
// phase B alone), epilogue y (fp32), optionally the int32 block dots.
// A step runs A and B in one launch without a grid barrier: a phase-B unit
// waits only until the 8 blocks of h its segment reads are rotated.  The
// producer never waits for the consumers' phases: weights do not depend on
// activations, so it streams the next phase's tiles (and this launch's first
// few tiles while the previous launch drains and the input is staged).
#pragma once

#include <cuda.h>

#include "tq_dp4a.cuh"
#include "tq_rotq.cuh"
#include "tq_stage.cuh"

namespace tq {

constexpr int kConsumerWarps = 15;      // compute warps (warp 15 is the producer)
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
// Thread count the compiler budgets registers for: the launch's own, so
// every instantiation may use 128 registers per thread (2-bit m = 3, 4 once
// measured faster capped at 96; with the hint-free barrier waits 128 is
// faster: m = 4 step 47.6 -> 47.0 us, m = 8 95.2 -> 93.7 us).
template <int FMT, int M>
constexpr int kBoundThreads = kThreads;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kCodesSlot = 4096;        // 16 rows x 8 blocks of codes (2-bit: two 2 KB planes)
constexpr int kScalesSlot = 256;        // 16 rows x 8 fp16 scales
constexpr int kMaxSlots = 48;
constexpr int kMaxRowsPerPass = 4;
// blocks of a unit per iteration of the unit core's block loop (8: the loop
// fully unrolled; fewer: a smaller hot loop)
constexpr int kOneRowBlocksPerIter = 8;
constexpr int kRowsBlocksPerIter = 4;
// Producer lanes; lane l issues units k = l (mod L), L = KArgs::lanes.  The
// ring has a multiple of L slots, so every fill of a slot comes from one
// lane, in order: when that lane waits for a slot's previous fill to be
// released, every earlier release of the slot has happened, and the phase
// parity it waits on cannot alias an older phase.  One or two rows consume a
// unit fastest and want more copies in the issue pipe (6 lanes where the
// ring has 12 slots or more); from four rows on, 4 lanes leave the compute
// warps more issue slots.
constexpr int kProducerLanesMax = 6;
static_assert(kMaxSlots % kProducerLanesMax == 0 && kMaxSlots % 4 == 0, "a full ring splits evenly among the lanes");
constexpr int kTilesPerHBlock = kBlock / kTileRows;   // 16-row tiles per 128-block of h

// How a phase's 16-row tiles are dealt to the CTAs.  CTA d (in dealing
// order) takes lv[0] tiles if d < t[0], else lv[1] if d < t[1], else lv[2] if
// d < t[2], else lv[3]; lv is non-increasing, so the CTAs that take more than
// i tiles are a prefix of the dealing order for every i.  Tiles go out in
// rounds: round i gives the next tile to each CTA of that prefix in turn, so
// every round covers a contiguous range of tiles, and the blocks of h fill up
// round after round over phase A.
struct Deal {
    int lv[4];
    int t[3];
};

__host__ __device__ inline int deal_count(const Deal &d, int c) {
    return c < d.t[0] ? d.lv[0] : c < d.t[1] ? d.lv[1] : c < d.t[2] ? d.lv[2] : d.lv[3];
}

// Tile of the j-th local tile of CTA c: the tiles of rounds 0..j-1, plus c.
__host__ __device__ inline int deal_tile(const Deal &d, int G, int c, int j) {
    // rounds [0, lv[3]) serve G CTAs, [lv[3], lv[2]) t[2], [lv[2], lv[1]) t[1], [lv[1], lv[0]) t[0]
    int base = min(j, d.lv[3]) * G;
    base += max(0, min(j, d.lv[2]) - d.lv[3]) * d.t[2];
    base += max(0, min(j, d.lv[1]) - d.lv[2]) * d.t[1];
    base += max(0, min(j, d.lv[0]) - d.lv[1]) * d.t[0];
    return base + c;
}

struct MatDesc {
    CUtensorMap tm_codes;     // uint8 {row bytes, n}, box {128, 16}, 128-byte swizzle; or
                              // (codes3d) {128, row bytes/128, n}, box {128, 2, 16}
    CUtensorMap tm_scales;    // uint16 {k/128, n}, box {8, 16} (valid when scales_tma)
    const uint8_t *codes;
    const uint16_t *scales;
    int n, k, scales_tma, codes3d;
};

enum : int { kInRotX = 0, kInNormY = 1, kInPlain = 2 };

struct KArgs {
    MatDesc mat[3];           // phase A: gate, up; phase B: mat[2]
    int do_a, do_b;
    Deal deal_a, deal_b;      // tiles per CTA of each phase
    int slots;                // ring slots (a multiple of lanes)
    int lazy_b;               // phase-B-only: stage the input by segments on demand
    int lanes;                // producer lanes issuing the units
    int prologue_slots;       // units the producer issues before the input is staged
    // dynamic shared memory: ring codes | ring scales | phase A activation +
    // (scale, magic - sum) pairs | phase B activation + pairs | segment sums |
    // int counters: units per tile, tiles folded, phase B segment state
    uint32_t off_scales, off_act, off_sn, off_acth, off_snh, off_part, off_tcnt;
    uint32_t off_scr;         // phase-B-only launches with split tiles: two tiles' segment sums
    int tiles_max, nseg_max;
    // phase A input
    int in_mode;
    const uint16_t *x;        // bf16 [M][hidden]                 (kInRotX)
    const float *y_in;        // fp32 [M][hidden]                 (kInNormY)
    float eps;
    const int8_t *qa;         // int8 [M][hidden], fp32 sa [M][hidden/128] (kInPlain)
    const float *sa;
    int8_t *qx;               // plain copy of the quantised input (CTA 0), may be null
    float *sx;
    // phase A output
    uint16_t *h;              // bf16 [M][inter]
    int rotate_h;
    int8_t *qh;               // [M][inter], [M][inter/128]
    float *sh;
    uint8_t *hst;             // h staged for phase B: [inter/128][M][128] int8
    float2 *hsn;              // [inter/128][M] (scale, magic - sum q as int bits)
    float *hp;                // [M][inter]: h after spans 1..8 of the transform, per block
                              // element e at 4 (e mod 32) + e / 32
    unsigned *hcount;         // rows of each 128-block of h published; zero on entry and on exit
    // phase B input: staged (bst/bsn, as phase A's rotation writes them) or
    // plain int8 qb [M][kB] + fp32 sb [M][kB/128]
    const uint8_t *bst;
    const float2 *bsn;
    const int8_t *qb;
    const float *sb;
    float *y;                 // fp32 [M][nB]
    int32_t *dots;            // int32 [M][nB][kB/128] or null
    // A+B launches: per 8-block segment of h, the count of its 128-blocks
    // rotated, over every launch on this workspace (never reset: launch e
    // waits for (e + 1) x blocks); the launch ticket gives e: every CTA takes
    // one ticket per launch, so launch e's CTAs hold tickets [e G, (e + 1) G)
    unsigned *segready;
    unsigned long long *ticket;
    // phase-B-only launches: when gcnt is set, CTA c takes an equal share
    // [c U / G, (c + 1) U / G) of the U units in tile-major order, and a tile
    // shared with a neighbouring CTA is folded by the CTA that completes it:
    // gpart [tiles][segments][M][16] its segment sums, gcnt [tiles] units
    // counted (zero between launches)
    float *gpart;
    unsigned *gcnt;
    unsigned *err;            // wait that ran out: bit 0 producer (slot free), 1 producer drain,
                              // 2 consumer (slot data), 3 consumer (slot issued), 4 producer
                              // (input staged), 6 phase B (segment of h); bit 5 is unused
};

// The tiles and units of one phase for CTA c of G.  Phase A deals in CTA
// order, phase B in reverse (dealing index G - 1 - c), so the CTAs holding
// one more phase-B tile are the ones the host gave fewer phase-A tiles.  Unit
// order: phase A tile-major (tile, matrix, segment); phase B of a launch that
// also runs phase A segment-major (segment, tile), so that a CTA needs the
// segments of h in the order they become ready; a phase-B-only launch
// (its whole input present at the start) tile-major (tile, segment), so
// that a CTA reads each tile's rows in one pass.
struct PhaseGeo {
    int n, k, nb, nseg, upt, ntiles, dc, count, units;
    Deal deal;
};

__host__ __device__ inline PhaseGeo phase_geo(int n, int k, int nmat, int G, int c, bool reverse, const Deal &d) {
    PhaseGeo p{};
    if (n <= 0) return p;
    p.n = n;
    p.k = k;
    p.nb = k / kBlock;
    p.nseg = (p.nb + kSegBlocks - 1) / kSegBlocks;
    p.upt = nmat * p.nseg;
    p.ntiles = (n + kTileRows - 1) / kTileRows;
    p.dc = reverse ? G - 1 - c : c;
    p.deal = d;
    p.count = deal_count(d, p.dc);
    p.units = p.count * p.upt;
    return p;
}

__device__ __forceinline__ int phase_tile(const PhaseGeo &p, int G, int lt) { return deal_tile(p.deal, G, p.dc, lt); }


// (scale, 0x4b400000 - sum q) of one staged block: the second word turns a
// biased dp4a sum into the exact fp32 block dot (int_to_float_exact).
__device__ __forceinline__ float2 block_sn(float sc, int sum) {
    return make_float2(sc, __int_as_float(kMagic - sum));
}


// Rotate + quantise rows into the staged layout, up to kRotGroup blocks per
// warp at a time so their shuffle chains overlap; load(r, b, v) fills v with
// the four values of block b of row r that this lane holds in staged order
// (rotq_staged).  CTA 0 also writes the plain copy q_out [rows][k] (natural
// order) and s_out [rows][k/128].
constexpr int kRotGroup = 3;

template <int FMT, int M, typename LoadFn>
__device__ __forceinline__ void stage_rotated(LoadFn load, int k, uint8_t *act, float2 *sn, int warp, int lane,
                                              int8_t *q_out, float *s_out, int r_only = -1) {
    const int nb = k / kBlock;
    const int rows = r_only >= 0 ? 1 : M;
    for (int blk0 = warp; blk0 < rows * nb; blk0 += kRotGroup * kConsumerWarps) {
        float v[kRotGroup][4];
#pragma unroll
        for (int u = 0; u < kRotGroup; ++u) {
            const int blk = blk0 + u * kConsumerWarps;
            const int r = r_only >= 0 ? r_only : blk / nb;
            const int b = r_only >= 0 ? blk : blk - r * nb;
            if (blk < rows * nb) load(r, b, v[u]);
            else v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0.0f;
        }
        int8_t q[kRotGroup][4];
        uint32_t word[kRotGroup];
        int sum[kRotGroup];
        float sc[kRotGroup];
#pragma unroll
        for (int u = 0; u < kRotGroup; ++u) sc[u] = rotq_staged<FMT>(v[u], lane, q[u], word[u], sum[u]);
#pragma unroll
        for (int u = 0; u < kRotGroup; ++u) {
            const int blk = blk0 + u * kConsumerWarps;
            if (blk >= rows * nb) break;
            const int r = r_only >= 0 ? r_only : blk / nb;
            const int b = r_only >= 0 ? blk : blk - r * nb;
            *reinterpret_cast<uint32_t *>(act + static_cast<size_t>(b * M + r) * kBlock + 4 * lane) = word[u];
            if (lane == 0) sn[b * M + r] = block_sn(sc[u], sum[u]);
            if (q_out != nullptr) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    q_out[static_cast<size_t>(r) * k + b * kBlock + staged_elem<FMT>(4 * lane + c)] = q[u][c];
                if (lane == 0) s_out[static_cast<size_t>(r) * nb + b] = sc[u];
            }
        }
    }
}


// One unit: 16 weight rows x the segment's blocks.  Lane l = 2r + h works
// on row r, half h of every block (with the 128-byte swizzle, each quarter
// warp then reads 8 distinct 16-byte bank groups of the codes) (2-bit: words 4h..4h+3, 64 weights; 1-bit:
// words 2h, 2h+1); each code word feeds its own dp4a chain, the chains and
// the two halves meet in adds and one shuffle, and lanes 2r, 2r + 1 fold
// t_b = (float)d * (ws * sa) into the segment sums acc[mm] in ascending block
// order.  dots (may be null) receives every block dot.  FAST: a full
// segment, no dots, 2-bit codes in the 3D layout (the common case, compiled
// without the per-block checks).
template <int FMT, int M, bool FAST>
__device__ __forceinline__ void unit_dp4a_1row(const uint8_t *cs, bool codes3d, const uint8_t *act, const float2 *sn,
                                          int b0, int bcount, const uint32_t (&wsr)[4], int lane, float (&acc)[M],
                                          int32_t *dots, int row, int n, int nb) {
    const int r = lane >> 1, h = lane & 1;
    if (FAST) codes3d = true;
    (void)codes3d;
    // kOneRowBlocksPerIter blocks per iteration (as unit_dp4a_rows)
    constexpr int U = kOneRowBlocksPerIter;
    uint32_t wsq[4] = {wsr[0], wsr[1], wsr[2], wsr[3]};
#pragma unroll 1
    for (int bi = 0; bi < kSegBlocks; bi += U) {
#pragma unroll
    for (int bj = 0; bj < U; ++bj) {
        const int bl = bi + bj;
        if (!FAST && bl >= bcount) break;
        const int b = b0 + bl;
        int dot[M];
        const uint8_t *ab = act + static_cast<size_t>(b) * M * kBlock + h * 64;
        if constexpr (FMT == 0) {
            // 128-byte line of (row r, plane bl/4): 3D copies lay rows out
            // [row][plane], 2D copies [plane][row]; the swizzle XORs the
            // 16-byte chunk with the line index mod 8
            const int line = codes3d ? 2 * r + (bl >> 2) : (bl >> 2) * kTileRows + r;
            const uint4 cw = *reinterpret_cast<const uint4 *>(cs + line * 128 +
                                                              ((((bl & 3) * 2 + h) ^ (line & 7)) * 16));
            const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
            int part[M][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t p0, p1, p2, p3;
                decode_t2(words[i], p0, p1, p2, p3);
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    const uint4 av = *reinterpret_cast<const uint4 *>(ab + mm * kBlock + i * 16);
                    int d = __dp4a(static_cast<int>(p0), static_cast<int>(av.x), 0);
                    d = __dp4a(static_cast<int>(p1), static_cast<int>(av.y), d);
                    d = __dp4a(static_cast<int>(p2), static_cast<int>(av.z), d);
                    part[mm][i] = __dp4a(static_cast<int>(p3), static_cast<int>(av.w), d);
                }
            }
#pragma unroll
            for (int mm = 0; mm < M; ++mm) dot[mm] = (part[mm][0] + part[mm][1]) + (part[mm][2] + part[mm][3]);
        } else {
            const uint2 cw = *reinterpret_cast<const uint2 *>(cs + r * 128 + ((bl ^ (r & 7)) * 16) + h * 8);
            const uint32_t words[2] = {cw.x, cw.y};
            int part[M][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    const uint4 a0 = *reinterpret_cast<const uint4 *>(ab + mm * kBlock + i * 32);
                    const uint4 a1 = *reinterpret_cast<const uint4 *>(ab + mm * kBlock + i * 32 + 16);
                    const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    int d0 = 0, d1 = 0;
#pragma unroll
                    for (int sb = 0; sb < 8; sb += 2) {
                        d0 = __dp4a(static_cast<int>((words[i] >> sb) & 0x01010101u), static_cast<int>(av[sb]), d0);
                        d1 = __dp4a(static_cast<int>((words[i] >> (sb + 1)) & 0x01010101u), static_cast<int>(av[sb + 1]), d1);
                    }
                    part[mm][2 * i] = d0;
                    part[mm][2 * i + 1] = d1;
                }
            }
#pragma unroll
            for (int mm = 0; mm < M; ++mm) dot[mm] = (part[mm][0] + part[mm][1]) + (part[mm][2] + part[mm][3]);
        }
        const uint32_t wsw = wsq[bj >> 1];
        const float ws = f16_bits_to_f32(static_cast<uint16_t>((bj & 1) ? (wsw >> 16) : (wsw & 0xffffu)));
#pragma unroll
        for (int mm = 0; mm < M; ++mm) {
            int d = dot[mm] + __shfl_xor_sync(0xffffffffu, dot[mm], 1);
            if (FMT == 1) d *= 2;
            const float2 sv = sn[b * M + mm];                // (activation scale, magic - sum q)
            const float v = int_to_float_exact(d, __float_as_int(sv.y));
            acc[mm] = __fadd_rn(acc[mm], __fmul_rn(v, __fmul_rn(ws, sv.x)));
            if (!FAST && dots != nullptr && h == 0 && row < n)
                dots[(static_cast<size_t>(mm) * n + row) * nb + b] = __float2int_rn(v);
        }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) wsq[t] = t + U / 2 < 4 ? wsq[(t + U / 2) & 3] : 0u;
    }
}

template <int FMT, int M, bool FAST>
__device__ __forceinline__ void unit_dp4a_rows(const uint8_t *cs, bool codes3d, const uint8_t *act, const float2 *sn,
                                          int b0, int bcount, const uint32_t (&wsr)[4], int lane, float (&acc)[M],
                                          int32_t *dots, int row, int n, int nb) {
    const int r = lane >> 1, h = lane & 1;
    if (FAST) codes3d = true;
    (void)codes3d;
    // kRowsBlocksPerIter blocks per iteration of a loop that is not
    // unrolled (a smaller hot loop); the scale words shift down in registers
    constexpr int U = kRowsBlocksPerIter;
    uint32_t wsq[4] = {wsr[0], wsr[1], wsr[2], wsr[3]};
#pragma unroll 1
    for (int bi = 0; bi < kSegBlocks; bi += U) {
#pragma unroll
    for (int bj = 0; bj < U; ++bj) {
        const int bl = bi + bj;
        if (!FAST && bl >= bcount) break;
        const int b = b0 + bl;
        int dot[M];
        float2 sv[M];                                        // (activation scale, magic - sum q)
#pragma unroll
        for (int mm = 0; mm < M; ++mm) sv[mm] = sn[b * M + mm];
        const uint8_t *ab = act + static_cast<size_t>(b) * M * kBlock + h * 64;
        if constexpr (FMT == 0) {
            // 128-byte line of (row r, plane bl/4): 3D copies lay rows out
            // [row][plane], 2D copies [plane][row]; the swizzle XORs the
            // 16-byte chunk with the line index mod 8
            const int line = codes3d ? 2 * r + (bl >> 2) : (bl >> 2) * kTileRows + r;
            const uint4 cw = *reinterpret_cast<const uint4 *>(cs + line * 128 +
                                                              ((((bl & 3) * 2 + h) ^ (line & 7)) * 16));
            const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
            // two dp4a chains per row (words 0-1, words 2-3); the h = 0 half's
            // first chain starts from the block's magic - sum q, so the halves'
            // sum is the biased value the exact conversion needs
            constexpr int kChains = 2;
            int part[M][kChains];
#pragma unroll
            for (int mm = 0; mm < M; ++mm) {
                part[mm][0] = h == 0 ? __float_as_int(sv[mm].y) : 0;
#pragma unroll
                for (int ch = 1; ch < kChains; ++ch) part[mm][ch] = 0;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t p0, p1, p2, p3;
                decode_t2(words[i], p0, p1, p2, p3);
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    const uint4 av = *reinterpret_cast<const uint4 *>(ab + mm * kBlock + i * 16);
                    int d = part[mm][i * kChains / 4];
                    d = __dp4a(static_cast<int>(p0), static_cast<int>(av.x), d);
                    d = __dp4a(static_cast<int>(p1), static_cast<int>(av.y), d);
                    d = __dp4a(static_cast<int>(p2), static_cast<int>(av.z), d);
                    part[mm][i * kChains / 4] = __dp4a(static_cast<int>(p3), static_cast<int>(av.w), d);
                }
            }
#pragma unroll
            for (int mm = 0; mm < M; ++mm) {
                int sum = part[mm][0];
#pragma unroll
                for (int ch = 1; ch < kChains; ++ch) sum += part[mm][ch];
                dot[mm] = sum;
            }
        } else {
            const uint2 cw = *reinterpret_cast<const uint2 *>(cs + r * 128 + ((bl ^ (r & 7)) * 16) + h * 8);
            const uint32_t words[2] = {cw.x, cw.y};
            int part[M][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    const uint4 a0 = *reinterpret_cast<const uint4 *>(ab + mm * kBlock + i * 32);
                    const uint4 a1 = *reinterpret_cast<const uint4 *>(ab + mm * kBlock + i * 32 + 16);
                    const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    int d0 = 0, d1 = 0;
#pragma unroll
                    for (int sb = 0; sb < 8; sb += 2) {
                        d0 = __dp4a(static_cast<int>((words[i] >> sb) & 0x01010101u), static_cast<int>(av[sb]), d0);
                        d1 = __dp4a(static_cast<int>((words[i] >> (sb + 1)) & 0x01010101u), static_cast<int>(av[sb + 1]), d1);
                    }
                    part[mm][2 * i] = d0;
                    part[mm][2 * i + 1] = d1;
                }
            }
#pragma unroll
            for (int mm = 0; mm < M; ++mm) dot[mm] = (part[mm][0] + part[mm][1]) + (part[mm][2] + part[mm][3]);
        }
        const uint32_t wsw = wsq[bj >> 1];
        const float ws = f16_bits_to_f32(static_cast<uint16_t>((bj & 1) ? (wsw >> 16) : (wsw & 0xffffu)));
#pragma unroll
        for (int mm = 0; mm < M; ++mm) {
            const int d = dot[mm] + __shfl_xor_sync(0xffffffffu, dot[mm], 1);
            // 2-bit: d already holds magic - sum; 1-bit: 2 d + (magic - sum)
            const int biased = FMT == 0 ? d : 2 * d + __float_as_int(sv[mm].y);
            const float v = __fsub_rn(__int_as_float(biased), 12582912.0f);   // exact: |d| < 2^22
            acc[mm] = __fadd_rn(acc[mm], __fmul_rn(v, __fmul_rn(ws, sv[mm].x)));
            if (!FAST && dots != nullptr && h == 0 && row < n)
                dots[(static_cast<size_t>(mm) * n + row) * nb + b] = __float2int_rn(v);
        }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) wsq[t] = t + U / 2 < 4 ? wsq[(t + U / 2) & 3] : 0u;
    }
}

// One unit, dispatched on the row count: one row keeps four short dp4a
// chains per block (latency); more rows use two longer chains per row and fold
// the block's magic - sum q into the first (fewer integer adds).
template <int FMT, int M, bool FAST>
__device__ __forceinline__ void unit_dp4a(const uint8_t *cs, bool codes3d, const uint8_t *act, const float2 *sn,
                                          int b0, int bcount, const uint32_t (&wsr)[4], int lane, float (&acc)[M],
                                          int32_t *dots, int row, int n, int nb) {
    if constexpr (M == 1)
        unit_dp4a_1row<FMT, M, FAST>(cs, codes3d, act, sn, b0, bcount, wsr, lane, acc, dots, row, n, nb);
    else
        unit_dp4a_rows<FMT, M, FAST>(cs, codes3d, act, sn, b0, bcount, wsr, lane, acc, dots, row, n, nb);
}

// Stage blocks [b_begin, b_end) of int8 rows q [M][k] (+ fp32 s [M][k/128])
// from global memory, warps w, w + nw, ... taking (row, block) pairs; each
// warp loads a group of up to 8 blocks (a segment of one row) before working
// on any of them.
template <int FMT, int M>
__device__ __forceinline__ void stage_plain_range(const int8_t *__restrict__ q, const float *__restrict__ s, int k,
                                                  int b_begin, int b_end, uint8_t *act, float2 *sn, int w, int nw,
                                                  int lane) {
    const int nb = k / kBlock, cnt = b_end - b_begin;
    constexpr int kGroup = 8;
    for (int p0 = w; p0 < M * cnt; p0 += kGroup * nw) {
        uint32_t wd[kGroup];
        float sc[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int p = p0 + u * nw;
            wd[u] = 0u;
            sc[u] = 0.0f;
            if (p < M * cnt) {
                const int r = p / cnt, b = b_begin + (p - r * cnt);
                wd[u] = __ldcg(reinterpret_cast<const unsigned *>(q + static_cast<size_t>(r) * k + static_cast<size_t>(b) * kBlock) + lane);
                sc[u] = __ldcg(s + static_cast<size_t>(r) * nb + b);
            }
        }
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            const int p = p0 + u * nw;
            if (p >= M * cnt) break;
            const int r = p / cnt, b = b_begin + (p - r * cnt);
            uint8_t *dst = act + static_cast<size_t>(b * M + r) * kBlock;
            int sum = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int v = static_cast<int8_t>(wd[u] >> (8 * i));
                dst[staged_pos<FMT>(4 * lane + i)] = static_cast<uint8_t>(v);
                sum += v;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (lane == 0) sn[b * M + r] = block_sn(sc[u], sum);
        }
    }
}

// Make segment j of phase B's activation present in shared memory.  The
// first warp to need it stages it (after, in a launch that also runs phase
// A, the segment's 128-blocks of h have all been rotated somewhere on the
// GPU); other warps wait for it.  Returns false if a bounded wait ran out.
template <int FMT, int M>
__device__ bool stage_segment_b(const KArgs &a, const PhaseGeo &P, int j, uint8_t *act_h, float2 *sn_h,
                                int *segst, unsigned epoch, int lane) {
    volatile int *vst = segst;
    // lane 0 reads the segment's state and claims it; the warp follows its
    // broadcast (per-lane reads of a flag can differ and split the warp)
    int state = 0;
    if (lane == 0) {
        state = vst[j];
        if (state != 2) state = atomicCAS(&segst[j], 0, 1) == 0 ? 3 : 1;
    }
    state = __shfl_sync(0xffffffffu, state, 0);
    if (state == 2) {
        __threadfence_block();
        return true;
    }
    const int claim = state == 3;
    const int b0 = j * kSegBlocks, bc = min(kSegBlocks, P.nb - b0);
    int ok = 1;
    if (claim) {
        if (a.do_a && lane == 0) {
            const long long t0 = clock64();
            // counts wrap modulo 2^32; this launch's target is never more
            // than bc ahead of the count
            const unsigned target = (epoch + 1u) * static_cast<unsigned>(bc);
            while (static_cast<int>(ld_acquire_u32(a.segready + j) - target) < 0) {
                if (clock64() - t0 > kWaitBudgetCycles) {
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (a.bst != nullptr) {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.bst + static_cast<size_t>(b0) * M * kBlock);
            uint4 *dst = reinterpret_cast<uint4 *>(act_h + static_cast<size_t>(b0) * M * kBlock);
            for (int i = lane; i < bc * M * kBlock / 16; i += 32) dst[i] = __ldcg(src + i);
            for (int i = lane; i < bc * M; i += 32) sn_h[b0 * M + i] = __ldcg(a.bsn + b0 * M + i);
        } else {
            stage_plain_range<FMT, M>(a.qb, a.sb, P.k, b0, b0 + bc, act_h, sn_h, 0, 1, lane);
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) atomicExch(&segst[j], 2);
    } else if (lane == 0) {
        const long long t0 = clock64();
        while (vst[j] != 2) {
            if (clock64() - t0 > kWaitBudgetCycles) {
                ok = 0;
                break;
            }
            __nanosleep(32);
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __threadfence_block();
    return ok != 0;
}

// Decoded position of a phase's unit: phase A (outer = tile, inner = matrix
// x segment), phase B (outer = segment, inner = tile, or tile-major as phase
// A); inner runs fastest.
struct UnitPos {
    int outer, inner;
};

__device__ __forceinline__ void unit_advance(UnitPos &u, int step, int extent) {
    u.inner += step;
    while (u.inner >= extent) {
        u.inner -= extent;
        ++u.outer;
    }
}

// Rotate and quantise 128-block hb of h (all M rows, every row of it
// published).  The transform runs in the staged order phase B reads: the
// stages go in element-span order 1, 2, ..., 64, each elementwise, so the
// values are those of the natural-order transform, and each lane's four codes
// are four consecutive staged bytes (one store).  The staged copy hst/hsn is
// written first and released (a release add to its segment's ready counter
// when phase B runs in this launch); qh/sh for the caller and the block's
// count reset come after.
template <int FMT, int M>
__device__ __forceinline__ void rotate_h_block(const KArgs &a, int n, int hb, int lane) {
    const int nbh = n / kBlock;
    // hp holds the block after spans 1..8 (applied by the warps that folded
    // its tiles); lane l reads elements l, l+32, l+64, l+96
    float v[M][4];
#pragma unroll
    for (int rr = 0; rr < M; ++rr) {
        const float4 w = __ldcg(reinterpret_cast<const float4 *>(a.hp + static_cast<size_t>(rr) * n + hb * kBlock) + lane);
        v[rr][0] = w.x; v[rr][1] = w.y; v[rr][2] = w.z; v[rr][3] = w.w;
    }
    int8_t q[M][4];
    float sc[M];
#pragma unroll
    for (int rr = 0; rr < M; ++rr) {
        // spans 16 (lane bit 4), 32 and 64 (register bits 0 and 1)
        wht_stage(v[rr], lane, 16, 0);
        wht_stage(v[rr], lane, 0, 1);
        wht_stage(v[rr], lane, 0, 2);
        int sum;
        sc[rr] = scale_quant4(v[rr], q[rr], sum);
        uint8_t *hst = a.hst + static_cast<size_t>(hb * M + rr) * kBlock;
#pragma unroll
        for (int c = 0; c < 4; ++c) hst[staged_pos<FMT>(lane + 32 * c)] = static_cast<uint8_t>(q[rr][c]);
        if (lane == 0) a.hsn[hb * M + rr] = block_sn(sc[rr], sum);
    }
    __syncwarp();
    if (lane == 0 && a.do_b) red_add_release_gpu(a.segready + hb / kSegBlocks, 1u);
#pragma unroll
    for (int rr = 0; rr < M; ++rr) {
#pragma unroll
        for (int c = 0; c < 4; ++c) a.qh[static_cast<size_t>(rr) * n + hb * kBlock + lane + 32 * c] = q[rr][c];
        if (lane == 0) a.sh[static_cast<size_t>(rr) * nbh + hb] = sc[rr];
    }
    if (lane == 0) a.hcount[hb] = 0u;
}

// BO: a launch of phase B alone (a GEMV, or the down projection of a staged
// h), compiled separately: no phase-A code, the input staged up front (or by
// segments as warps first need them, KArgs::lazy_b), units tile-major (whole tiles per CTA, or equal shares of the units with
// the shared tiles folded across CTAs, see KArgs::gcnt).
template <int FMT, int M, bool BO>
__global__ void __launch_bounds__(kBoundThreads<FMT, M>, 1) tq_kernel(const __grid_constant__ KArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kMaxSlots];
    __shared__ __align__(8) uint64_t empty_bar[kMaxSlots];
    __shared__ __align__(8) uint64_t input_bar;     // phase A's input staged (one arrival)
    __shared__ float s_warp[8];
    __shared__ int s_next;                           // next unit a compute warp claims
    __shared__ unsigned s_epoch;                     // this launch's index on the workspace (A+B launches)
    // unit the producer last issued into each slot.  A consumer waits for its
    // unit's number here before it waits for the slot's data: a warp may
    // claim unit k + S while unit k still waits for its data, and the slot's
    // barrier phase parity alone cannot tell those two fills apart.
    __shared__ int slot_unit[kMaxSlots];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int S = a.slots;
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *codes_ring = base;
    const uint16_t *scales_ring = reinterpret_cast<const uint16_t *>(base + a.off_scales);
    uint8_t *act_x = base + a.off_act;
    float2 *sn_x = reinterpret_cast<float2 *>(base + a.off_sn);
    uint8_t *act_h = base + a.off_acth;
    float2 *sn_h = reinterpret_cast<float2 *>(base + a.off_snh);
    float *part = reinterpret_cast<float *>(base + a.off_part);
    // int counters: units done per local tile of phase A, of phase B; phase B
    // segments (0 absent, 1 staging, 2 staged)
    int *tcnt = reinterpret_cast<int *>(base + a.off_tcnt);
    int *segst = tcnt + 2 * a.tiles_max;

    const PhaseGeo ga = (!BO && a.do_a) ? phase_geo(a.mat[0].n, a.mat[0].k, 2, G, cta, false, a.deal_a) : PhaseGeo{};
    const PhaseGeo gb = a.do_b ? phase_geo(a.mat[2].n, a.mat[2].k, 1, G, cta, true, a.deal_b) : PhaseGeo{};
    // a phase-B-only launch with split tiles: this CTA's units [u0, u1) of
    // the tile-major order, from (global) tile t0 on
    const bool split = BO && a.gcnt != nullptr;
    int u0 = 0, u1 = gb.units;
    if (split) {
        const long long U = static_cast<long long>(gb.ntiles) * gb.upt;
        u0 = static_cast<int>(cta * U / G);
        u1 = static_cast<int>((cta + 1) * U / G);
    }
    const int t0 = split ? u0 / max(gb.upt, 1) : 0;
    const int total = split ? u1 - u0 : ga.units + gb.units;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&input_bar), 1);
        mbar_init_fence();
        s_next = 0;
    }
    for (int i = threadIdx.x; i < kMaxSlots; i += kThreads) slot_unit[i] = -1;
    for (int i = threadIdx.x; i < 2 * a.tiles_max + a.nseg_max; i += kThreads) tcnt[i] = 0;
    __syncthreads();
    pdl_launch_dependents();

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        // Lanes 0..L-1 each issue every L-th unit (L = a.lanes),
        // so several units are in the issue pipe at once; unit positions and
        // (slot, round) = divmod(k, S) advance incrementally.  Only the first
        // prologue_slots units go out before the consumers have staged the
        // input: the input's loads would otherwise queue behind a full ring
        // of weight copies.
        const int L = a.lanes;
        if (lane < L) {
            bool ok = true;
            unsigned bad = 0u;
            int k = lane;
            bool in_a = !BO && k < ga.units;
            const int bext = max(BO ? gb.upt : gb.count, 1);   // phase B's inner extent
            // weights are read once per launch: evict them first, keeping
            // activations and other kernels' data in L2
            const uint64_t wpol = l2_policy_evict_first();
            UnitPos u{0, in_a ? k : k - ga.units + (split ? u0 : 0)};
            unit_advance(u, 0, in_a ? max(ga.upt, 1) : bext);
            int slot = k % S, round = k / S;
            for (; k < total && ok; k += L) {
                if (in_a && k >= ga.units) {
                    in_a = false;
                    u = UnitPos{0, k - ga.units};
                    unit_advance(u, 0, bext);
                }
                const PhaseGeo &P = in_a ? ga : gb;
                int mi, seg, lt;
                if (in_a) {
                    lt = u.outer;
                    mi = u.inner >= P.nseg ? 1 : 0;
                    seg = u.inner - mi * P.nseg;
                } else {
                    seg = BO ? u.inner : u.outer;
                    lt = BO ? u.outer - t0 : u.inner;
                    mi = 2;
                }
                const int tile = split ? t0 + lt : phase_tile(P, G, lt);
                const MatDesc &md = a.mat[mi];
                if (k >= a.prologue_slots && k < a.prologue_slots + L &&
                    !(ok = mbar_wait(smem_u32(&input_bar), 0))) {
                    bad |= 16u;
                    break;
                }
                if (round > 0 && !(ok = mbar_wait(smem_u32(&empty_bar[slot]), (round - 1) & 1))) {
                    bad |= 1u;
                    break;
                }
                reinterpret_cast<volatile int *>(slot_unit)[slot] = k;
                const uint32_t fb = smem_u32(&full_bar[slot]);
                const uint32_t dst = smem_u32(codes_ring + static_cast<size_t>(slot) * kCodesSlot);
                const bool sct = md.scales_tma != 0;
                if (FMT == 0 && md.codes3d) {
                    mbar_arrive_expect_tx(fb, 4096u + (sct ? kScalesSlot : 0u));
                    tma_load_3d(dst, &md.tm_codes, 0, seg * 2, tile * kTileRows, fb, wpol);
                } else {
                    const int planes = FMT == 0 ? (seg * kSegBlocks + 4 < P.nb ? 2 : 1) : 1;
                    mbar_arrive_expect_tx(fb, planes * 2048u + (sct ? kScalesSlot : 0u));
                    const int x0 = FMT == 0 ? seg * kSegBlocks * 32 : seg * kSegBlocks * 16;
                    tma_load_2d(dst, &md.tm_codes, x0, tile * kTileRows, fb, wpol);
                    if (planes == 2) tma_load_2d(dst + 2048, &md.tm_codes, x0 + 128, tile * kTileRows, fb, wpol);
                }
                if (sct)
                    tma_load_2d(smem_u32(scales_ring + static_cast<size_t>(slot) * (kScalesSlot / 2)), &md.tm_scales,
                                seg * kSegBlocks, tile * kTileRows, fb, wpol);
                unit_advance(u, L, in_a ? P.upt : bext);
                slot += L;
                if (slot >= S) {
                    slot -= S;
                    ++round;
                }
            }
            // no copy may still be landing in shared memory when the CTA
            // exits.  Every fill of a slot comes from one lane, so this lane's
            // last S / L units are the last fills of its slots
            // (earlier fills were consumed before their slot was refilled):
            // wait for those, newest first.  When the consumers took every
            // unit, all have landed and each check returns at once.
            for (int kk = k - L, n = 0; kk >= 0 && n < S / L; kk -= L, ++n)
                if (!mbar_wait(smem_u32(&full_bar[kk % S]), (kk / S) & 1)) {
                    bad |= 2u;
                    break;
                }
            if (bad != 0u && a.err != nullptr) atomicOr(a.err, bad);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int tid = threadIdx.x;             // 0 .. kConsumers-1
    bool ok = true;
    unsigned bad = 0u;                       // error bits of the waits that ran out
    pdl_wait();
    // A+B launches that rotate h take a launch ticket; its result is needed
    // only in phase B, so it is stored after the input is staged
    const bool ticketed = !BO && a.do_a && a.do_b && a.rotate_h;
    unsigned long long ticket = 0;
    if (ticketed && tid == 0) ticket = atomicAdd(a.ticket, 1ull);

    // ---- phase A's activation: every CTA rotates + quantises the input
    if (!BO && a.do_a) {
        const int hidden = ga.k;
        if (a.in_mode == kInRotX) {
            const uint16_t *x = a.x;
            stage_rotated<FMT, M>([&](int r, int b, float (&v)[4]) {
                load_staged_bf16<FMT>(x + static_cast<size_t>(r) * hidden + b * kBlock, lane, v, false);
            }, hidden, act_x, sn_x, warp, lane, cta == 0 ? a.qx : nullptr, a.sx);
        } else if (a.in_mode == kInNormY) {
            for (int r = 0; r < M; ++r) {
                // 1/rms: 256 partial sums (thread i adds y[i], y[i+256], ...),
                // each warp's 32 combined at distance 1, 2, ..., 16, then
                // ((w0+w1)+(w2+w3)) + ((w4+w5)+(w6+w7))
                const float *yr = a.y_in + static_cast<size_t>(r) * hidden;
                float acc = 0.0f;
                if (tid < 256)
                    for (int i = tid; i < hidden; i += 256) {
                        const float v = __ldcg(yr + i);
                        acc = __fadd_rn(acc, __fmul_rn(v, v));
                    }
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
                if (lane == 0 && warp < 8) s_warp[warp] = acc;
                named_barrier(1, kConsumers);
                const float w01 = __fadd_rn(s_warp[0], s_warp[1]), w23 = __fadd_rn(s_warp[2], s_warp[3]);
                const float w45 = __fadd_rn(s_warp[4], s_warp[5]), w67 = __fadd_rn(s_warp[6], s_warp[7]);
                const float ss = __fadd_rn(__fadd_rn(w01, w23), __fadd_rn(w45, w67));
                const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(hidden)), a.eps)));
                named_barrier(1, kConsumers);
                stage_rotated<FMT, M>([&](int, int b, float (&v)[4]) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        v[c] = bf16_bits_to_f32(f32_to_bf16_bits(
                            __fmul_rn(__ldcg(yr + b * kBlock + staged_elem<FMT>(4 * lane + c)), inv)));
                }, hidden, act_x, sn_x, warp, lane, cta == 0 ? a.qx : nullptr, a.sx, r);
            }
        } else {
            stage_plain_range<FMT, M>(a.qa, a.sa, hidden, 0, ga.nb, act_x, sn_x, warp, kConsumerWarps, lane);
        }
        if (ticketed && tid == 0) s_epoch = static_cast<unsigned>(ticket / static_cast<unsigned long long>(G));
        named_barrier(1, kConsumers);
    } else if (BO && !a.lazy_b) {
        // ---- a phase-B-only launch: its whole input is in memory already
        // (the grid-dependency wait above); stage it once, all warps.  With
        // lazy_b the first warp to need a segment stages it instead, as
        // phase B does in a fused launch (a long input at one or two rows:
        // no warp waits for the whole input before its first unit)
        if (a.bst != nullptr) {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.bst);
            uint4 *dst = reinterpret_cast<uint4 *>(act_h);
            for (int i = tid; i < gb.nb * M * kBlock / 16; i += kConsumers) dst[i] = __ldcg(src + i);
            for (int i = tid; i < gb.nb * M; i += kConsumers) sn_h[i] = __ldcg(a.bsn + i);
        } else {
            stage_plain_range<FMT, M>(a.qb, a.sb, gb.k, 0, gb.nb, act_h, sn_h, warp, kConsumerWarps, lane);
        }
        named_barrier(1, kConsumers);
    }
    if (tid == 0) mbar_arrive(smem_u32(&input_bar));

    // ---- units: CTA-local index k over phase A then phase B.  A compute
    // warp claims the next unit from a shared counter when it is free, so a
    // warp that runs slow (or waits for a segment of h) holds up no other
    // warp's units.  A warp's claims increase, so its unit positions and
    // (slot, round) = divmod(k, S) advance incrementally.
    const int ncw = kConsumerWarps;
    int *tcnt_a = tcnt, *tcnt_b = tcnt + a.tiles_max;
    float *part_a = part, *part_b = part + static_cast<size_t>(ga.units) * M * kTileRows;
    if (warp < ncw) {
        int kp = 0, slot = 0, round = 0;
        bool in_a = !BO && ga.units > 0;
        const int bext = max(BO ? gb.upt : gb.count, 1);   // phase B's inner extent
        UnitPos u{0, split ? u0 : 0};
        int staged_seg = -1;
        for (;;) {
            int k = 0;
            if (lane == 0) k = atomicAdd(&s_next, 1);
            k = __shfl_sync(0xffffffffu, k, 0);
            if (k >= total) break;
            if (in_a && k >= ga.units) {
                in_a = false;
                u = UnitPos{0, 0};
                unit_advance(u, k - ga.units, bext);
            } else {
                unit_advance(u, k - kp, in_a ? ga.upt : bext);
            }
            slot += k - kp;
            while (slot >= S) {
                slot -= S;
                ++round;
            }
            kp = k;
            const PhaseGeo &P = in_a ? ga : gb;
            int mi, seg, lt;
            if (in_a) {
                lt = u.outer;
                mi = u.inner >= P.nseg ? 1 : 0;
                seg = u.inner - mi * P.nseg;
            } else {
                seg = BO ? u.inner : u.outer;
                lt = BO ? u.outer - t0 : u.inner;
                mi = 2;
                if ((!BO || a.lazy_b) && seg != staged_seg) {
                    if (!stage_segment_b<FMT, M>(a, P, seg, act_h, sn_h, segst, s_epoch, lane)) {
                        ok = false;
                        bad |= 64u;
                    }
                    staged_seg = seg;
                }
            }
            const int i = in_a ? k : k - ga.units;          // unit index within its phase
            if (ok && lane == 0) {
                const volatile int *vsu = slot_unit;
                const long long t0 = clock64();
                while (vsu[slot] != k) {
                    if (clock64() - t0 > kWaitBudgetCycles) {
                        ok = false;
                        bad |= 8u;
                        break;
                    }
                    __nanosleep(20);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (ok && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&full_bar[slot]), round & 1))) {
                ok = false;
                bad |= 4u;
            }
            if (!ok) break;
            const int tile = split ? t0 + lt : phase_tile(P, G, lt);
            const MatDesc &md = a.mat[mi];
            const uint8_t *cs = codes_ring + static_cast<size_t>(slot) * kCodesSlot;
            const int bcount = min(kSegBlocks, P.nb - seg * kSegBlocks);

            // weight scales of the lane's row (lane 2r + h: row r of the tile)
            // for the segment's blocks
            const int urow = tile * kTileRows + (lane >> 1);
            uint32_t wsr[4];
            if (md.scales_tma) {
                const uint4 u0 = *reinterpret_cast<const uint4 *>(scales_ring + static_cast<size_t>(slot) * (kScalesSlot / 2) + (lane >> 1) * 8);
                wsr[0] = u0.x; wsr[1] = u0.y; wsr[2] = u0.z; wsr[3] = u0.w;
            } else {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t lo = 0, hi = 0;
                    const int bb = seg * kSegBlocks + 2 * w;
                    if (urow < P.n && 2 * w < bcount) lo = ldg_u16(md.scales + static_cast<size_t>(urow) * P.nb + bb);
                    if (urow < P.n && 2 * w + 1 < bcount) hi = ldg_u16(md.scales + static_cast<size_t>(urow) * P.nb + bb + 1);
                    wsr[w] = lo | (hi << 16);
                }
            }

            float acc[M];
#pragma unroll
            for (int mm = 0; mm < M; ++mm) acc[mm] = 0.0f;
            int32_t *const dots = in_a ? nullptr : a.dots;
            if (bcount == kSegBlocks && dots == nullptr && (FMT == 1 || md.codes3d))
                unit_dp4a<FMT, M, true>(cs, true, in_a ? act_x : act_h, in_a ? sn_x : sn_h, seg * kSegBlocks,
                                        bcount, wsr, lane, acc, nullptr, urow, P.n, P.nb);
            else
                unit_dp4a<FMT, M, false>(cs, md.codes3d != 0, in_a ? act_x : act_h, in_a ? sn_x : sn_h,
                                         seg * kSegBlocks, bcount, wsr, lane, acc, dots, urow, P.n, P.nb);
            // the slot's codes and scales are all in registers: hand it back
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));

            // segment sums of this unit -> shared memory; count the tile
            float *pu = (in_a ? part_a : part_b) + static_cast<size_t>(i) * M * kTileRows;
            if ((lane & 1) == 0) {
#pragma unroll
                for (int mm = 0; mm < M; ++mm) pu[mm * kTileRows + (lane >> 1)] = acc[mm];
            }
            __syncwarp();
            // this CTA's units of the tile: all of them, or (split tiles) the
            // ones inside [u0, u1), local units i_lo .. i_lo + nloc - 1
            const int tb = tile * P.upt;
            const int nloc = split ? min(u1, tb + P.upt) - max(u0, tb) : P.upt;
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                last = atomicAdd(&(in_a ? tcnt_a : tcnt_b)[lt], 1) == nloc - 1;
            }
            if (!__shfl_sync(0xffffffffu, last, 0)) continue;
            __threadfence_block();
            // a tile shared with another CTA: publish this CTA's segment sums
            // and count its units in; the CTA whose count completes the tile
            // gathers all of them into its scratch and folds them there
            float *tile_sums = nullptr;
            if (split && nloc < P.upt) {
                const int i_lo = max(u0, tb) - u0, s_lo = max(u0, tb) - tb;
                const size_t w = static_cast<size_t>(M) * kTileRows;
                float *gp = a.gpart + static_cast<size_t>(tb) * w;
                for (int e = lane; e < nloc * static_cast<int>(w); e += 32)
                    gp[s_lo * w + e] = part_b[static_cast<size_t>(i_lo) * w + e];
                __syncwarp();
                int done = 0;
                if (lane == 0) {
                    __threadfence();
                    done = atom_add_acq_rel_gpu(a.gcnt + tile, static_cast<unsigned>(nloc)) + nloc ==
                           static_cast<unsigned>(P.upt);
                }
                if (!__shfl_sync(0xffffffffu, done, 0)) continue;
                float *scr = reinterpret_cast<float *>(base + a.off_scr) + (lt == 0 ? 0 : static_cast<size_t>(P.upt) * w);
                for (int e = lane; e < P.upt * static_cast<int>(w); e += 32) scr[e] = __ldcg(gp + e);
                if (lane == 0) a.gcnt[tile] = 0u;
                __syncwarp();
                tile_sums = scr;
            } else if (split) {
                tile_sums = part_b + static_cast<size_t>(tb - u0) * M * kTileRows;
            }

            // ---- the tile's last unit: fold its segment sums with the pairwise
            // tree and store h (phase A) or y (phase B).  A tile's units are
            // consecutive in tile-major order, `count` apart in segment-major.
            const int r = lane >> 4;            // activation rows r, r + 2, ... of the tile's 16 outputs
            const int rr16 = lane & 15;         // output row of the tile
            const int row = tile * kTileRows + rr16;
            const bool tmaj = in_a || BO;
            const size_t ustride = static_cast<size_t>(tmaj ? 1 : P.count) * M * kTileRows;
            float *pt = (tile_sums != nullptr ? tile_sums
                                              : (in_a ? part_a : part_b) + static_cast<size_t>(lt) * (tmaj ? P.upt : 1) * M * kTileRows) +
                        r * kTileRows + rr16;
            for (int k2 = 0; 2 * k2 < M; ++k2) {
                const int ra = r + 2 * k2;
                const bool act = ra < M;
                float *pr = pt + 2 * k2 * kTileRows;
                if (in_a) {
                    uint16_t hv = 0;
                    if (act) {
                        const float gv = fold_tree(pr, P.nseg, static_cast<int>(ustride));
                        const float uv = fold_tree(pr + P.nseg * ustride, P.nseg, static_cast<int>(ustride));
                        hv = f32_to_bf16_bits(__fmul_rn(tq_silu(gv), uv));
                        if (row < P.n) a.h[static_cast<size_t>(ra) * P.n + row] = hv;
                    }
                    if (a.rotate_h) {
                        // the transform's spans 1, 2, 4, 8 stay inside the
                        // tile's 16 rows (lanes of one half-warp): apply them
                        // here, for the block's rotator to finish
                        float pv = bf16_bits_to_f32(hv);
#pragma unroll
                        for (int sp = 1; sp < kTileRows; sp <<= 1) {
                            const float other = __shfl_xor_sync(0xffffffffu, pv, sp);
                            // lower row: rn(a + b) = fma(+1, a, b); upper row:
                            // rn(b - a) = fma(-1, a, b) (the product is exact)
                            pv = __fmaf_rn((rr16 & sp) ? -1.0f : 1.0f, pv, other);
                        }
                        const int e = (tile % kTilesPerHBlock) * kTileRows + rr16;
                        if (act)
                            a.hp[static_cast<size_t>(ra) * P.n + (tile / kTilesPerHBlock) * kBlock + 4 * (e & 31) + (e >> 5)] = pv;
                    }
                } else if (act) {
                    const float yv = fold_tree(pr, P.nseg, static_cast<int>(ustride));
                    if (row < P.n) a.y[static_cast<size_t>(ra) * P.n + row] = yv;
                }
            }
            if (in_a && a.rotate_h) {
                // publish the tile's rows of h and hp: an acquire-release add
                // of its rows to the block's count (its release is cumulative
                // over the warp's stores, ordered before it by __syncwarp).  The add that completes the block
                // makes this warp the block's rotator; it acquires the other
                // tiles' rows and rotates at once.  Only this warp waits; the
                // others keep claiming units.
                __syncwarp();
                int completes = 0;
                if (lane == 0) {
                    const unsigned rows = static_cast<unsigned>(min(kTileRows, P.n - tile * kTileRows));
                    completes = atom_add_acq_rel_gpu(&a.hcount[tile / kTilesPerHBlock], rows) + rows ==
                                static_cast<unsigned>(kBlock);
                }
                if (__shfl_sync(0xffffffffu, completes, 0)) rotate_h_block<FMT, M>(a, P.n, tile / kTilesPerHBlock, lane);
            }
        }
    }

    if (bad != 0u && lane == 0 && a.err != nullptr) atomicOr(a.err, bad);
}

}  // namespace tq
