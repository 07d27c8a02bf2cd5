// tq_ffn_fused.cuh -- the whole decode FFN step (or a stack of steps) as one
// persistent kernel: one CTA per SM, a producer warp streaming weights through
// a shared-memory ring with bulk copies, consumer warps computing.
//
// Per layer:
//   phase A  rotate + quantise the layer input in every CTA (x for layer 0, the
//            RMS-normalised previous output after that); gate/up GEMVs over
//            this CTA's output range; h = bf16(silu(g) * u); the last CTA to
//            finish a 128-block of h rotates and quantises it.
//   barrier  all CTAs (bounded spin on a workspace counter)
//   phase B  stage qh; down GEMV over this CTA's output range -> y.
//   barrier  (stacks only: y must be complete before the next normalisation)
// The producer never waits on a barrier: weights do not depend on activations,
// so it keeps the ring full of the next phase's rows while consumers wait.
//
// Consumers split work into (output, block) tasks balanced over all lanes:
// a task computes the exact int32 block dot(s) and t = (float)d * (sw * s)
// into shared memory; then 8 fold lanes per output add the t's of blocks
// p, p+8, ... in ascending order and meet in the xor tree (1, 2, 4) -- the
// documented order, so results equal the single-step kernels bit for bit.
#pragma once

#include "tq_device.cuh"
#include "tq_gemv.cuh"
#include "tq_rotq.cuh"

namespace tq {

constexpr int kFusedMaxLayers = 64;
constexpr int kFusedConsumerWarps = 15;
constexpr int kFusedThreads = 32 * (kFusedConsumerWarps + 1);
constexpr int kFusedConsumers = 32 * kFusedConsumerWarps;
constexpr int kFusedStages = 4;
constexpr int kFusedSlotBytes = 33 * 1024;          // one ring stage

struct FfnLayerPtrs {
    const uint8_t *codes[3];     // gate, up, down
    const uint16_t *scales[3];
};

struct FfnFusedArgs {
    FfnLayerPtrs layer[kFusedMaxLayers];
    int num_layers;
    int hidden, inter;
    float eps;
    int input_is_y;              // layer 0 input: 0 = bf16 x, 1 = rmsnorm(y_in)
    const uint16_t *x;           // [M][hidden] bf16
    const float *y_in;           // [M][hidden] (input_is_y)
    float *y;                    // [M][hidden] output of the last layer
    float *ybuf;                 // [M][hidden] outputs of the other layers
    int8_t *qx;                  // [M][hidden] the layer input's int8 codes (CTA 0 writes)
    float *sx;                   // [M][hidden/128]
    uint16_t *h;                 // [M][inter]
    int8_t *qh;                  // [M][inter]
    float *sh;                   // [M][inter/128]
    unsigned *counters;          // [inter/128], zero on entry and exit
    unsigned *gbar;              // grid barrier {count, generation}
    unsigned *err;
};

// outputs per ring stage (phase A counts an output's gate and up rows)
__host__ __device__ inline int fused_rows_per_stage(int mats, int k, int fmt) {
    const int nb = k / kBlock;
    const int row = nb * (fmt == 0 ? 32 : 16) + nb * 2;        // codes + scales
    int r = kFusedSlotBytes / (mats * row);
    // at most 8 fold lanes per output-row within the consumers
    const int cap = kFusedConsumers / (8 * mats);
    return r < cap ? r : cap;
}

__host__ __device__ inline size_t fused_act_bytes(int m, int k) {
    return (static_cast<size_t>(m) * (k / kBlock) * (kActStride + 8) + 15) / 16 * 16;
}

// bytes of dynamic shared memory the fused kernel needs (m rows)
__host__ inline size_t fused_smem_bytes(int m, int hidden, int inter, int fmt) {
    const int ra = fused_rows_per_stage(2, hidden, fmt), rb = fused_rows_per_stage(1, inter, fmt);
    const size_t ta = static_cast<size_t>(ra) * 2 * (hidden / kBlock), tb = static_cast<size_t>(rb) * (inter / kBlock);
    const size_t tbuf = static_cast<size_t>(2) * m * (ta > tb ? ta : tb) * 4;
    return 1024 + static_cast<size_t>(kFusedStages) * kFusedSlotBytes + fused_act_bytes(m, hidden) +
           fused_act_bytes(m, inter) + tbuf + 16;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier among gridDim.x co-resident CTAs, run by one thread per
// CTA between CTA-level barriers.  Bounded: after kWaitBudgetCycles it sets
// err bit 16 and returns false instead of waiting further.
__device__ __forceinline__ bool grid_barrier(unsigned *gbar, unsigned *err) {
    const unsigned gen = ld_acquire_u32(gbar + 1);
    __threadfence();
    const unsigned ticket = atomicAdd(gbar, 1u);
    if (ticket == gridDim.x - 1) {
        atomicExch(gbar, 0u);
        __threadfence();
        atomicAdd(gbar + 1, 1u);
        return true;
    }
    const long long t0 = clock64();
    while (ld_acquire_u32(gbar + 1) == gen) {
        if (clock64() - t0 > kWaitBudgetCycles) {
            if (err != nullptr) atomicOr(err, 16u);
            return false;
        }
        __nanosleep(64);
    }
    __threadfence();
    return true;
}

// Staged (permuted, padded) position of element e (0..127) of a block.
template <int FMT>
__device__ __forceinline__ int staged_pos(int e) {
    if (FMT == 0) {
        // per 16 elements: evens then odds
        const int g = e >> 4, r = e & 15;
        return 16 * g + (r >> 1) + 8 * (r & 1);
    }
    // per 32 elements: position 4*s + i holds element 8*i + s
    const int g = e >> 5, r = e & 31;
    return 32 * g + 4 * (r & 7) + (r >> 3);
}

// Rotate + quantise M rows of a k-vector into the staged layout (consumer
// warps; warp w handles blocks w, w+NW, ...).  Input element i of row mm is
// in_fn(mm, i) (a bf16 value as float).
template <int FMT, int M, typename InFn>
__device__ __forceinline__ void rotq_stage(InFn in_fn, int k, uint8_t *act, float *sact, int *cmag,
                                           int warp, int lane, int nwarps, int8_t *q_out = nullptr,
                                           float *s_out = nullptr) {
    const int nb = k / kBlock;
    for (int t = warp; t < M * nb; t += nwarps) {
        const int mm = t / nb, b = t % nb;
        float v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = in_fn(mm, b * kBlock + lane + 32 * c);
        wht128_warp(v, lane);
        int8_t q[4];
        const float s = quant_block_warp(v, q);
        uint8_t *dst = act + (mm * nb + b) * kActStride;
        int part = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            dst[staged_pos<FMT>(lane + 32 * c)] = static_cast<uint8_t>(q[c]);
            part += q[c];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) {
            sact[mm * nb + b] = s;
            cmag[mm * nb + b] = 0x4b400000 - part;
        }
        if (q_out != nullptr) {           // also the plain layout, for inspection
#pragma unroll
            for (int c = 0; c < 4; ++c) q_out[static_cast<size_t>(mm) * k + b * kBlock + lane + 32 * c] = q[c];
            if (lane == 0) s_out[mm * nb + b] = s;
        }
    }
}

// Stage an already quantised activation (q int8 [M][k], s [M][k/128]) from
// global memory into the staged layout (consumer threads).
template <int FMT, int M>
__device__ __forceinline__ void stage_q(const int8_t *__restrict__ q, const float *__restrict__ s, int k,
                                        uint8_t *act, float *sact, int *cmag, int tid, int nthr) {
    const int nb = k / kBlock;
    for (int i = tid; i < M * nb; i += nthr) sact[i] = __ldcg(s + i);
    // one 128-element block per iteration: 8 x 16 bytes
    for (int t = tid; t < M * nb * 4; t += nthr) {
        const int blk = t >> 2, part = t & 3;      // 32-byte quarter of the block
        const int mm = blk / nb, b = blk % nb;
        const uint4 *src = reinterpret_cast<const uint4 *>(q + static_cast<size_t>(mm) * k + b * kBlock + 32 * part);
        const uint4 lo = __ldcg(src), hi = __ldcg(src + 1);
        const uint32_t X[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        uint8_t *dst = act + blk * kActStride + 32 * part;
        if (FMT == 0) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint4 o;
                o.x = prmt(X[4 * h2 + 0], X[4 * h2 + 1], 0x6420u);
                o.y = prmt(X[4 * h2 + 2], X[4 * h2 + 3], 0x6420u);
                o.z = prmt(X[4 * h2 + 0], X[4 * h2 + 1], 0x7531u);
                o.w = prmt(X[4 * h2 + 2], X[4 * h2 + 3], 0x7531u);
                *reinterpret_cast<uint4 *>(dst + 16 * h2) = o;
            }
        } else {
            uint32_t o[8];
#pragma unroll
            for (int sl = 0; sl < 8; ++sl) {
                const int j = sl >> 2, by = sl & 3;
                const uint32_t sel = static_cast<uint32_t>(by) | (static_cast<uint32_t>(by + 4) << 4);
                o[sl] = prmt(prmt(X[j], X[j + 2], sel), prmt(X[j + 4], X[j + 6], sel), 0x5410u);
            }
            reinterpret_cast<uint4 *>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<uint4 *>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
        int sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) sum = __dp4a(static_cast<int>(X[j]), 0x01010101, sum);
        // the four quarters of a block are 4 consecutive lanes: add them up
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (part == 0) cmag[blk] = 0x4b400000 - sum;
    }
}

template <int FMT, int M>
__global__ void __launch_bounds__(kFusedThreads, 1) ffn_fused_kernel(const __grid_constant__ FfnFusedArgs a) {
    constexpr int BB = FmtTraits<FMT>::kBlockBytes;
    constexpr int S = kFusedStages;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[S];
    __shared__ __align__(8) uint64_t empty_bar[S];
    __shared__ int s_last[2];
    __shared__ float s_warp[kFusedConsumerWarps];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hidden = a.hidden, inter = a.inter;
    const int nbh = hidden / kBlock, nbi = inter / kBlock;
    const int G = gridDim.x, c = blockIdx.x;
    const int a_beg = static_cast<int>(static_cast<long long>(inter) * c / G);
    const int a_end = static_cast<int>(static_cast<long long>(inter) * (c + 1) / G);
    const int b_beg = static_cast<int>(static_cast<long long>(hidden) * c / G);
    const int b_end = static_cast<int>(static_cast<long long>(hidden) * (c + 1) / G);
    const int ra = fused_rows_per_stage(2, hidden, FMT), rb = fused_rows_per_stage(1, inter, FMT);
    const int sta = (a_end - a_beg + ra - 1) / ra, stb = (b_end - b_beg + rb - 1) / rb;
    const size_t rowa = static_cast<size_t>(nbh) * BB, rowb = static_cast<size_t>(nbi) * BB;

    uint8_t *ring = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
    uint8_t *xact = ring + static_cast<size_t>(S) * kFusedSlotBytes;
    float *xs = reinterpret_cast<float *>(xact + static_cast<size_t>(M) * nbh * kActStride);
    int *xc = reinterpret_cast<int *>(xs + M * nbh);
    uint8_t *hact = xact + fused_act_bytes(M, hidden);
    float *hs = reinterpret_cast<float *>(hact + static_cast<size_t>(M) * nbi * kActStride);
    int *hc = reinterpret_cast<int *>(hs + M * nbi);
    float *tbuf = reinterpret_cast<float *>(hact + fused_act_bytes(M, inter));
    const int tstride = M * (ra * 2 * nbh > rb * nbi ? ra * 2 * nbh : rb * nbi);   // floats per buffer

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), kFusedConsumerWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_launch_dependents();

    const int per_layer = sta + stb;
    const int total = a.num_layers * per_layer;

    if (warp == kFusedConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            for (int st = 0; st < total && ok; ++st) {
                const int slot = st % S;
                if (st >= S && !(ok = mbar_wait(smem_u32(&empty_bar[slot]), ((st / S) - 1) & 1))) break;
                const int l = st / per_layer, js = st % per_layer;
                const FfnLayerPtrs &L = a.layer[l];
                const uint32_t full = smem_u32(&full_bar[slot]);
                uint8_t *dst = ring + static_cast<size_t>(slot) * kFusedSlotBytes;
                if (js < sta) {
                    const int o0 = a_beg + js * ra, cnt = min(ra, a_end - o0);
                    const uint32_t cb = static_cast<uint32_t>(cnt * rowa), sb = static_cast<uint32_t>(cnt * nbh * 2);
                    mbar_arrive_expect_tx(full, 2 * (cb + sb));
                    bulk_copy_g2s(smem_u32(dst), L.codes[0] + o0 * rowa, cb, full);
                    bulk_copy_g2s(smem_u32(dst + ra * rowa), L.codes[1] + o0 * rowa, cb, full);
                    bulk_copy_g2s(smem_u32(dst + 2 * ra * rowa), L.scales[0] + static_cast<size_t>(o0) * nbh, sb, full);
                    bulk_copy_g2s(smem_u32(dst + 2 * ra * rowa + ra * nbh * 2),
                                  L.scales[1] + static_cast<size_t>(o0) * nbh, sb, full);
                } else {
                    const int o0 = b_beg + (js - sta) * rb, cnt = min(rb, b_end - o0);
                    const uint32_t cb = static_cast<uint32_t>(cnt * rowb), sb = static_cast<uint32_t>(cnt * nbi * 2);
                    mbar_arrive_expect_tx(full, cb + sb);
                    bulk_copy_g2s(smem_u32(dst), L.codes[2] + o0 * rowb, cb, full);
                    bulk_copy_g2s(smem_u32(dst + rb * rowb), L.scales[2] + static_cast<size_t>(o0) * nbi, sb, full);
                }
                issued = st + 1;
            }
            if (!ok && a.err != nullptr) atomicOr(a.err, 1u);
            for (int st = issued > S ? issued - S : 0; st < issued; ++st)
                if (!mbar_wait(smem_u32(&full_bar[st % S]), (st / S) & 1) && a.err != nullptr)
                    atomicOr(a.err, 2u);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int tid = threadIdx.x;                 // 0 .. kFusedConsumers-1
    bool ok = true;
    int st = 0;
    for (int l = 0; l < a.num_layers; ++l) {
        const FfnLayerPtrs &L = a.layer[l];
        // ---- layer input: rotate + quantise into xact
        if (l == 0 && !a.input_is_y) {
            pdl_wait();
            const uint16_t *x = a.x;
            rotq_stage<FMT, M>([&](int mm, int i) { return bf16_bits_to_f32(x[static_cast<size_t>(mm) * hidden + i]); },
                               hidden, xact, xs, xc, warp, lane, kFusedConsumerWarps,
                               c == 0 ? a.qx : nullptr, a.sx);
        } else {
            if (l == 0) pdl_wait();
            const float *yin = l == 0 ? a.y_in : a.ybuf;
            // RMS norm of each row: the documented 256-partial order (threads 0..255)
            for (int mm = 0; mm < M; ++mm) {
                const float *yr = yin + static_cast<size_t>(mm) * hidden;
                float acc = 0.0f;
                if (tid < 256)
                    for (int i = tid; i < hidden; i += 256) {
                        const float v = __ldcg(yr + i);
                        acc = __fadd_rn(acc, __fmul_rn(v, v));
                    }
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
                if (lane == 0 && warp < 8) s_warp[warp] = acc;
                named_barrier(1, kFusedConsumers);
                const float w01 = __fadd_rn(s_warp[0], s_warp[1]), w23 = __fadd_rn(s_warp[2], s_warp[3]);
                const float w45 = __fadd_rn(s_warp[4], s_warp[5]), w67 = __fadd_rn(s_warp[6], s_warp[7]);
                const float ss = __fadd_rn(__fadd_rn(w01, w23), __fadd_rn(w45, w67));
                const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(hidden)), a.eps)));
                named_barrier(1, kFusedConsumers);
                // rows are independent: rotate this row now
                rotq_stage<FMT, 1>([&](int, int i) {
                    return bf16_bits_to_f32(f32_to_bf16_bits(__fmul_rn(__ldcg(yr + i), inv)));
                }, hidden, xact + static_cast<size_t>(mm) * nbh * kActStride, xs + mm * nbh, xc + mm * nbh,
                   warp, lane, kFusedConsumerWarps, c == 0 ? a.qx + static_cast<size_t>(mm) * hidden : nullptr,
                   a.sx + mm * nbh);
            }
        }
        named_barrier(1, kFusedConsumers);

        // ---- phase A: gate/up
        for (int js = 0; js < sta; ++js, ++st) {
            const int slot = st % S;
            if (ok && !mbar_wait(smem_u32(&full_bar[slot]), (st / S) & 1)) ok = false;
            const uint8_t *stage = ring + static_cast<size_t>(slot) * kFusedSlotBytes;
            const int o0 = a_beg + js * ra, cnt = min(ra, a_end - o0);
            float *tb = tbuf + (st & 1) * tstride;        // [2][ra][nbh]
            const __half *sc0 = reinterpret_cast<const __half *>(stage + 2 * ra * rowa);
            const __half *sc1 = sc0 + ra * nbh;
            for (int task = tid; ok && task < cnt * nbh; task += kFusedConsumers) {
                const int o = task / nbh, b = task % nbh;
                uint32_t w[1][2][8];
                const uint8_t *const act_b[1] = {xact + b * kActStride};
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint8_t *seg = stage + (r * ra + o) * rowa + b * BB;
                    const uint4 x0 = *reinterpret_cast<const uint4 *>(seg);
                    w[0][r][0] = x0.x; w[0][r][1] = x0.y; w[0][r][2] = x0.z; w[0][r][3] = x0.w;
                    if constexpr (FMT == 0) {
                        const uint4 x1 = *reinterpret_cast<const uint4 *>(seg + 16);
                        w[0][r][4] = x1.x; w[0][r][5] = x1.y; w[0][r][6] = x1.z; w[0][r][7] = x1.w;
                    } else {
                        w[0][r][4] = w[0][r][5] = w[0][r][6] = w[0][r][7] = 0u;
                    }
                }
                int dot[1][2][M];
                block_dots<FMT, M, 1, 2>(w, act_b, nbh, dot);
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    const float sa = xs[mm * nbh + b];
                    const int cm = xc[mm * nbh + b];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int raw = FMT == 0 ? dot[0][r][mm] : 2 * dot[0][r][mm];
                        const float ws = __half2float((r == 0 ? sc0 : sc1)[o * nbh + b]);
                        tb[((mm * 2 + r) * ra + o) * nbh + b] =
                            __fmul_rn(int_to_float_exact(raw, cm), __fmul_rn(ws, sa));
                    }
                }
            }
            // the stage's codes are consumed: release the slot, then fold
            named_barrier(1, kFusedConsumers);
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
            // fold lane f: output o = f / 16, matrix r = (f / 8) & 1, chain p = f & 7
            if (warp < (16 * ra + 31) / 32) {            // whole warps: the tree shuffles
                const int o = tid >> 4, r = (tid >> 3) & 1, p = tid & 7;
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    float acc = 0.0f;
                    if (o < cnt)
                        for (int b = p; b < nbh; b += 8)
                            acc = __fadd_rn(acc, tb[((mm * 2 + r) * ra + o) * nbh + b]);
                    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 1));
                    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 2));
                    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 4));
                    const float up = __shfl_xor_sync(0xffffffffu, acc, 8);   // the up row of o
                    if (o < cnt && r == 0 && p == 0) {
                        const float hv = __fmul_rn(tq_silu(acc), up);
                        a.h[static_cast<size_t>(mm) * inter + o0 + o] = f32_to_bf16_bits(hv);
                    }
                }
            }
        }
        // ---- h blocks this CTA completed last: rotate + quantise them
        named_barrier(1, kFusedConsumers);
        {
            const int hb0 = a_beg / kBlock, hb1 = (a_end - 1) / kBlock;
            if (tid == 0) {
                __threadfence();
                for (int j = 0; j < 2; ++j) {
                    const int hb = hb0 + j;
                    s_last[j] = 0;
                    if (hb > hb1 || a_end <= a_beg) continue;
                    const int lo = max(a_beg, hb * kBlock), hi = min(a_end, (hb + 1) * kBlock);
                    const unsigned add = static_cast<unsigned>(hi - lo);
                    const unsigned before = atomicAdd(&a.counters[hb], add);
                    if (before + add == static_cast<unsigned>(kBlock)) {
                        a.counters[hb] = 0u;
                        s_last[j] = 1;
                    }
                }
                __threadfence();
            }
            named_barrier(1, kFusedConsumers);
            for (int j = 0; j < 2; ++j) {
                if (!s_last[j]) continue;
                const int hb = hb0 + j;
                for (int mm = warp; mm < M; mm += kFusedConsumerWarps) {
                    const uint16_t *hrow = a.h + static_cast<size_t>(mm) * inter + hb * kBlock;
                    float v[4];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) v[cc] = bf16_bits_to_f32(__ldcg(hrow + lane + 32 * cc));
                    rotq_block_store(v, lane, a.qh + static_cast<size_t>(mm) * inter + hb * kBlock,
                                     a.sh + static_cast<size_t>(mm) * nbi + hb);
                }
            }
        }
        // ---- every CTA's h blocks are rotated
        named_barrier(1, kFusedConsumers);
        if (tid == 0) grid_barrier(a.gbar, a.err);
        named_barrier(1, kFusedConsumers);
        stage_q<FMT, M>(a.qh, a.sh, inter, hact, hs, hc, tid, kFusedConsumers);
        named_barrier(1, kFusedConsumers);

        // ---- phase B: down
        float *yout = l + 1 == a.num_layers ? a.y : a.ybuf;
        for (int js = 0; js < stb; ++js, ++st) {
            const int slot = st % S;
            if (ok && !mbar_wait(smem_u32(&full_bar[slot]), (st / S) & 1)) ok = false;
            const uint8_t *stage = ring + static_cast<size_t>(slot) * kFusedSlotBytes;
            const int o0 = b_beg + js * rb, cnt = min(rb, b_end - o0);
            float *tb = tbuf + (st & 1) * tstride;        // [M][rb][nbi]
            const __half *sc = reinterpret_cast<const __half *>(stage + rb * rowb);
            for (int task = tid; ok && task < cnt * nbi; task += kFusedConsumers) {
                const int o = task / nbi, b = task % nbi;
                uint32_t w[1][1][8];
                const uint8_t *const act_b[1] = {hact + b * kActStride};
                const uint8_t *seg = stage + o * rowb + b * BB;
                const uint4 x0 = *reinterpret_cast<const uint4 *>(seg);
                w[0][0][0] = x0.x; w[0][0][1] = x0.y; w[0][0][2] = x0.z; w[0][0][3] = x0.w;
                if constexpr (FMT == 0) {
                    const uint4 x1 = *reinterpret_cast<const uint4 *>(seg + 16);
                    w[0][0][4] = x1.x; w[0][0][5] = x1.y; w[0][0][6] = x1.z; w[0][0][7] = x1.w;
                } else {
                    w[0][0][4] = w[0][0][5] = w[0][0][6] = w[0][0][7] = 0u;
                }
                int dot[1][1][M];
                block_dots<FMT, M, 1, 1>(w, act_b, nbi, dot);
                const float ws = __half2float(sc[o * nbi + b]);
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    const int raw = FMT == 0 ? dot[0][0][mm] : 2 * dot[0][0][mm];
                    tb[(mm * rb + o) * nbi + b] =
                        __fmul_rn(int_to_float_exact(raw, hc[mm * nbi + b]), __fmul_rn(ws, hs[mm * nbi + b]));
                }
            }
            named_barrier(1, kFusedConsumers);
            if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
            if (warp < (8 * rb + 31) / 32) {             // whole warps: the tree shuffles
                const int o = tid >> 3, p = tid & 7;
#pragma unroll
                for (int mm = 0; mm < M; ++mm) {
                    float acc = 0.0f;
                    if (o < cnt)
                        for (int b = p; b < nbi; b += 8) acc = __fadd_rn(acc, tb[(mm * rb + o) * nbi + b]);
                    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 1));
                    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 2));
                    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 4));
                    if (o < cnt && p == 0) yout[static_cast<size_t>(mm) * hidden + o0 + o] = acc;
                }
            }
        }
        if (l + 1 < a.num_layers) {
            // the next layer normalises all of y
            __threadfence();
            named_barrier(1, kFusedConsumers);
            if (tid == 0) grid_barrier(a.gbar, a.err);
            named_barrier(1, kFusedConsumers);
        }
    }
    if (!ok && lane == 0 && a.err != nullptr) atomicOr(a.err, 4u);
}

}  // namespace tq
