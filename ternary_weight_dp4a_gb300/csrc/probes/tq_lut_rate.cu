// tq_lut_rate.cu -- the inner loop of a 1-bit dot product (weights +1/-1,
// int8 activations) three ways, timed on every SM:
//   dp4a : the library's 1-bit core: per 32 weights one code word, then for
//          each bit position s a shift and mask picks bits s, 8+s, 16+s, 24+s
//          as bytes 0/1 and one dp4a meets the activation word that holds
//          those four weights (d = 2 sum(b q) - sum(q));
//   lut4 : a lookup table per group of 4 activations: 16 entries, the sum of
//          +-q for every sign pattern (int16); per 4 weights one nibble of the
//          code word indexes the table and one add accumulates;
//   lut8 : the same with groups of 8 activations (256 entries per group).
// The tables are built from the activations in shared memory; the codes sit
// row-interleaved (word i of rows 0..31 consecutive), so each lane of a warp
// owns one weight row and every code load is one conflict-free wavefront.
// The decision it informs: whether a lookup-table kernel beats the dp4a core
// on weights per cycle (bonsai-edge-serve README, kernels section, proposes
// one for 1-bit weights on the CPU).
//
// One CTA of 16 warps per SM, K = 1024 weights per row, 8 code tiles of 32
// rows cycled over 200 repetitions; each mode's sums are checked against a
// host computation.  All indexing stays inside the shared arrays (nibble <
// 16, byte < 256, word < 32 per row).  Build: nvcc -gencode
// arch=compute_103a,code=sm_103a -O3 -o tq_lut_rate tq_lut_rate.cu
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include <cuda_runtime.h>

#define CK(x)                                                                                \
    do {                                                                                     \
        cudaError_t e_ = (x);                                                                \
        if (e_ != cudaSuccess) {                                                             \
            printf("CUDA %s at %d: %s\n", #x, __LINE__, cudaGetErrorString(e_));             \
            exit(1);                                                                         \
        }                                                                                    \
    } while (0)

constexpr int kK = 1024;                 // weights per row
constexpr int kWords = kK / 32;          // code words per row
constexpr int kTiles = 8;                // code tiles of 32 rows
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kReps = 200;

// shared-memory layout (bytes)
constexpr int kCodesBytes = kTiles * kWords * 32 * 4;   // 32 KB
constexpr int kActBytes = kK;                           // staged int8 activations
constexpr int kT4Bytes = (kK / 4) * 16 * 2;             // 8 KB
constexpr int kT8Bytes = (kK / 8) * 256 * 2;            // 64 KB
constexpr int kSmem = kCodesBytes + kActBytes + kT4Bytes + kT8Bytes;

__host__ __device__ inline int8_t act_value(int e) { return static_cast<int8_t>((e * 37 + 11) % 255 - 127); }
__host__ __device__ inline uint32_t code_word(int tile, int row, int i) {
    uint32_t x = static_cast<uint32_t>(tile * 7919 + row * 104729 + i * 1299709) ^ 0x9e3779b9u;
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) lut_rate(int *out, long long *cycles) {
    extern __shared__ __align__(16) uint8_t sm[];
    uint32_t *codes = reinterpret_cast<uint32_t *>(sm);
    int8_t *act = reinterpret_cast<int8_t *>(sm + kCodesBytes);
    int16_t *t4 = reinterpret_cast<int16_t *>(sm + kCodesBytes + kActBytes);
    int16_t *t8 = reinterpret_cast<int16_t *>(sm + kCodesBytes + kActBytes + kT4Bytes);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // codes: tile t, word i, row r at (t * kWords + i) * 32 + r
    for (int x = tid; x < kTiles * kWords * 32; x += kThreads) {
        const int r = x & 31, i = (x >> 5) % kWords, t = x / (32 * kWords);
        codes[x] = code_word(t, r, i);
    }
    // activations staged for the dp4a core: byte 4s + k of group i holds
    // weight 32 i + 8 k + s
    for (int e = tid; e < kK; e += kThreads) {
        const int i = e >> 5, w = e & 31, k = w >> 3, s = w & 7;
        act[32 * i + 4 * s + k] = act_value(e);
    }
    for (int x = tid; x < (kK / 4) * 16; x += kThreads) {
        const int j = x >> 4, idx = x & 15;
        int v = 0;
        for (int t = 0; t < 4; ++t) v += ((idx >> t) & 1) ? act_value(4 * j + t) : -act_value(4 * j + t);
        t4[x] = static_cast<int16_t>(v);
    }
    for (int x = tid; x < (kK / 8) * 256; x += kThreads) {
        const int j = x >> 8, idx = x & 255;
        int v = 0;
        for (int t = 0; t < 8; ++t) v += ((idx >> t) & 1) ? act_value(8 * j + t) : -act_value(8 * j + t);
        t8[x] = static_cast<int16_t>(v);
    }
    int sumq = 0;
    for (int e = 0; e < kK; ++e) sumq += act_value(e);
    __syncthreads();

    const long long c0 = clock64();
    int total = 0;
#pragma unroll 1
    for (int rep = 0; rep < kReps; ++rep) {
        const uint32_t *cw = codes + ((warp + rep) % kTiles) * kWords * 32 + lane;
        int d;
        if (MODE == 0) {
            int d0 = 0, d1 = 0;
            const uint4 *a4 = reinterpret_cast<const uint4 *>(act);
#pragma unroll 4
            for (int i = 0; i < kWords; ++i) {
                const uint32_t w = cw[i * 32];
                const uint4 a0 = a4[2 * i], a1 = a4[2 * i + 1];
                const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int s = 0; s < 8; s += 2) {
                    d0 = __dp4a(static_cast<int>((w >> s) & 0x01010101u), static_cast<int>(av[s]), d0);
                    d1 = __dp4a(static_cast<int>((w >> (s + 1)) & 0x01010101u), static_cast<int>(av[s + 1]), d1);
                }
            }
            d = 2 * (d0 + d1) - sumq;
        } else if (MODE == 1) {
            int d0 = 0, d1 = 0;
#pragma unroll 4
            for (int i = 0; i < kWords; ++i) {
                const uint32_t w = cw[i * 32];
                const int16_t *tb = t4 + (8 * i) * 16;
#pragma unroll
                for (int t = 0; t < 8; t += 2) {
                    d0 += tb[t * 16 + ((w >> (4 * t)) & 15u)];
                    d1 += tb[(t + 1) * 16 + ((w >> (4 * t + 4)) & 15u)];
                }
            }
            d = d0 + d1;
        } else {
            int d0 = 0, d1 = 0;
#pragma unroll 4
            for (int i = 0; i < kWords; ++i) {
                const uint32_t w = cw[i * 32];
                const int16_t *tb = t8 + (4 * i) * 256;
                d0 += tb[(w & 255u)];
                d1 += tb[256 + ((w >> 8) & 255u)];
                d0 += tb[512 + ((w >> 16) & 255u)];
                d1 += tb[768 + (w >> 24)];
            }
            d = d0 + d1;
        }
        total += d;
    }
    const long long c1 = clock64();
    out[blockIdx.x * kThreads + tid] = total;
    if (tid == 0) cycles[blockIdx.x] = c1 - c0;
}

int main() {
    int dev = 0, sms = 0;
    CK(cudaSetDevice(dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    // expected sums (identical on every CTA): the plain dot of each tile row,
    // summed over the repetitions' tiles
    std::vector<long long> dot(kTiles * 32, 0);
    for (int tile = 0; tile < kTiles; ++tile)
        for (int row = 0; row < 32; ++row)
            for (int e = 0; e < kK; ++e) {
                const uint32_t w = code_word(tile, row, e >> 5);
                const int q = act_value(e);
                dot[tile * 32 + row] += ((w >> (e & 31)) & 1u) ? q : -q;
            }
    std::vector<int> expect(kThreads);
    for (int warp = 0; warp < kWarps; ++warp)
        for (int lane = 0; lane < 32; ++lane) {
            long long tot = 0;
            for (int rep = 0; rep < kReps; ++rep) tot += dot[((warp + rep) % kTiles) * 32 + lane];
            expect[warp * 32 + lane] = static_cast<int>(tot);
        }
    int *d_out = nullptr;
    long long *d_cyc = nullptr;
    CK(cudaMalloc(&d_out, sizeof(int) * sms * kThreads));
    CK(cudaMalloc(&d_cyc, sizeof(long long) * sms));
    CK(cudaFuncSetAttribute(lut_rate<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
    CK(cudaFuncSetAttribute(lut_rate<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
    CK(cudaFuncSetAttribute(lut_rate<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
    const char *names[3] = {"dp4a", "lut4", "lut8"};
    const double weights_per_cta = static_cast<double>(kWarps) * 32 * kK * kReps;
    printf("1-bit inner loop, %d SMs, one %d-thread CTA each, K = %d, %d reps\n", sms, kThreads, kK, kReps);
    printf("%-6s %10s %14s %18s %8s\n", "mode", "ms", "Gweights/s", "weights/cycle/SM", "check");
    for (int mode = 0; mode < 3; ++mode) {
        cudaEvent_t e0, e1;
        CK(cudaEventCreate(&e0));
        CK(cudaEventCreate(&e1));
        float best = 1e30f;
        double cyc_best = 0;
        bool ok = true;
        for (int it = 0; it < 4; ++it) {
            CK(cudaEventRecord(e0));
            if (mode == 0) lut_rate<0><<<sms, kThreads, kSmem>>>(d_out, d_cyc);
            if (mode == 1) lut_rate<1><<<sms, kThreads, kSmem>>>(d_out, d_cyc);
            if (mode == 2) lut_rate<2><<<sms, kThreads, kSmem>>>(d_out, d_cyc);
            CK(cudaGetLastError());
            CK(cudaEventRecord(e1));
            CK(cudaEventSynchronize(e1));
            float ms = 0;
            CK(cudaEventElapsedTime(&ms, e0, e1));
            std::vector<int> out(static_cast<size_t>(sms) * kThreads);
            std::vector<long long> cyc(sms);
            CK(cudaMemcpy(out.data(), d_out, sizeof(int) * out.size(), cudaMemcpyDeviceToHost));
            CK(cudaMemcpy(cyc.data(), d_cyc, sizeof(long long) * sms, cudaMemcpyDeviceToHost));
            for (int c = 0; c < sms; ++c)
                for (int t = 0; t < kThreads; ++t)
                    if (out[static_cast<size_t>(c) * kThreads + t] != expect[t]) ok = false;
            double cavg = 0;
            for (int c = 0; c < sms; ++c) cavg += static_cast<double>(cyc[c]) / sms;
            if (it > 0 && ms < best) {
                best = ms;
                cyc_best = cavg;
            }
        }
        printf("%-6s %10.4f %14.1f %18.1f %8s\n", names[mode], best, weights_per_cta * sms / (best * 1e-3) / 1e9,
               weights_per_cta / cyc_best, ok ? "ok" : "FAIL");
        CK(cudaEventDestroy(e0));
        CK(cudaEventDestroy(e1));
        if (!ok) return 1;
    }
    CK(cudaFree(d_out));
    CK(cudaFree(d_cyc));
    return 0;
}
