// tq_gemv_inst.cuh -- instantiates gemv_kernel for M = 1..8 (plain and fused
// gate/up) and dispatches on the runtime row count.  Included once per format
// so the two formats compile in parallel.
#pragma once

#include <atomic>
#include <cstdint>

#include "tq_launch.h"
#include "tq_tmap.h"

namespace tq {

constexpr int kMaxDevices = 64;

template <int FMT, int M, bool GATEUP>
struct GemvShape {
    // consumer warps (tile = 4 * NCW outputs) and ring stages; CTAs stay small
    // enough for several to share an SM, so consecutive kernels overlap
    static constexpr int kNcw = 4;
    static constexpr int kStages = GATEUP ? 2 : 4;
};

// CTAs per launch: at most kCtasPerSm per SM, and no more than one per tile
constexpr int kCtasPerSm = 4;

inline int gemv_grid(int n, int tile) {
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        sms = 1;
    const int tiles = (n + tile - 1) / tile;
    return tiles < kCtasPerSm * sms ? tiles : kCtasPerSm * sms;
}

template <int FMT, int M, bool GATEUP>
size_t gemv_smem(int nb, int n) {
    using S = GemvShape<FMT, M, GATEUP>;
    const int outs = gemv_cta_outputs_max(n, gemv_grid(n, 4 * S::kNcw));
    return gemv_ring_bytes(FMT, GATEUP ? 2 : 1, S::kNcw, S::kStages) + gemv_act_bytes(M, nb) +
           gemv_scale_bytes(GATEUP ? 2 : 1, outs, nb);
}

template <int FMT, int M, bool GATEUP>
static cudaError_t launch_one(const GemvArgs &a_in, cudaStream_t stream) {
    using S = GemvShape<FMT, M, GATEUP>;
    GemvArgs a = a_in;
    const int nb = a.k / kBlock;
    {
        // tensor maps of the code matrices: box = 8 blocks (or the whole row) x tile rows
        constexpr int BB = FMT == 0 ? 32 : 16;
        const size_t row_bytes = static_cast<size_t>(nb) * BB;
        const uint32_t box_bytes = static_cast<uint32_t>(nb < kBlocksPerBox ? row_bytes : kBlocksPerBox * BB);
        const uint32_t box_rows = static_cast<uint32_t>(a.n < 4 * S::kNcw ? a.n : 4 * S::kNcw);
        for (int r = 0; r < (GATEUP ? 2 : 1); ++r) {
            const cudaError_t e = make_codes_tmap(&a.tmap[r], a.codes[r], a.n, row_bytes, box_bytes, box_rows);
            if (e != cudaSuccess) return e;
        }
    }
    const size_t smem = gemv_smem<FMT, M, GATEUP>(nb, a.n);
    auto kernel = gemv_kernel<FMT, M, GATEUP, S::kNcw, S::kStages>;
    if (smem + 1024 > 48 * 1024) {   // the static part (mbarriers, flags) counts too
        // opt in to this much dynamic shared memory (once per device and size
        // for this instantiation; the kernel's static shared memory comes on top)
        static std::atomic<int> configured[kMaxDevices] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const int want = static_cast<int>(smem);
        if (dev >= kMaxDevices || configured[dev].load(std::memory_order_acquire) < want) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
            if (e != cudaSuccess) return e;
            if (dev < kMaxDevices) {
                int cur = configured[dev].load(std::memory_order_acquire);
                while (cur < want && !configured[dev].compare_exchange_weak(cur, want)) {
                }
            }
        }
    }
    const unsigned grid = static_cast<unsigned>(gemv_grid(a.n, 4 * S::kNcw));
    return launch_pdl(kernel, dim3(grid), dim3(32 * (S::kNcw + 1)), smem, stream, a);
}

template <int FMT, bool GATEUP>
static cudaError_t dispatch_m(const GemvArgs &a, int m, cudaStream_t stream) {
    switch (m) {
        case 1: return launch_one<FMT, 1, GATEUP>(a, stream);
        case 2: return launch_one<FMT, 2, GATEUP>(a, stream);
        case 3: return launch_one<FMT, 3, GATEUP>(a, stream);
        case 4: return launch_one<FMT, 4, GATEUP>(a, stream);
        case 5: return launch_one<FMT, 5, GATEUP>(a, stream);
        case 6: return launch_one<FMT, 6, GATEUP>(a, stream);
        case 7: return launch_one<FMT, 7, GATEUP>(a, stream);
        case 8: return launch_one<FMT, 8, GATEUP>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int FMT>
static cudaError_t dispatch_gemv(const GemvArgs &a, int m, bool gateup, cudaStream_t stream) {
    return gateup ? dispatch_m<FMT, true>(a, m, stream) : dispatch_m<FMT, false>(a, m, stream);
}

}  // namespace tq
