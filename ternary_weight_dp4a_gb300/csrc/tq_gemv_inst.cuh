// tq_gemv_inst.cuh -- instantiates gemv_kernel<FMT, M, NW> for M = 1..8 and
// NW = 1, 2 and dispatches on the runtime row count.  Included once per format
// so the two formats compile in parallel.
#pragma once

#include <atomic>
#include <cstdint>

#include "tq_launch.h"

namespace tq {

template <int FMT, int M, int NW>
static cudaError_t launch_one(const GemvArgs &a, cudaStream_t stream) {
    const int nb = a.k / kBlock;
    const size_t smem = gemv_smem_bytes(FMT, M, nb);
    auto kernel = gemv_kernel<FMT, M, NW>;
    if (smem > 48 * 1024) {
        // opt in to large shared memory once per device for this instantiation
        static std::atomic<uint64_t> configured{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
        if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(max_smem_optin()));
            if (e != cudaSuccess) return e;
            configured.fetch_or(bit, std::memory_order_acq_rel);
        }
    }
    const unsigned grid = static_cast<unsigned>((a.n + kTilesPerCta - 1) / kTilesPerCta);
    kernel<<<grid, kGemvThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int FMT, int NW>
static cudaError_t dispatch_m(const GemvArgs &a, int m, cudaStream_t stream) {
    switch (m) {
        case 1: return launch_one<FMT, 1, NW>(a, stream);
        case 2: return launch_one<FMT, 2, NW>(a, stream);
        case 3: return launch_one<FMT, 3, NW>(a, stream);
        case 4: return launch_one<FMT, 4, NW>(a, stream);
        case 5: return launch_one<FMT, 5, NW>(a, stream);
        case 6: return launch_one<FMT, 6, NW>(a, stream);
        case 7: return launch_one<FMT, 7, NW>(a, stream);
        case 8: return launch_one<FMT, 8, NW>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int FMT>
static cudaError_t dispatch_gemv(const GemvArgs &a, int m, int nw, cudaStream_t stream) {
    return nw == 1 ? dispatch_m<FMT, 1>(a, m, stream) : dispatch_m<FMT, 2>(a, m, stream);
}

}  // namespace tq
