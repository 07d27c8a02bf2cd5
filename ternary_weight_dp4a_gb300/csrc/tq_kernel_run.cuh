// tq_kernel_run.cuh -- launch of one instantiation of the persistent kernel
// (programmatic dependent launch; cooperative when its phases wait on one
// another).  Included by the two translation units that instantiate the
// kernel: launches with phase A (tq_kernel.cu) and phase-B-only launches
// (tq_kernel_b.cu), so each compiles half of the instantiations.
#pragma once

#include <mutex>

#include "tq_kernel.cuh"

namespace tq {

constexpr int kMaxDev = 64;

template <int FMT, int M, bool BO>
cudaError_t launch_t(const KArgs &a, int grid, size_t bytes, bool coop, cudaStream_t stream) {
    auto kernel = tq_kernel<FMT, M, BO>;
    // the attribute is raised once per device, under a lock, to the largest
    // size any plan can ask for, so concurrent first calls cannot lower it
    static std::mutex mu;
    static bool configured[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= kMaxDev || !configured[dev]) {
            int optin = 0;
            if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
                return e;
            if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - 2048)) !=
                cudaSuccess)
                return e;
            if (dev < kMaxDev) configured[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (coop) {
        // phase B waits on blocks of h rotated by other CTAs: every CTA
        // must be resident at once
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na].val.cooperative = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess && coop) {
        // a driver that refuses the two attributes together: keep the
        // co-residency guarantee, drop the overlap with the previous launch
        (void)cudaGetLastError();
        cfg.attrs = attr + 1;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel, a);
    }
    return e;
}

// Phase-B-only launches (defined in tq_kernel_b.cu): fmt and m select the
// instantiation; never cooperative (no CTA waits on another).
cudaError_t launch_b_only(const KArgs &a, int fmt, int m, int grid, size_t bytes, cudaStream_t stream);

}  // namespace tq
