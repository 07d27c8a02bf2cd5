// tq_ffn_fused.cu -- launch of the persistent fused FFN kernel.
#include <atomic>

#include "tq_ffn_fused.cuh"
#include "tq_fused_launch.h"
#include "tq_launch.h"

namespace tq {

namespace {

constexpr int kMaxDev = 64;

template <int FMT, int M>
cudaError_t launch_fused_t(const FfnFusedArgs &a, cudaStream_t stream) {
    auto kernel = ffn_fused_kernel<FMT, M>;
    const size_t smem = fused_smem_bytes(M, a.hidden, a.inter, FMT);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    static std::atomic<int> configured[kMaxDev] = {};
    if (dev >= kMaxDev || configured[dev].load() < static_cast<int>(smem)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (dev < kMaxDev) configured[dev].store(static_cast<int>(smem));
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // all CTAs must be resident at once (grid barriers): cooperative launch
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess) {
        // some drivers refuse the two attributes together: drop overlap
        (void)cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel, a);
    }
    return e;
}

}  // namespace

bool fused_supported(int fmt, int m, int hidden, int inter) {
    if (m < 1 || m > kFusedMaxRows) return false;
    if (hidden % 1024 != 0 || inter % 1024 != 0) return false;        // scale rows 16-byte aligned
    (void)fmt;
    return fused_rows_per_stage(2, hidden, fmt) >= 1 && fused_rows_per_stage(1, inter, fmt) >= 1;
}

size_t fused_smem(int fmt, int m, int hidden, int inter) { return fused_smem_bytes(m, hidden, inter, fmt); }

cudaError_t launch_ffn_fused(const FfnFusedArgs &a, int fmt, int m, cudaStream_t stream) {
    if (fmt == 0) return m == 1 ? launch_fused_t<0, 1>(a, stream) : launch_fused_t<0, 2>(a, stream);
    return m == 1 ? launch_fused_t<1, 1>(a, stream) : launch_fused_t<1, 2>(a, stream);
}

}  // namespace tq
