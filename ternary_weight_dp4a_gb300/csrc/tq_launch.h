// tq_launch.h -- host-side launch helpers shared by the libtq translation units.
#pragma once

#include <cuda_runtime.h>

#include "tq_gemv.cuh"

namespace tq {

// Launch `kernel` with programmatic stream serialisation: it may start while
// the previous work in the stream drains, and synchronises inside through
// pdl_wait().  Every libtq kernel reads nothing produced by earlier stream
// work before that wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch the GEMV (gateup = false) or the fused gate/up + SiLU*up kernel for
// format fmt and m packed rows.  Arguments are already validated.
cudaError_t launch_gemv_t2(const GemvArgs &a, int m, bool gateup, cudaStream_t stream);
cudaError_t launch_gemv_b1(const GemvArgs &a, int m, bool gateup, cudaStream_t stream);

// Largest dynamic shared memory a CTA may use on the current device.
size_t max_smem_optin(cudaError_t *err = nullptr);

// Dynamic shared memory the GEMV kernel for (fmt, m, gateup) needs at (k, n).
size_t gemv_smem_needed(int fmt, int m, bool gateup, int k, int n);

}  // namespace tq
