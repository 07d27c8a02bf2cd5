// tq_launch.h -- host-side launch helper shared by the libtq translation units.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace tq {

// Launch `kernel` with programmatic stream serialisation: it may start while
// the previous work in the stream drains, and synchronises inside through
// pdl_wait().  Every libtq kernel reads nothing produced by earlier stream
// work before that wait (weights excepted: nothing in a stream of libtq calls
// writes them).
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

}  // namespace tq
