// tq_kernel_b.cu -- instantiations of the persistent kernel for launches of
// phase B alone (tq_gemv, the down projection of a staged h).
#include "tq.h"
#include "tq_kernel_run.cuh"

namespace tq {

cudaError_t launch_b_only(const KArgs &a, int fmt, int m, int grid, size_t bytes, cudaStream_t stream) {
    if (fmt == TQ_FMT_TERNARY2) {
        switch (m) {
            case 1: return launch_t<0, 1, true>(a, grid, bytes, false, stream);
            case 2: return launch_t<0, 2, true>(a, grid, bytes, false, stream);
            case 3: return launch_t<0, 3, true>(a, grid, bytes, false, stream);
            default: return launch_t<0, 4, true>(a, grid, bytes, false, stream);
        }
    }
    switch (m) {
        case 1: return launch_t<1, 1, true>(a, grid, bytes, false, stream);
        case 2: return launch_t<1, 2, true>(a, grid, bytes, false, stream);
        case 3: return launch_t<1, 3, true>(a, grid, bytes, false, stream);
        default: return launch_t<1, 4, true>(a, grid, bytes, false, stream);
    }
}

}  // namespace tq
