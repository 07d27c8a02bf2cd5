// 1-bit binary GEMV instantiations.
#include "tq_gemv_inst.cuh"

namespace tq {
cudaError_t launch_gemv_b1(const GemvArgs &a, int m, int nw, cudaStream_t stream) {
    return dispatch_gemv<1>(a, m, nw, stream);
}
}  // namespace tq
