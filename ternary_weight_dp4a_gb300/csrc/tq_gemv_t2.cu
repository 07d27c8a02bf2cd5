// 2-bit ternary GEMV instantiations.
#include "tq_gemv_inst.cuh"

namespace tq {
cudaError_t launch_gemv_t2(const GemvArgs &a, int m, int nw, cudaStream_t stream) {
    return dispatch_gemv<0>(a, m, nw, stream);
}
}  // namespace tq
