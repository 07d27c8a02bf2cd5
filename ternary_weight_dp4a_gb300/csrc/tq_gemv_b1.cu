// 1-bit binary GEMV instantiations.
#include "tq_gemv_inst.cuh"

namespace tq {
cudaError_t launch_gemv_b1(const GemvArgs &a, int m, bool gateup, cudaStream_t stream) {
    return dispatch_gemv<1>(a, m, gateup, stream);
}
}  // namespace tq
