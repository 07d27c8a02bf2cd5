// 2-bit ternary GEMV instantiations.
#include "tq_gemv_inst.cuh"

namespace tq {
cudaError_t launch_gemv_t2(const GemvArgs &a, int m, bool gateup, cudaStream_t stream) {
    return dispatch_gemv<0>(a, m, gateup, stream);
}

// shared memory per CTA, both formats (defined once, here)
template <int FMT, bool GATEUP>
static size_t smem_for(int m, int nb, int n) {
    switch (m) {
        case 1: return gemv_smem<FMT, 1, GATEUP>(nb, n);
        case 2: return gemv_smem<FMT, 2, GATEUP>(nb, n);
        case 3: return gemv_smem<FMT, 3, GATEUP>(nb, n);
        case 4: return gemv_smem<FMT, 4, GATEUP>(nb, n);
        case 5: return gemv_smem<FMT, 5, GATEUP>(nb, n);
        case 6: return gemv_smem<FMT, 6, GATEUP>(nb, n);
        case 7: return gemv_smem<FMT, 7, GATEUP>(nb, n);
        default: return gemv_smem<FMT, 8, GATEUP>(nb, n);
    }
}

size_t gemv_smem_needed(int fmt, int m, bool gateup, int k, int n) {
    const int nb = k / kBlock;
    if (fmt == 0) return gateup ? smem_for<0, true>(m, nb, n) : smem_for<0, false>(m, nb, n);
    return gateup ? smem_for<1, true>(m, nb, n) : smem_for<1, false>(m, nb, n);
}
}  // namespace tq
