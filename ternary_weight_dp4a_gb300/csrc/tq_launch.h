// tq_launch.h -- host-side launch helpers shared by the libtq translation units.
#pragma once

#include <cuda_runtime.h>

#include "tq_gemv.cuh"

namespace tq {

// Launch the GEMV (nw = 1) or the fused gate/up + SiLU*up kernel (nw = 2) for
// format fmt and m packed rows.  Arguments are already validated.
cudaError_t launch_gemv_t2(const GemvArgs &a, int m, int nw, cudaStream_t stream);
cudaError_t launch_gemv_b1(const GemvArgs &a, int m, int nw, cudaStream_t stream);

// Largest dynamic shared memory a CTA may use on the current device.
size_t max_smem_optin(cudaError_t *err = nullptr);

}  // namespace tq
