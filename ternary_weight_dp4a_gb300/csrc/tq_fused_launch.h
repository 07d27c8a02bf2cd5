// tq_fused_launch.h -- host entry to the persistent fused FFN kernel.
#pragma once

#include <cuda_runtime.h>

#include "tq_ffn_fused.cuh"

namespace tq {

constexpr int kFusedMaxRows = 2;     // activation rows the fused kernel takes

// Shapes the fused kernel takes: m <= kFusedMaxRows, hidden and inter
// multiples of 1024.
bool fused_supported(int fmt, int m, int hidden, int inter);
size_t fused_smem(int fmt, int m, int hidden, int inter);
cudaError_t launch_ffn_fused(const FfnFusedArgs &a, int fmt, int m, cudaStream_t stream);

}  // namespace tq
