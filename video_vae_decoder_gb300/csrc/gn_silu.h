// Internal interface of the GroupNorm + SiLU kernels (gn_silu.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "wan.h"

namespace wan {
bool gn_silu_supported(int C, int groups);
size_t gn_silu_workspace(int N, int T, int H, int W, int C, int groups, int sms);
cudaError_t gn_silu_launch(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta,
                           int N, int T, int H, int W, int C, int groups, float eps, void* ws,
                           int sms, cudaStream_t stream);
}  // namespace wan
