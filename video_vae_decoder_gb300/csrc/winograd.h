// Internal interface of the Winograd F(2x2, 3x3) causal convolution (winograd.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "wan.h"

namespace wan {
// Sizes the variant takes: Cin % 64 == 0, Cout % 256 == 0.
bool wino_supported(int Cin, int Cout);
// Workspace of one call: the transformed input V (fp16) and the component products M (fp32).
size_t wino_workspace(int N, int T, int H, int W, int Cin, int Cout);
// u[16][Cout][3][Cin] (fp16 bits) = G g G^T of w[Cout][3][3][3][Cin] per temporal tap.
cudaError_t wino_weights_launch(const wan_bf16* w, uint16_t* u, int Cin, int Cout, int sms, cudaStream_t s);
// y = causal conv of a (silu(a S + B) with the blocked GroupNorm coefficients `coef`, if given;
// the cache frames as they are) through F(2x2, 3x3) with the transformed weights u.
cudaError_t wino_conv_launch(const wan_bf16* a, const float4* coef, const wan_bf16* cache_in, const uint16_t* u,
                             const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W,
                             int Cin, int Cout, void* ws, int sms, unsigned* err, cudaStream_t s,
                             wan_bf16* cache_out = nullptr, void* st_buf = nullptr, int st_groups = 0);
// cache_out (optional, never cache_in): receives frames max(T - 2, 0) .. T - 1 of the conv's
// input (silu(a S + B) with coef) at cache frames t - T + 2, from the input transform's staging.
// st_buf (optional): the output transform also writes the GroupNorm statistics of y for
// st_groups groups, in the layout of the CTA-pair conv's statistics (conv_tc.h), one record per
// (frame, group, 2x2 output tile): q = ceil(H/2) ceil(W/2) records per (frame, group).
bool wino_gn_stats_supported(int Cout, int groups);  // Winograd sizes, channels per group 4 .. 64, a power of two
int wino_gn_stats_records(int H, int W);
size_t wino_gn_stats_bytes(int N, int T, int H, int W, int groups);
}  // namespace wan
