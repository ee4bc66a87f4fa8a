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
                           int sms, cudaStream_t stream, bool apply = true, float4* coef_out = nullptr,
                           bool whole_clip = false, long long wait_cycles = 0, unsigned bar_extra = 0);
// apply = false: stop once the per-(frame, channel) coefficients are written (to coef_out, else
// into the workspace: gn_silu_coef), y is not touched; C % 64 == 0 then, and the coefficients of
// a frame are in the blocked layout (coef_blocked_index: 64-channel slices, channel 8 j + m at
// 8 m + j).
// whole_clip: statistics per (n, group) over all T frames of n instead of per frame; every frame
// of n gets the same coefficients.
// wait_cycles (0: the library's bound) and bar_extra (0) are for the self-test of the timeout path
// only: the bound of the grid-barrier waits in SM cycles, and arrivals the first barrier waits for
// beyond the grid's own (1 makes it unreachable, so every CTA gives up and returns).
// The coefficients from the statistics the CTA-pair conv's epilogue emitted for x (conv_tc.h:
// the buffer, its header and records), per (frame, group) in a fixed order: into coef ([N*T][C]
// float4, blocked layout if `blocked`, else channel order), the same quantities as the norm's own
// pass. stats_bytes bounds the record count the header gives (a larger one is recorded as
// kDevErrBadStats and nothing is written).
cudaError_t gn_coef_from_stats_launch(const void* stats, size_t stats_bytes, const float* gamma, const float* beta,
                                      int N, int T, int H, int W, int C, int groups, float eps, float4* coef,
                                      bool blocked, unsigned* err, cudaStream_t stream);
// Coefficients (S_hi, S_lo, B_hi, B_lo) per (frame, channel), [N*T][C] float4, inside ws.
const float4* gn_silu_coef(const void* ws, int N, int T, int H, int W, int C, int groups);
// The apply pass alone on frames [t_lo, T): y[n, o + t - t_lo] = silu(x[n, t] S + B), y with To
// frames per n, from blocked coefficients (apply = false); bit for bit what gn_silu_launch
// writes for those frames.
cudaError_t gn_apply_frames_launch(const wan_bf16* x, const float4* coef, wan_bf16* y, int N, int T, int H, int W,
                                   int C, int t_lo, int To, int o, int sms, cudaStream_t stream);
}  // namespace wan
