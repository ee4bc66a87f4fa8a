// Internal interface of the tensor-core convolutions and their helpers (conv_tc.cu).
#pragma once
#include <cuda_runtime.h>

#include "wan.h"

namespace wan {
// mode 0: causal 3x3x3 conv (w [Cout, 27, Cin]); mode 1: 2x2 phase convs (w [4, Cout, 4, Cin]).
cudaError_t conv_launch(int mode, const wan_bf16* a, const wan_bf16* cache_in, const wan_bf16* w,
                        const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T,
                        int H, int W, int Cin, int Cout, int sms, unsigned* err, cudaStream_t stream,
                        void* st_buf = nullptr, int st_groups = 0);
// The same convolutions on CTA pairs (tcgen05 .cta_group::2), for Cout >= 256 (conv_tc2.cu).
bool conv_pair_supported(int Cout);
cudaError_t conv_pair_launch(int mode, const wan_bf16* a, const wan_bf16* cache_in, const wan_bf16* w,
                             const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W,
                             int Cin, int Cout, int sms, unsigned* err, cudaStream_t stream,
                             void* st_buf = nullptr, int st_groups = 0, const float4* coef = nullptr,
                             int a_frames = 0, int y_frames = 0, int y_frame0 = 0, wan_bf16* cache_out = nullptr);
// Modes of conv_pair_launch beyond conv_launch's: 2, the causal 3x1x1 time conv to Cout = 2 C
// channels (w [Cout, 3, Cin]) whose output frame t, channel half i lands in frame
// y_frame0 + 2 t + i of y ([N, y_frames, H, W, Cout / 2]; Cout % 512 == 0, no residual), one
// output frame per CTA (wan_time_upsample runs time_up_launch below, two frames per CTA);
// 3, the 1x1x1 conv (w [Cout, Cin], no cache). a_frames: frames per n of the tensor `a` points
// into (0: T), so `a` may start at a later frame of a longer video.
// coef (optional, mode 0): GroupNorm + SiLU of `a` applied to the conv's operand tiles as they
// arrive (per (frame n*T + t, Cin channel) float4 coefficients as the norm's coefficients-only
// pass leaves them, blocked layout); the cache frames are used as they are.
// cache_out (optional, with coef; never cache_in): receives frames max(T - 2, 0) .. T - 1 of
// silu(a S + B) at cache frames t - T + 2, written by the prologue from its normalised tiles.
// GroupNorm statistics of the causal conv's output, emitted by the CTA-pair kernel's epilogue
// (Cout a multiple of 256, channels per group a power of two from 4 to 64; with or without the
// operand prologue). The buffer: a header of kGnStatsHeader bytes whose first int is q, the
// records per (frame, group) (pixel tiles x 4 epilogue warps of the launch that wrote them; the
// Winograd output transform writes the same layout with one record per 2x2 output tile), then
// per (frame, group, part < q) the float-float sums of d and d^2 of d = y - s as a float4, then
// the (s, count) pairs as float2 in the same order.
constexpr size_t kGnStatsHeader = 256;
bool conv_gn_stats_supported(int Cout, int groups);
size_t conv_gn_stats_bytes(int N, int T, int H, int W, int Cout, int groups);  // for either tiling
// The record counts q of the two tilings a launch at H x W may use (8 x 16 and 16 x 8 pixels).
void conv_gn_stats_records(int H, int W, int* q_a, int* q_b);
// The causal 3x1x1 time conv of the time upsample (time_up_tc2.cu), two output frames per CTA:
// conv output frame t of x's nf frames (x: frame stride a_frames per n; frames before it from
// cache_in [N, 2, H, W, C], else zeros) with w [2 C, 3, C] and bias [2 C], channel half i written
// to frame y_frame0 + 2 t + i of y [N, y_frames, H, W, C]. C % 256 == 0.
bool time_up_supported(int C);
cudaError_t time_up_launch(const wan_bf16* x, const wan_bf16* cache_in, const wan_bf16* w, const wan_bf16* bias,
                           wan_bf16* y, int N, int nf, int H, int W, int C, int a_frames, int y_frames, int y_frame0,
                           int sms, unsigned* err, cudaStream_t stream);
// cache_out[n, j] = ([cache_in or zeros; a])[n, T + j], j = 0, 1.
cudaError_t cache_update_launch(const wan_bf16* a, const wan_bf16* cache_in, wan_bf16* cache_out,
                                int N, int T, int H, int W, int C, int sms, cudaStream_t stream);
// Causal conv to exactly 12 output channels (the output head), Cin % 64 == 0 and Cin <= 256.
bool head_supported(int Cin, int Cout);
cudaError_t head_launch(const wan_bf16* a, const wan_bf16* cache_in, const wan_bf16* w, const wan_bf16* bias,
                        const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W, int Cin, int sms,
                        unsigned* err, cudaStream_t stream);
cudaError_t phase_weights_launch(const wan_bf16* w3, wan_bf16* wp, int Cin, int Cout, int sms,
                                 cudaStream_t stream);
// out = bf16(b2 + b_shortcut) per channel: the shortcut bias folded into the second conv's.
cudaError_t fold_bias_launch(const wan_bf16* b2, const wan_bf16* bsc, wan_bf16* out, int C, cudaStream_t stream);
}  // namespace wan
