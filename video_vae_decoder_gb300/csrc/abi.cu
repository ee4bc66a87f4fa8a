// The extern "C" entry points of include/wan.h: host-side validation, workspace layout and the
// ordering of the kernels on the caller's stream. Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <stdint.h>
#include <string.h>

#include "abi_util.h"
#include "common.cuh"
#include "conv_tc.h"
#include "gn_silu.h"
#include "wan.h"
#include "winograd.h"

namespace wan {

// Device error word: kernels that give up a bounded wait set bits here.
__device__ unsigned g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

}  // namespace

int sm_count() {
  static std::atomic<int> cached[kMaxDevices];  // 0 until queried; every query gives the same answer
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 148;
  int n = cached[d].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 148;
    cached[d].store(n, std::memory_order_relaxed);
  }
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t abytes, const void* b, size_t bbytes) {
  if (!a || !b || !abytes || !bbytes) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

wan_status cuda_status(cudaError_t e) { return e == cudaSuccess ? WAN_OK : WAN_ERR_CUDA; }

namespace {

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

bool positive(int a, int b, int c, int d, int e) { return a > 0 && b > 0 && c > 0 && d > 0 && e > 0; }

// Sizes the kernels index with 32-bit integers stay below 2^31.
bool fits(int N, int T, int H, int W, int C) {
  const long long px = (long long)H * W;
  return px * C < (1LL << 31) && (long long)N * T * 4 < (1LL << 31) && C <= 65536;
}

}  // namespace

wan_status check_gn(const void* x, const void* y, const float* gamma, const float* beta, int N, int T,
                    int H, int W, int C, int groups, float eps) {
  if (!x || !y || !gamma || !beta) return WAN_ERR_INVALID_ARG;
  if (!positive(N, T, H, W, C) || groups <= 0 || C % groups != 0) return WAN_ERR_INVALID_ARG;
  if (!(eps > 0.0f) || eps != eps || eps > 3.0e38f) return WAN_ERR_INVALID_ARG;
  if (!gn_silu_supported(C, groups) || !fits(N, T, H, W, C)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(y) || !aligned16(gamma) || !aligned16(beta)) return WAN_ERR_MISALIGNED;
  return WAN_OK;
}

namespace {

wan_status check_conv(const void* a, const void* w, const void* y, int N, int T, int H, int W, int Cin,
                      int Cout) {
  if (!a || !w || !y) return WAN_ERR_INVALID_ARG;
  if (!positive(N, T, H, W, Cin) || Cout <= 0) return WAN_ERR_INVALID_ARG;
  if (Cin % 64 != 0 || Cout % 2 != 0 || !fits(N, T, H, W, Cin) || !fits(N, T, H, W, Cout))
    return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a) || !aligned16(w) || !aligned16(y)) return WAN_ERR_MISALIGNED;
  return WAN_OK;
}

// GroupNorm + SiLU feeding a causal conv. The CTA-pair conv (Cout >= 256) normalises its operand
// tiles as they arrive: the norm's statistics pass writes coefficients only and the activation
// a = silu(gn(x)) is never stored, except its last two frames, which go to the cache. Otherwise a
// is materialised in the workspace and the conv reads it.
bool gn_conv_fused(int Cout) { return conv_pair_supported(Cout); }

size_t gn_conv_workspace(int N, int T, int H, int W, int Cin, int Cout, int groups) {
  const size_t gnws = align256(gn_silu_workspace(N, T, H, W, Cin, groups, sm_count()));
  if (gn_conv_fused(Cout)) return gnws;
  return gnws + align256((size_t)N * T * H * W * Cin * sizeof(wan_bf16));
}

// cache_out = the last two frames of [cache_in or zeros; silu(x S + B)] with the blocked
// coefficients of x. T >= 2: the normalised last two frames of x, written once. T = 1: the old
// frame 1 (or zeros) moves to frame 0 first (one strided copy; in place it reads frame 1 before
// anything writes it), then frame 0 of x goes to frame 1.
cudaError_t gn_cache_update(const wan_bf16* x, const float4* coef, const wan_bf16* cache_in, wan_bf16* cache_out,
                            int N, int T, int H, int W, int C, int sms, cudaStream_t s) {
  if (T >= 2) return gn_apply_frames_launch(x, coef, cache_out, N, T, H, W, C, T - 2, 2, 0, sms, s);
  const size_t fb = (size_t)H * W * C * sizeof(wan_bf16);
  cudaError_t e = cache_in ? cudaMemcpy2DAsync(cache_out, 2 * fb, cache_in + fb / sizeof(wan_bf16), 2 * fb, fb, N,
                                               cudaMemcpyDeviceToDevice, s)
                           : cudaMemset2DAsync(cache_out, 2 * fb, 0, fb, N, s);
  if (e != cudaSuccess) return e;
  return gn_apply_frames_launch(x, coef, cache_out, N, 1, H, W, C, 0, 2, 1, sms, s);
}

// cache_out[:, 0] = cache_in[:, 1] (zeros without cache_in): the part of a one-frame chunk's new
// history that the conv's prologue does not write.
cudaError_t cache_keep_last(const wan_bf16* cache_in, wan_bf16* cache_out, int N, int H, int W, int C,
                            cudaStream_t s) {
  const size_t fb = (size_t)H * W * C * sizeof(wan_bf16);
  return cache_in ? cudaMemcpy2DAsync(cache_out, 2 * fb, cache_in + fb / sizeof(wan_bf16), 2 * fb, fb, N,
                                      cudaMemcpyDeviceToDevice, s)
                  : cudaMemset2DAsync(cache_out, 2 * fb, 0, fb, N, s);
}

}  // namespace

unsigned* device_error_word() {
  static unsigned* cached[kMaxDevices] = {nullptr};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  if (!cached[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    cached[d] = static_cast<unsigned*>(p);
  }
  return cached[d];
}

}  // namespace wan

using namespace wan;

extern "C" {

const char* wan_status_string(wan_status s) {
  switch (s) {
    case WAN_OK: return "WAN_OK";
    case WAN_ERR_INVALID_ARG: return "WAN_ERR_INVALID_ARG: a pointer is NULL or a size/parameter is invalid";
    case WAN_ERR_UNSUPPORTED_SHAPE: return "WAN_ERR_UNSUPPORTED_SHAPE: no kernel for these sizes";
    case WAN_ERR_MISALIGNED: return "WAN_ERR_MISALIGNED: a pointer is not 16-byte aligned";
    case WAN_ERR_WORKSPACE: return "WAN_ERR_WORKSPACE: workspace missing or too small";
    case WAN_ERR_CUDA: return "WAN_ERR_CUDA: a CUDA call or kernel launch failed";
    case WAN_ERR_TIMEOUT: return "WAN_ERR_TIMEOUT: a kernel gave up a bounded wait";
  }
  return "WAN_ERR_UNKNOWN";
}

size_t wan_workspace_size(wan_op op, int N, int T, int H, int W, int Cin, int Cout, int groups) {
  if (!positive(N, T, H, W, Cin)) return 0;
  switch (op) {
    case WAN_OP_GN_SILU:
      if (groups <= 0 || Cin % groups || !gn_silu_supported(Cin, groups)) return 0;
      return gn_silu_workspace(N, T, H, W, Cin, groups, sm_count());
    case WAN_OP_CAUSAL_CONV3D:
    case WAN_OP_UPSAMPLE_PHASE_CONV:
      return 0;
    case WAN_OP_RESBLOCK: {  // h, then the norm-into-conv workspace
      if (groups <= 0 || Cin % groups || !gn_silu_supported(Cin, groups)) return 0;
      const size_t h = (size_t)N * T * H * W * Cin * sizeof(wan_bf16);
      return align256(h) + gn_conv_workspace(N, T, H, W, Cin, Cin, groups);
    }
    case WAN_OP_GN_STATS:
      if (!positive(Cout, groups, 1, 1, 1) || !conv_gn_stats_supported(Cout, groups)) return 0;
      return conv_gn_stats_bytes(N, T, H, W, Cout, groups);
    case WAN_OP_GN_SILU_CONV3D:
      if (Cout <= 0 || groups <= 0 || Cin % groups || !gn_silu_supported(Cin, groups)) return 0;
      return gn_conv_workspace(N, T, H, W, Cin, Cout, groups);
    case WAN_OP_WINOGRAD_CONV3D:
      if (!wino_supported(Cin, Cout)) return 0;
      return wino_workspace(N, T, H, W, Cin, Cout);
    case WAN_OP_RESBLOCK_WINOGRAD: {  // h, the coefficients, h's statistics, the norm's workspace, the conv's
      if (groups <= 0 || Cin % groups || !gn_silu_supported(Cin, groups) || !wino_supported(Cin, Cin)) return 0;
      return align256((size_t)N * T * H * W * Cin * sizeof(wan_bf16)) + align256((size_t)N * T * Cin * 16) +
             (wino_gn_stats_supported(Cin, groups) ? align256(wino_gn_stats_bytes(N, T, H, W, groups)) : 0) +
             align256(gn_silu_workspace(N, T, H, W, Cin, groups, sm_count())) + wino_workspace(N, T, H, W, Cin, Cin);
    }
    case WAN_OP_GN_STATS_WINOGRAD:
      if (!wino_gn_stats_supported(Cout, groups)) return 0;
      return wino_gn_stats_bytes(N, T, H, W, groups);
    case WAN_OP_RESBLOCK_SHORTCUT: {  // h, the shortcut, then the norm-into-conv workspace
      if (Cout <= 0 || groups <= 0 || Cin % groups || Cout % groups || !gn_silu_supported(Cin, groups) ||
          !gn_silu_supported(Cout, groups))
        return 0;
      const size_t y = (size_t)N * T * H * W * Cout * sizeof(wan_bf16);
      return 2 * align256(y) + std::max(gn_conv_workspace(N, T, H, W, Cin, Cout, groups),
                                        gn_conv_workspace(N, T, H, W, Cout, Cout, groups));
    }
  }
  return 0;
}

wan_status wan_gn_silu(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta, int N, int T,
                       int H, int W, int C, int groups, float eps, void* ws, size_t ws_bytes, void* stream) {
  WAN_CALL_RANGE();
  wan_status st = check_gn(x, y, gamma, beta, N, T, H, W, C, groups, eps);
  if (st != WAN_OK) return st;
  const size_t bytes = (size_t)N * T * H * W * C * sizeof(wan_bf16);
  if (overlap(x, bytes, y, bytes)) return WAN_ERR_INVALID_ARG;
  const size_t need = wan_workspace_size(WAN_OP_GN_SILU, N, T, H, W, C, 0, groups);
  if (!ws || ws_bytes < need) return WAN_ERR_WORKSPACE;
  if (!aligned16(ws)) return WAN_ERR_MISALIGNED;
  return cuda_status(gn_silu_launch(x, y, gamma, beta, N, T, H, W, C, groups, eps, ws, sm_count(),
                                    static_cast<cudaStream_t>(stream)));
}

wan_status wan_gn_silu_clip(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta, int N, int T,
                            int H, int W, int C, int groups, float eps, void* ws, size_t ws_bytes, void* stream) {
  WAN_CALL_RANGE();
  wan_status st = check_gn(x, y, gamma, beta, N, T, H, W, C, groups, eps);
  if (st != WAN_OK) return st;
  const size_t bytes = (size_t)N * T * H * W * C * sizeof(wan_bf16);
  if (overlap(x, bytes, y, bytes)) return WAN_ERR_INVALID_ARG;
  if ((double)H * W * (C / groups) >= 16777216.0) return WAN_ERR_UNSUPPORTED_SHAPE;  // a frame's count exact in fp32
  const size_t need = wan_workspace_size(WAN_OP_GN_SILU, N, T, H, W, C, 0, groups);
  if (!ws || ws_bytes < need) return WAN_ERR_WORKSPACE;
  if (!aligned16(ws)) return WAN_ERR_MISALIGNED;
  return cuda_status(gn_silu_launch(x, y, gamma, beta, N, T, H, W, C, groups, eps, ws, sm_count(),
                                    static_cast<cudaStream_t>(stream), true, nullptr, true));
}

}  // extern "C"

namespace {

// The smallest statistics buffer a producer (the pair conv in either tiling, or the Winograd
// output transform) writes for these sizes; the finalize kernel checks the record count in the
// header against the buffer's length before it reads a record.
size_t gn_stats_min_bytes(int N, int T, int H, int W, int groups) {
  int q_a, q_b;
  conv_gn_stats_records(H, W, &q_a, &q_b);
  const int q = std::min(std::min(q_a, q_b), wino_gn_stats_records(H, W));
  return kGnStatsHeader + (size_t)N * T * groups * q * (sizeof(float4) + sizeof(float2));
}

}  // namespace

extern "C" {

wan_status wan_gn_silu_from_stats(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta, int N,
                                  int T, int H, int W, int C, int groups, float eps, const void* stats,
                                  size_t stats_bytes, void* ws, size_t ws_bytes, void* stream) {
  WAN_CALL_RANGE();
  wan_status st = check_gn(x, y, gamma, beta, N, T, H, W, C, groups, eps);
  if (st != WAN_OK) return st;
  if (!stats) return WAN_ERR_INVALID_ARG;
  if (!conv_gn_stats_supported(C, groups)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(stats)) return WAN_ERR_MISALIGNED;
  if (stats_bytes < gn_stats_min_bytes(N, T, H, W, groups)) return WAN_ERR_INVALID_ARG;
  const size_t bytes = (size_t)N * T * H * W * C * sizeof(wan_bf16);
  if (overlap(x, bytes, y, bytes)) return WAN_ERR_INVALID_ARG;
  const size_t need = wan_workspace_size(WAN_OP_GN_SILU, N, T, H, W, C, 0, groups);
  if (!ws || ws_bytes < need) return WAN_ERR_WORKSPACE;
  if (!aligned16(ws)) return WAN_ERR_MISALIGNED;
  if (overlap(stats, stats_bytes, y, bytes) || overlap(ws, ws_bytes, y, bytes) || overlap(ws, ws_bytes, stats, stats_bytes))
    return WAN_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  // The coefficients from the statistics (into the workspace's coefficient area, blocked), then
  // the apply pass over every frame.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float4* coef = const_cast<float4*>(gn_silu_coef(ws, N, T, H, W, C, groups));
  cudaError_t e = gn_coef_from_stats_launch(stats, stats_bytes, gamma, beta, N, T, H, W, C, groups, eps, coef, true,
                                            err, s);
  if (e == cudaSuccess) e = gn_apply_frames_launch(x, coef, y, N, T, H, W, C, 0, T, 0, sm_count(), s);
  return cuda_status(e);
}

wan_status wan_gn_silu_coefficients_from_stats(const void* stats, size_t stats_bytes, const float* gamma,
                                               const float* beta, int N, int T, int H, int W, int C, int groups,
                                               float eps, void* coef, void* stream) {
  WAN_CALL_RANGE();
  if (!stats || !gamma || !beta || !coef) return WAN_ERR_INVALID_ARG;
  if (!positive(N, T, H, W, C) || groups <= 0 || C % groups != 0) return WAN_ERR_INVALID_ARG;
  if (!(eps > 0.0f) || eps != eps || eps > 3.0e38f) return WAN_ERR_INVALID_ARG;  // as check_gn
  if (!conv_gn_stats_supported(C, groups) || !gn_silu_supported(C, groups) || !fits(N, T, H, W, C))
    return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(stats) || !aligned16(coef) || !aligned16(gamma) || !aligned16(beta)) return WAN_ERR_MISALIGNED;
  if (stats_bytes < gn_stats_min_bytes(N, T, H, W, groups)) return WAN_ERR_INVALID_ARG;
  const size_t cbytes = (size_t)N * T * C * 16;
  if (overlap(stats, stats_bytes, coef, cbytes)) return WAN_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  return cuda_status(gn_coef_from_stats_launch(stats, stats_bytes, gamma, beta, N, T, H, W, C, groups, eps,
                                               static_cast<float4*>(coef), true, err,
                                               static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The conv kernel for these sizes: the 12-channel output head, else the general causal conv
// (stats: null or the checked statistics buffer of y).
cudaError_t launch_causal_conv(const wan_bf16* a, const wan_bf16* cache_in, const wan_bf16* w, const wan_bf16* bias,
                               const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W, int Cin, int Cout,
                               void* stats, int groups, unsigned* err, cudaStream_t s) {
  if (head_supported(Cin, Cout) && !stats)
    return head_launch(a, cache_in, w, bias, residual, y, N, T, H, W, Cin, sm_count(), err, s);
  return conv_launch(0, a, cache_in, w, bias, residual, y, N, T, H, W, Cin, Cout, sm_count(), err, s, stats, groups);
}

// The causal conv behind wan_causal_conv3d and wan_causal_conv3d_gn_stats (stats: null or the
// checked statistics buffer of y).
wan_status causal_conv(const wan_bf16* a, const wan_bf16* cache_in, wan_bf16* cache_out, const wan_bf16* w,
                       const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W,
                       int Cin, int Cout, void* stats, int groups, void* stream) {
  wan_status st = check_conv(a, w, y, N, T, H, W, Cin, Cout);
  if (st != WAN_OK) return st;
  if (!aligned16(cache_in) && cache_in) return WAN_ERR_MISALIGNED;
  if (!aligned16(cache_out) && cache_out) return WAN_ERR_MISALIGNED;
  if (!aligned16(bias) && bias) return WAN_ERR_MISALIGNED;
  if (!aligned16(residual) && residual) return WAN_ERR_MISALIGNED;
  const size_t abytes = (size_t)N * T * H * W * Cin * 2, ybytes = (size_t)N * T * H * W * Cout * 2;
  const size_t cbytes = (size_t)N * 2 * H * W * Cin * 2;
  if (overlap(a, abytes, y, ybytes) || overlap(residual, ybytes, y, ybytes) || overlap(cache_in, cbytes, y, ybytes) ||
      overlap(cache_out, cbytes, y, ybytes) || overlap(cache_out, cbytes, a, abytes))
    return WAN_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = cuda_status(launch_causal_conv(a, cache_in, w, bias, residual, y, N, T, H, W, Cin, Cout, stats, groups, err, s));
  if (st != WAN_OK || !cache_out) return st;
  return cuda_status(cache_update_launch(a, cache_in, cache_out, N, T, H, W, Cin, sm_count(), s));
}

// silu(gn(x)) into the causal conv, and the cache update, on checked arguments (gn_conv_fused
// above says how). cache_out may be cache_in: every conv read of it precedes the cache writes.
cudaError_t gn_conv(const wan_bf16* x, const float* gamma, const float* beta, int groups, float eps,
                    const wan_bf16* cache_in, wan_bf16* cache_out, const wan_bf16* w, const wan_bf16* bias,
                    const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W, int Cin, int Cout, void* ws,
                    unsigned* err, cudaStream_t s) {
  const int sms = sm_count();
  char* base = static_cast<char*>(ws);
  wan_bf16* act = reinterpret_cast<wan_bf16*>(base + align256(gn_silu_workspace(N, T, H, W, Cin, groups, sms)));
  cudaError_t e;
  if (!gn_conv_fused(Cout)) {
    e = gn_silu_launch(x, act, gamma, beta, N, T, H, W, Cin, groups, eps, ws, sms, s);
    if (e == cudaSuccess) e = launch_causal_conv(act, cache_in, w, bias, residual, y, N, T, H, W, Cin, Cout,
                                                 nullptr, 0, err, s);
    if (e == cudaSuccess && cache_out) e = cache_update_launch(act, cache_in, cache_out, N, T, H, W, Cin, sms, s);
    return e;
  }
  e = gn_silu_launch(x, nullptr, gamma, beta, N, T, H, W, Cin, groups, eps, ws, sms, s, false);
  const float4* coef = gn_silu_coef(ws, N, T, H, W, Cin, groups);
  // A cache_out apart from cache_in is written by the conv's prologue itself; in place, the new
  // history can only be written once the conv has read the old one.
  const bool direct = cache_out && cache_out != cache_in;
  if (e == cudaSuccess && direct && T == 1) e = cache_keep_last(cache_in, cache_out, N, H, W, Cin, s);
  if (e == cudaSuccess)
    e = conv_pair_launch(0, x, cache_in, w, bias, residual, y, N, T, H, W, Cin, Cout, sms, err, s, nullptr, 0, coef, 0,
                         0, 0, direct ? cache_out : nullptr);
  if (e != cudaSuccess || !cache_out || direct) return e;
  return gn_cache_update(x, coef, cache_in, cache_out, N, T, H, W, Cin, sms, s);
}

}  // namespace

extern "C" {

wan_status wan_causal_conv3d(const wan_bf16* a, const wan_bf16* cache_in, wan_bf16* cache_out,
                             const wan_bf16* w, const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y,
                             int N, int T, int H, int W, int Cin, int Cout, void* ws, size_t ws_bytes,
                             void* stream) {
  WAN_CALL_RANGE();
  (void)ws;
  (void)ws_bytes;
  return causal_conv(a, cache_in, cache_out, w, bias, residual, y, N, T, H, W, Cin, Cout, nullptr, 0, stream);
}

wan_status wan_causal_conv3d_gn_stats(const wan_bf16* a, const wan_bf16* cache_in, wan_bf16* cache_out,
                                      const wan_bf16* w, const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y,
                                      int N, int T, int H, int W, int Cin, int Cout, int groups, void* stats,
                                      size_t stats_bytes, void* stream) {
  WAN_CALL_RANGE();
  if (!stats || groups <= 0) return WAN_ERR_INVALID_ARG;
  if (!positive(N, T, H, W, Cin) || Cout <= 0) return WAN_ERR_INVALID_ARG;
  if (!conv_gn_stats_supported(Cout, groups)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(stats)) return WAN_ERR_MISALIGNED;
  if (stats_bytes < conv_gn_stats_bytes(N, T, H, W, Cout, groups)) return WAN_ERR_INVALID_ARG;
  return causal_conv(a, cache_in, cache_out, w, bias, residual, y, N, T, H, W, Cin, Cout, stats, groups, stream);
}

wan_status wan_gn_silu_causal_conv3d(const wan_bf16* x, const float* gamma, const float* beta, int groups,
                                     float eps, const wan_bf16* cache_in, wan_bf16* cache_out, const wan_bf16* w,
                                     const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T, int H,
                                     int W, int Cin, int Cout, void* ws, size_t ws_bytes, void* stream) {
  WAN_CALL_RANGE();
  wan_status st = check_gn(x, y, gamma, beta, N, T, H, W, Cin, groups, eps);
  if (st != WAN_OK) return st;
  st = check_conv(x, w, y, N, T, H, W, Cin, Cout);
  if (st != WAN_OK) return st;
  if ((cache_in && !aligned16(cache_in)) || (cache_out && !aligned16(cache_out)) || (bias && !aligned16(bias)) ||
      (residual && !aligned16(residual)))
    return WAN_ERR_MISALIGNED;
  const size_t xbytes = (size_t)N * T * H * W * Cin * 2, ybytes = (size_t)N * T * H * W * Cout * 2;
  const size_t cbytes = (size_t)N * 2 * H * W * Cin * 2;
  if (overlap(x, xbytes, y, ybytes) || overlap(residual, ybytes, y, ybytes) || overlap(cache_in, cbytes, y, ybytes) ||
      overlap(cache_out, cbytes, y, ybytes) || overlap(cache_out, cbytes, x, xbytes) ||
      (cache_in && cache_in != cache_out && overlap(cache_in, cbytes, cache_out, cbytes)))
    return WAN_ERR_INVALID_ARG;
  const size_t need = gn_conv_workspace(N, T, H, W, Cin, Cout, groups);
  if (!ws || ws_bytes < need) return WAN_ERR_WORKSPACE;
  if (!aligned16(ws)) return WAN_ERR_MISALIGNED;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  return cuda_status(gn_conv(x, gamma, beta, groups, eps, cache_in, cache_out, w, bias, residual, y, N, T, H, W, Cin,
                             Cout, ws, err, static_cast<cudaStream_t>(stream)));
}

wan_status wan_gn_silu_coefficients(const wan_bf16* x, const float* gamma, const float* beta, int N, int T, int H,
                                    int W, int C, int groups, float eps, void* coef, void* ws, size_t ws_bytes,
                                    void* stream) {
  WAN_CALL_RANGE();
  wan_status st = check_gn(x, coef, gamma, beta, N, T, H, W, C, groups, eps);
  if (st != WAN_OK) return st;
  if (C % 64 != 0) return WAN_ERR_UNSUPPORTED_SHAPE;
  const size_t xbytes = (size_t)N * T * H * W * C * 2, cbytes = (size_t)N * T * C * 16;
  if (overlap(x, xbytes, coef, cbytes)) return WAN_ERR_INVALID_ARG;
  const size_t need = wan_workspace_size(WAN_OP_GN_SILU, N, T, H, W, C, 0, groups);
  if (!ws || ws_bytes < need) return WAN_ERR_WORKSPACE;
  if (!aligned16(ws)) return WAN_ERR_MISALIGNED;
  return cuda_status(gn_silu_launch(x, nullptr, gamma, beta, N, T, H, W, C, groups, eps, ws, sm_count(),
                                    static_cast<cudaStream_t>(stream), false, static_cast<float4*>(coef)));
}

}  // extern "C"

namespace {

// wan_causal_conv3d_gn_input and its statistics-emitting form (stats: null, or a buffer of
// stats_bytes for `groups` groups of y).
wan_status gn_input_conv(const wan_bf16* x, const void* coef, const wan_bf16* cache_in, wan_bf16* cache_out,
                         const wan_bf16* w, const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T,
                         int H, int W, int Cin, int Cout, int groups, void* stats, size_t stats_bytes, void* stream) {
  if (!coef) return WAN_ERR_INVALID_ARG;
  wan_status st = check_conv(x, w, y, N, T, H, W, Cin, Cout);
  if (st != WAN_OK) return st;
  if (!gn_conv_fused(Cout)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (stats) {
    if (groups <= 0) return WAN_ERR_INVALID_ARG;
    if (!conv_gn_stats_supported(Cout, groups)) return WAN_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(stats)) return WAN_ERR_MISALIGNED;
    if (stats_bytes < conv_gn_stats_bytes(N, T, H, W, Cout, groups)) return WAN_ERR_INVALID_ARG;
  }
  if (!aligned16(coef) || (cache_in && !aligned16(cache_in)) || (cache_out && !aligned16(cache_out)) ||
      (bias && !aligned16(bias)) || (residual && !aligned16(residual)))
    return WAN_ERR_MISALIGNED;
  const size_t xbytes = (size_t)N * T * H * W * Cin * 2, ybytes = (size_t)N * T * H * W * Cout * 2;
  const size_t cbytes = (size_t)N * 2 * H * W * Cin * 2;
  if (overlap(x, xbytes, y, ybytes) || overlap(residual, ybytes, y, ybytes) || overlap(cache_in, cbytes, y, ybytes) ||
      overlap(coef, (size_t)N * T * Cin * 16, y, ybytes) || overlap(cache_out, cbytes, y, ybytes) ||
      overlap(cache_out, cbytes, x, xbytes) || overlap(cache_out, cbytes, coef, (size_t)N * T * Cin * 16) ||
      (cache_in && cache_out && cache_in != cache_out && overlap(cache_in, cbytes, cache_out, cbytes)))
    return WAN_ERR_INVALID_ARG;
  if (stats && (overlap(stats, stats_bytes, y, ybytes) || overlap(stats, stats_bytes, x, xbytes) ||
                overlap(stats, stats_bytes, coef, (size_t)N * T * Cin * 16) ||
                overlap(stats, stats_bytes, cache_out, cbytes) || overlap(stats, stats_bytes, residual, ybytes) ||
                overlap(stats, stats_bytes, cache_in, cbytes)))
    return WAN_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float4* cf = static_cast<const float4*>(coef);
  const bool direct = cache_out && cache_out != cache_in;
  cudaError_t e = cudaSuccess;
  if (direct && T == 1) e = cache_keep_last(cache_in, cache_out, N, H, W, Cin, s);
  if (e == cudaSuccess)
    e = conv_pair_launch(0, x, cache_in, w, bias, residual, y, N, T, H, W, Cin, Cout, sm_count(), err, s, stats,
                         stats ? groups : 0, cf, 0, 0, 0, direct ? cache_out : nullptr);
  if (e != cudaSuccess || !cache_out || direct) return cuda_status(e);
  return cuda_status(gn_cache_update(x, cf, cache_in, cache_out, N, T, H, W, Cin, sm_count(), s));
}

}  // namespace

extern "C" {

wan_status wan_causal_conv3d_gn_input(const wan_bf16* x, const void* coef, const wan_bf16* cache_in, wan_bf16* cache_out,
                                      const wan_bf16* w, const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y,
                                      int N, int T, int H, int W, int Cin, int Cout, void* stream) {
  WAN_CALL_RANGE();
  return gn_input_conv(x, coef, cache_in, cache_out, w, bias, residual, y, N, T, H, W, Cin, Cout, 0, nullptr, 0,
                       stream);
}

wan_status wan_causal_conv3d_gn_input_stats(const wan_bf16* x, const void* coef, const wan_bf16* cache_in,
                                            wan_bf16* cache_out, const wan_bf16* w, const wan_bf16* bias,
                                            const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W, int Cin,
                                            int Cout, int groups, void* stats, size_t stats_bytes, void* stream) {
  WAN_CALL_RANGE();
  if (!stats) return WAN_ERR_INVALID_ARG;
  return gn_input_conv(x, coef, cache_in, cache_out, w, bias, residual, y, N, T, H, W, Cin, Cout, groups, stats,
                       stats_bytes, stream);
}

wan_status wan_gn_silu_cache_update(const wan_bf16* x, const void* coef, const wan_bf16* cache_in, wan_bf16* cache_out,
                                    int N, int T, int H, int W, int C, void* stream) {
  WAN_CALL_RANGE();
  if (!x || !coef || !cache_out) return WAN_ERR_INVALID_ARG;
  if (!positive(N, T, H, W, C)) return WAN_ERR_INVALID_ARG;
  if (C % 64 != 0 || C > 2048 || !fits(N, T, H, W, C)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(coef) || !aligned16(cache_out) || (cache_in && !aligned16(cache_in)))
    return WAN_ERR_MISALIGNED;
  const size_t xbytes = (size_t)N * T * H * W * C * 2, cbytes = (size_t)N * 2 * H * W * C * 2;
  if (overlap(cache_out, cbytes, x, xbytes) || overlap(cache_out, cbytes, coef, (size_t)N * T * C * 16) ||
      (cache_in && cache_in != cache_out && overlap(cache_in, cbytes, cache_out, cbytes)))
    return WAN_ERR_INVALID_ARG;
  return cuda_status(gn_cache_update(x, static_cast<const float4*>(coef), cache_in, cache_out, N, T, H, W, C,
                                     sm_count(), static_cast<cudaStream_t>(stream)));
}

wan_status wan_cache_update(const wan_bf16* a, const wan_bf16* cache_in, wan_bf16* cache_out, int N, int T, int H,
                            int W, int C, void* stream) {
  WAN_CALL_RANGE();
  if (!a || !cache_out) return WAN_ERR_INVALID_ARG;
  if (!positive(N, T, H, W, C)) return WAN_ERR_INVALID_ARG;
  if (C % 8 != 0 || !fits(N, T, H, W, C)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a) || !aligned16(cache_out) || (cache_in && !aligned16(cache_in))) return WAN_ERR_MISALIGNED;
  const size_t abytes = (size_t)N * T * H * W * C * 2, cbytes = (size_t)N * 2 * H * W * C * 2;
  if (overlap(cache_out, cbytes, a, abytes)) return WAN_ERR_INVALID_ARG;
  if (cache_in && cache_in != cache_out && overlap(cache_in, cbytes, cache_out, cbytes)) return WAN_ERR_INVALID_ARG;
  return cuda_status(cache_update_launch(a, cache_in, cache_out, N, T, H, W, C, sm_count(),
                                         static_cast<cudaStream_t>(stream)));
}

wan_status wan_upsample_phase_weights(const wan_bf16* w3, wan_bf16* wp, int Cin, int Cout, void* stream) {
  WAN_CALL_RANGE();
  if (!w3 || !wp || Cin <= 0 || Cout <= 0) return WAN_ERR_INVALID_ARG;
  if ((long long)Cin * Cout * 16 >= (1LL << 40)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(w3) || !aligned16(wp)) return WAN_ERR_MISALIGNED;
  if (overlap(w3, (size_t)Cout * 9 * Cin * 2, wp, (size_t)Cout * 16 * Cin * 2)) return WAN_ERR_INVALID_ARG;
  return cuda_status(phase_weights_launch(w3, wp, Cin, Cout, sm_count(), static_cast<cudaStream_t>(stream)));
}

wan_status wan_upsample_phase_conv(const wan_bf16* x, const wan_bf16* wp, const wan_bf16* bias, wan_bf16* y,
                                   int N, int T, int H, int W, int Cin, int Cout, void* stream) {
  WAN_CALL_RANGE();
  wan_status st = check_conv(x, wp, y, N, T, 2 * H, 2 * W, Cin, Cout);
  if (st != WAN_OK) return st;
  if (bias && !aligned16(bias)) return WAN_ERR_MISALIGNED;
  const size_t xbytes = (size_t)N * T * H * W * Cin * 2, ybytes = (size_t)N * T * 4 * H * W * Cout * 2;
  if (overlap(x, xbytes, y, ybytes) || overlap(wp, (size_t)16 * Cout * Cin * 2, y, ybytes)) return WAN_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  return cuda_status(conv_launch(1, x, nullptr, wp, bias, nullptr, y, N, T, H, W, Cin, Cout, sm_count(), err,
                                 static_cast<cudaStream_t>(stream)));
}

wan_status wan_resblock(const wan_bf16* x, wan_bf16* out, const wan_resblock_params* p, wan_bf16* cache1,
                        wan_bf16* cache2, int cache_valid, int N, int T, int H, int W, int C, void* ws,
                        size_t ws_bytes, void* stream) {
  WAN_CALL_RANGE();
  if (!p || !cache1 || !cache2) return WAN_ERR_INVALID_ARG;
  wan_status st = check_gn(x, out, p->gamma1, p->beta1, N, T, H, W, C, p->groups, p->eps);
  if (st != WAN_OK) return st;
  st = check_gn(x, out, p->gamma2, p->beta2, N, T, H, W, C, p->groups, p->eps);
  if (st != WAN_OK) return st;
  st = check_conv(x, p->w1, out, N, T, H, W, C, C);
  if (st != WAN_OK) return st;
  st = check_conv(x, p->w2, out, N, T, H, W, C, C);
  if (st != WAN_OK) return st;
  if (!aligned16(cache1) || !aligned16(cache2) || (p->b1 && !aligned16(p->b1)) || (p->b2 && !aligned16(p->b2)))
    return WAN_ERR_MISALIGNED;
  const size_t bytes = (size_t)N * T * H * W * C * 2, cbytes = (size_t)N * 2 * H * W * C * 2;
  if (overlap(x, bytes, out, bytes) || overlap(cache1, cbytes, cache2, cbytes) || overlap(cache1, cbytes, out, bytes) ||
      overlap(cache2, cbytes, out, bytes) || overlap(cache1, cbytes, x, bytes) || overlap(cache2, cbytes, x, bytes))
    return WAN_ERR_INVALID_ARG;
  const size_t need = wan_workspace_size(WAN_OP_RESBLOCK, N, T, H, W, C, C, p->groups);
  if (!ws || ws_bytes < need) return WAN_ERR_WORKSPACE;
  if (!aligned16(ws)) return WAN_ERR_MISALIGNED;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  wan_bf16* h = reinterpret_cast<wan_bf16*>(base);
  void* gws = base + align256(bytes);
  const wan_bf16* c1_in = cache_valid ? cache1 : nullptr;
  const wan_bf16* c2_in = cache_valid ? cache2 : nullptr;
  // Each norm feeds its conv directly (the cache update of that conv's input included).
  cudaError_t e = gn_conv(x, p->gamma1, p->beta1, p->groups, p->eps, c1_in, cache1, p->w1, p->b1, nullptr, h, N, T,
                          H, W, C, C, gws, err, s);
  if (e == cudaSuccess)
    e = gn_conv(h, p->gamma2, p->beta2, p->groups, p->eps, c2_in, cache2, p->w2, p->b2, x, out, N, T, H, W, C, C, gws,
                err, s);
  return cuda_status(e);
}

wan_status wan_time_upsample(const wan_bf16* x, const wan_bf16* cache_in, wan_bf16* cache_out, const wan_bf16* w,
                             const wan_bf16* bias, wan_bf16* y, int N, int T, int H, int W, int C, int first,
                             void* stream) {
  WAN_CALL_RANGE();
  if (!x || !w || !y) return WAN_ERR_INVALID_ARG;
  if (!positive(N, T, H, W, C)) return WAN_ERR_INVALID_ARG;
  if (C % 256 != 0 || !fits(N, 2 * T, H, W, C)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)) ||
      (cache_in && !aligned16(cache_in)) || (cache_out && !aligned16(cache_out)))
    return WAN_ERR_MISALIGNED;
  const int start = first ? 1 : 0, nf = T - start, To = start + 2 * nf;
  const size_t fb = (size_t)H * W * C * sizeof(wan_bf16);
  const size_t xbytes = (size_t)N * T * fb, ybytes = (size_t)N * To * fb, cbytes = (size_t)N * 2 * fb;
  if (overlap(x, xbytes, y, ybytes) || overlap(cache_in, cbytes, y, ybytes) || overlap(cache_out, cbytes, y, ybytes) ||
      overlap(cache_out, cbytes, x, xbytes) || (cache_in && cache_in != cache_out && overlap(cache_in, cbytes, cache_out, cbytes)))
    return WAN_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  // The first frame of the first chunk passes through.
  if (first) e = cudaMemcpy2DAsync(y, To * fb, x, T * fb, fb, N, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && nf > 0)
    e = time_up_launch(x + (size_t)start * fb / sizeof(wan_bf16), cache_in, w, bias, y, N, nf, H, W, C, T, To, start,
                       sm_count(), err, s);
  if (e != cudaSuccess || !cache_out) return cuda_status(e);
  // The new history: the last two frames of [cache_in or zeros; x[:, start:]].
  const char* xb = reinterpret_cast<const char*>(x);
  char* cb = reinterpret_cast<char*>(cache_out);
  if (nf >= 2) {
    e = cudaMemcpy2DAsync(cb, 2 * fb, xb + (size_t)(T - 2) * fb, T * fb, 2 * fb, N, cudaMemcpyDeviceToDevice, s);
  } else {
    const int keep = 2 - nf;  // frames of the old history that stay: its last `keep`
    if (cache_in)
      e = cache_in == cache_out && keep == 2 ? cudaSuccess
                                             : cudaMemcpy2DAsync(cb, 2 * fb, reinterpret_cast<const char*>(cache_in) + (2 - keep) * fb,
                                                                 2 * fb, keep * fb, N, cudaMemcpyDeviceToDevice, s);
    else
      e = cudaMemset2DAsync(cb, 2 * fb, 0, keep * fb, N, s);
    if (e == cudaSuccess && nf == 1)
      e = cudaMemcpy2DAsync(cb + fb, 2 * fb, xb + (size_t)(T - 1) * fb, T * fb, fb, N, cudaMemcpyDeviceToDevice, s);
  }
  return cuda_status(e);
}

wan_status wan_conv1x1(const wan_bf16* x, const wan_bf16* w, wan_bf16* y, int N, int T, int H, int W, int Cin,
                       int Cout, void* stream) {
  WAN_CALL_RANGE();
  wan_status st = check_conv(x, w, y, N, T, H, W, Cin, Cout);
  if (st != WAN_OK) return st;
  if (!conv_pair_supported(Cout)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (overlap(x, (size_t)N * T * H * W * Cin * 2, y, (size_t)N * T * H * W * Cout * 2)) return WAN_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  return cuda_status(conv_pair_launch(3, x, nullptr, w, nullptr, nullptr, y, N, T, H, W, Cin, Cout, sm_count(), err,
                                      static_cast<cudaStream_t>(stream)));
}

wan_status wan_fold_bias(const wan_bf16* b2, const wan_bf16* b_shortcut, wan_bf16* out, int C, void* stream) {
  WAN_CALL_RANGE();
  if (!b2 || !b_shortcut || !out || C <= 0) return WAN_ERR_INVALID_ARG;
  return cuda_status(fold_bias_launch(b2, b_shortcut, out, C, static_cast<cudaStream_t>(stream)));
}

wan_status wan_resblock_shortcut(const wan_bf16* x, wan_bf16* out, const wan_resblock_params* p, const wan_bf16* w_sc,
                                 wan_bf16* cache1, wan_bf16* cache2, int cache_valid, int N, int T, int H, int W,
                                 int Cin, int Cout, void* ws, size_t ws_bytes, void* stream) {
  WAN_CALL_RANGE();
  if (!p || !cache1 || !cache2 || !w_sc) return WAN_ERR_INVALID_ARG;
  wan_status st = check_gn(x, out, p->gamma1, p->beta1, N, T, H, W, Cin, p->groups, p->eps);
  if (st != WAN_OK) return st;
  st = check_gn(out, out, p->gamma2, p->beta2, N, T, H, W, Cout, p->groups, p->eps);
  if (st != WAN_OK) return st;
  st = check_conv(x, p->w1, out, N, T, H, W, Cin, Cout);
  if (st != WAN_OK) return st;
  st = check_conv(out, p->w2, out, N, T, H, W, Cout, Cout);
  if (st != WAN_OK) return st;
  if (!conv_pair_supported(Cout)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(cache1) || !aligned16(cache2) || !aligned16(w_sc) || (p->b1 && !aligned16(p->b1)) ||
      (p->b2 && !aligned16(p->b2)))
    return WAN_ERR_MISALIGNED;
  const size_t xb = (size_t)N * T * H * W * Cin * 2, yb = (size_t)N * T * H * W * Cout * 2;
  const size_t c1b = (size_t)N * 2 * H * W * Cin * 2, c2b = (size_t)N * 2 * H * W * Cout * 2;
  if (overlap(x, xb, out, yb) || overlap(cache1, c1b, cache2, c2b) || overlap(cache1, c1b, out, yb) ||
      overlap(cache2, c2b, out, yb) || overlap(cache1, c1b, x, xb) || overlap(cache2, c2b, x, xb))
    return WAN_ERR_INVALID_ARG;
  const size_t need = wan_workspace_size(WAN_OP_RESBLOCK_SHORTCUT, N, T, H, W, Cin, Cout, p->groups);
  if (!ws || ws_bytes < need) return WAN_ERR_WORKSPACE;
  if (!aligned16(ws)) return WAN_ERR_MISALIGNED;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  wan_bf16* h = reinterpret_cast<wan_bf16*>(base);
  wan_bf16* skip = reinterpret_cast<wan_bf16*>(base + align256(yb));
  void* gws = base + 2 * align256(yb);
  const wan_bf16* c1_in = cache_valid ? cache1 : nullptr;
  const wan_bf16* c2_in = cache_valid ? cache2 : nullptr;
  // skip = the 1x1x1 conv of x without bias (p->b2 carries the folded shortcut bias), then the
  // two norm-into-conv steps, the second adding skip as its residual.
  cudaError_t e = conv_pair_launch(3, x, nullptr, w_sc, nullptr, nullptr, skip, N, T, H, W, Cin, Cout, sm_count(),
                                   err, s);
  if (e == cudaSuccess)
    e = gn_conv(x, p->gamma1, p->beta1, p->groups, p->eps, c1_in, cache1, p->w1, p->b1, nullptr, h, N, T, H, W, Cin,
                Cout, gws, err, s);
  if (e == cudaSuccess)
    e = gn_conv(h, p->gamma2, p->beta2, p->groups, p->eps, c2_in, cache2, p->w2, p->b2, skip, out, N, T, H, W, Cout,
                Cout, gws, err, s);
  return cuda_status(e);
}

wan_status wan_winograd_weights(const wan_bf16* w, wan_fp16* u, int Cin, int Cout, void* stream) {
  WAN_CALL_RANGE();
  if (!w || !u || Cin <= 0 || Cout <= 0) return WAN_ERR_INVALID_ARG;
  if (!wino_supported(Cin, Cout) || (long long)Cin * Cout * 27 >= (1LL << 40)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(w) || !aligned16(u)) return WAN_ERR_MISALIGNED;
  if (overlap(w, (size_t)Cout * 27 * Cin * 2, u, (size_t)16 * Cout * 3 * Cin * 2)) return WAN_ERR_INVALID_ARG;
  return cuda_status(wino_weights_launch(w, u, Cin, Cout, sm_count(), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The Winograd conv behind wan_causal_conv3d_winograd and wan_causal_conv3d_winograd_stats
// (stats: null, or a statistics buffer of stats_bytes for `groups` groups, checked here).
wan_status winograd_conv(const wan_bf16* a, const void* coef, const wan_bf16* cache_in, wan_bf16* cache_out,
                         const wan_fp16* u, const wan_bf16* bias, const wan_bf16* residual, wan_bf16* y, int N, int T,
                         int H, int W, int Cin, int Cout, void* ws, size_t ws_bytes, void* stats, size_t stats_bytes,
                         int groups, void* stream) {
  wan_status st = check_conv(a, u, y, N, T, H, W, Cin, Cout);
  if (st != WAN_OK) return st;
  if (!wino_supported(Cin, Cout) || Cin > 2048) return WAN_ERR_UNSUPPORTED_SHAPE;
  if ((coef && !aligned16(coef)) || (cache_in && !aligned16(cache_in)) || (cache_out && !aligned16(cache_out)) ||
      (bias && !aligned16(bias)) || (residual && !aligned16(residual)))
    return WAN_ERR_MISALIGNED;
  const size_t abytes = (size_t)N * T * H * W * Cin * 2, ybytes = (size_t)N * T * H * W * Cout * 2;
  const size_t cbytes = (size_t)N * 2 * H * W * Cin * 2;
  const size_t need = wino_workspace(N, T, H, W, Cin, Cout);
  if (overlap(a, abytes, y, ybytes) || overlap(residual, ybytes, y, ybytes) || overlap(cache_in, cbytes, y, ybytes) ||
      overlap(cache_out, cbytes, y, ybytes) || overlap(cache_out, cbytes, a, abytes) ||
      overlap(coef, (size_t)N * T * Cin * 16, y, ybytes) ||
      (cache_in && cache_out && cache_in != cache_out && overlap(cache_in, cbytes, cache_out, cbytes)) ||
      overlap(ws, need, a, abytes) || overlap(ws, need, y, ybytes) || overlap(ws, need, u, (size_t)96 * Cout * Cin))
    return WAN_ERR_INVALID_ARG;
  if (!ws || ws_bytes < need) return WAN_ERR_WORKSPACE;
  if (!aligned16(ws)) return WAN_ERR_MISALIGNED;
  if (stats) {
    if (!wino_gn_stats_supported(Cout, groups)) return WAN_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(stats)) return WAN_ERR_MISALIGNED;
    if (stats_bytes < wino_gn_stats_bytes(N, T, H, W, groups) || overlap(stats, stats_bytes, a, abytes) ||
        overlap(stats, stats_bytes, y, ybytes) || overlap(stats, stats_bytes, residual, ybytes) ||
        overlap(stats, stats_bytes, cache_in, cbytes) || overlap(stats, stats_bytes, cache_out, cbytes) ||
        overlap(stats, stats_bytes, ws, need) || overlap(stats, stats_bytes, coef, (size_t)N * T * Cin * 16))
      return WAN_ERR_INVALID_ARG;
  }
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float4* cf = static_cast<const float4*>(coef);
  // A cache_out apart from cache_in is written by the input transform from its staged pixels.
  const bool direct = cache_out && cache_out != cache_in;
  cudaError_t e = cudaSuccess;
  if (direct && T == 1) e = cache_keep_last(cache_in, cache_out, N, H, W, Cin, s);
  if (e == cudaSuccess)
    e = wino_conv_launch(a, cf, cache_in, u, bias, residual, y, N, T, H, W, Cin, Cout, ws, sm_count(), err, s,
                         direct ? cache_out : nullptr, stats, groups);
  if (e != cudaSuccess || !cache_out || direct) return cuda_status(e);
  if (cf) return cuda_status(gn_cache_update(a, cf, cache_in, cache_out, N, T, H, W, Cin, sm_count(), s));
  return cuda_status(cache_update_launch(a, cache_in, cache_out, N, T, H, W, Cin, sm_count(), s));
}

}  // namespace

extern "C" {

wan_status wan_causal_conv3d_winograd(const wan_bf16* a, const void* coef, const wan_bf16* cache_in,
                                      wan_bf16* cache_out, const wan_fp16* u, const wan_bf16* bias,
                                      const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W, int Cin,
                                      int Cout, void* ws, size_t ws_bytes, void* stream) {
  WAN_CALL_RANGE();
  return winograd_conv(a, coef, cache_in, cache_out, u, bias, residual, y, N, T, H, W, Cin, Cout, ws, ws_bytes,
                       nullptr, 0, 0, stream);
}

wan_status wan_causal_conv3d_winograd_stats(const wan_bf16* a, const void* coef, const wan_bf16* cache_in,
                                            wan_bf16* cache_out, const wan_fp16* u, const wan_bf16* bias,
                                            const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W,
                                            int Cin, int Cout, int groups, void* stats, size_t stats_bytes, void* ws,
                                            size_t ws_bytes, void* stream) {
  WAN_CALL_RANGE();
  if (!stats || groups <= 0) return WAN_ERR_INVALID_ARG;
  return winograd_conv(a, coef, cache_in, cache_out, u, bias, residual, y, N, T, H, W, Cin, Cout, ws, ws_bytes,
                       stats, stats_bytes, groups, stream);
}

wan_status wan_resblock_winograd(const wan_bf16* x, wan_bf16* out, const wan_resblock_params* p, const wan_fp16* u1,
                                 const wan_fp16* u2, wan_bf16* cache1, wan_bf16* cache2, int cache_valid, int N, int T,
                                 int H, int W, int C, void* ws, size_t ws_bytes, void* stream) {
  WAN_CALL_RANGE();
  if (!p || !cache1 || !cache2 || !u1 || !u2) return WAN_ERR_INVALID_ARG;
  wan_status st = check_gn(x, out, p->gamma1, p->beta1, N, T, H, W, C, p->groups, p->eps);
  if (st != WAN_OK) return st;
  st = check_gn(x, out, p->gamma2, p->beta2, N, T, H, W, C, p->groups, p->eps);
  if (st != WAN_OK) return st;
  st = check_conv(x, u1, out, N, T, H, W, C, C);
  if (st != WAN_OK) return st;
  if (!wino_supported(C, C)) return WAN_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(cache1) || !aligned16(cache2) || !aligned16(u2) || (p->b1 && !aligned16(p->b1)) ||
      (p->b2 && !aligned16(p->b2)))
    return WAN_ERR_MISALIGNED;
  const size_t bytes = (size_t)N * T * H * W * C * 2, cbytes = (size_t)N * 2 * H * W * C * 2;
  if (overlap(x, bytes, out, bytes) || overlap(cache1, cbytes, cache2, cbytes) || overlap(cache1, cbytes, out, bytes) ||
      overlap(cache2, cbytes, out, bytes) || overlap(cache1, cbytes, x, bytes) || overlap(cache2, cbytes, x, bytes))
    return WAN_ERR_INVALID_ARG;
  const size_t need = wan_workspace_size(WAN_OP_RESBLOCK_WINOGRAD, N, T, H, W, C, C, p->groups);
  if (!ws || ws_bytes < need) return WAN_ERR_WORKSPACE;
  if (!aligned16(ws)) return WAN_ERR_MISALIGNED;
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  char* base = static_cast<char*>(ws);
  wan_bf16* h = reinterpret_cast<wan_bf16*>(base);
  float4* coef = reinterpret_cast<float4*>(base + align256(bytes));
  char* stats = base + align256(bytes) + align256((size_t)N * T * C * 16);
  const bool chain = wino_gn_stats_supported(C, p->groups);  // h's statistics from conv 1
  const size_t stats_bytes = chain ? wino_gn_stats_bytes(N, T, H, W, p->groups) : 0;
  void* gws = stats + align256(stats_bytes);
  void* wws = static_cast<char*>(gws) + align256(gn_silu_workspace(N, T, H, W, C, p->groups, sms));
  const wan_bf16* c1_in = cache_valid ? cache1 : nullptr;
  const wan_bf16* c2_in = cache_valid ? cache2 : nullptr;
  // Each norm's coefficients, the Winograd conv applying them to its input tiles, then the
  // norm's last two frames into that conv's cache (after the conv has read the old ones). The
  // second norm's coefficients come from the statistics conv 1's output transform wrote with h.
  cudaError_t e = gn_silu_launch(x, nullptr, p->gamma1, p->beta1, N, T, H, W, C, p->groups, p->eps, gws, sms, s,
                                 false, coef);
  if (e == cudaSuccess)
    e = wino_conv_launch(x, coef, c1_in, u1, p->b1, nullptr, h, N, T, H, W, C, C, wws, sms, err, s, nullptr,
                         chain ? stats : nullptr, p->groups);
  if (e == cudaSuccess) e = gn_cache_update(x, coef, c1_in, cache1, N, T, H, W, C, sms, s);
  if (e == cudaSuccess)
    e = chain ? gn_coef_from_stats_launch(stats, stats_bytes, p->gamma2, p->beta2, N, T, H, W, C, p->groups, p->eps,
                                          coef, true, err, s)
              : gn_silu_launch(h, nullptr, p->gamma2, p->beta2, N, T, H, W, C, p->groups, p->eps, gws, sms, s, false,
                               coef);
  if (e == cudaSuccess) e = wino_conv_launch(h, coef, c2_in, u2, p->b2, x, out, N, T, H, W, C, C, wws, sms, err, s);
  if (e == cudaSuccess) e = gn_cache_update(h, coef, c2_in, cache2, N, T, H, W, C, sms, s);
  return cuda_status(e);
}

wan_status wan_device_status(void* stream) {
  WAN_CALL_RANGE();
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return WAN_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return WAN_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return WAN_ERR_CUDA;
    return (v & ~kDevErrBadStats) ? WAN_ERR_TIMEOUT : WAN_ERR_INVALID_ARG;
  }
  return WAN_OK;
}

}  // extern "C"
