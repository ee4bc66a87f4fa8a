/*
 * wan.h - C ABI of the GB300 (sm_103a) causal video-VAE decoder hot path.
 *
 * What the library computes, and where the method is stated:
 *   - GroupNorm + SiLU with FP32 arithmetic and one rounding to bf16:
 *     WanGP, shared/kernels/group_norm_silu.py (module docstring; `_apply_kernel`).
 *   - The causal 3x3x3 convolution whose two leading frames come from a carried temporal
 *     cache, the cache update, bias and residual:
 *     FastVideo, wan22_vae_decode/solution/binding.cpp (`Decoder::conv`, `Decoder::resnet`).
 *   - Nearest-x2 + 3x3 convolution as four 2x2 phase convolutions, and the phase-weight
 *     transform: binding.cpp (`prepare()`, `Decoder::up`).
 *
 * Conventions shared by every entry point
 *   - bf16 tensors are passed as `wan_bf16*` (16-bit patterns of bfloat16 values) and are
 *     channels-last video tensors [N, T, H, W, C] (NDHWC), dense, C innermost.
 *   - Every pointer is a DEVICE pointer, owned by the caller, 16-byte aligned (else
 *     WAN_ERR_MISALIGNED). The library allocates no device memory: scratch comes from the
 *     caller's workspace `ws` of `ws_bytes` bytes (query the size with wan_workspace_size;
 *     too small -> WAN_ERR_WORKSPACE). Inputs are only read; outputs must not overlap inputs
 *     unless an argument says otherwise.
 *   - `stream` is a cudaStream_t (0 = the legacy default stream). Work is enqueued
 *     asynchronously on it; the call returns once the work is enqueued.
 *   - Arguments are validated on the host before anything is enqueued: a call that returns an
 *     error status has launched nothing and written nothing. A launch failure returns
 *     WAN_ERR_CUDA. Faults that happen later on the device surface at the caller's next
 *     synchronisation; kernels that give up a bounded wait record WAN_ERR_TIMEOUT in a device
 *     word read by wan_device_status().
 *   - Results are deterministic: the same inputs on the same GPU give the same bits, whatever
 *     the chunking of the frame axis (see wan_causal_conv3d).
 */
#ifndef WAN_H
#define WAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t wan_bf16;
typedef uint16_t wan_fp16;  /* 16-bit patterns of IEEE half-precision values */

typedef enum wan_status {
  WAN_OK = 0,
  WAN_ERR_INVALID_ARG = 1,       /* null pointer, non-positive size, groups not dividing C ... */
  WAN_ERR_UNSUPPORTED_SHAPE = 2, /* a size this library has no kernel for (see each call) */
  WAN_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned */
  WAN_ERR_WORKSPACE = 4,         /* ws is NULL or ws_bytes below wan_workspace_size() */
  WAN_ERR_CUDA = 5,              /* a CUDA runtime call or kernel launch failed */
  WAN_ERR_TIMEOUT = 6            /* a kernel gave up a bounded wait (wan_device_status) */
} wan_status;

typedef enum wan_op {
  WAN_OP_GN_SILU = 0,
  WAN_OP_CAUSAL_CONV3D = 1,
  WAN_OP_RESBLOCK = 2,
  WAN_OP_UPSAMPLE_PHASE_CONV = 3,
  WAN_OP_GN_STATS = 4,           /* statistics buffer of wan_causal_conv3d_gn_stats (Cout, groups) */
  WAN_OP_GN_SILU_CONV3D = 5,     /* wan_gn_silu_causal_conv3d (Cin, Cout, groups) */
  WAN_OP_RESBLOCK_SHORTCUT = 6,  /* wan_resblock_shortcut (Cin, Cout, groups) */
  WAN_OP_WINOGRAD_CONV3D = 7,    /* wan_causal_conv3d_winograd (Cin, Cout) */
  WAN_OP_RESBLOCK_WINOGRAD = 8,  /* wan_resblock_winograd (Cin = C, groups) */
  WAN_OP_GN_STATS_WINOGRAD = 9   /* statistics buffer of wan_causal_conv3d_winograd_stats (Cout, groups) */
} wan_op;

/* Human-readable name of a status (static storage, never NULL). */
const char* wan_status_string(wan_status status);

/* Bytes of workspace `ws` the call `op` needs for these sizes (0 if it needs none).
 * Arguments that an op does not use are ignored (e.g. Cout and groups for the conv). */
size_t wan_workspace_size(wan_op op, int N, int T, int H, int W, int Cin, int Cout, int groups);

/*
 * y = silu(group_norm(x)), rounded once to bf16.
 *
 * Source: WanGP group_norm_silu.py (module docstring, `_group_stats`, `_apply_kernel`).
 * Statistics are per (n, t, group): each frame of the video is normalised as the pages'
 * NCHW image, over its C/groups channels of all H*W pixels; mean and POPULATION variance
 * (divided by the element count), eps inside the square root:
 *     z = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c],   y = z * sigmoid(z).
 * The statistics are accumulated with error-free (two-sum) fp32 partials per pixel span and
 * merged in a fixed order, so they stay exact however large the mean is against the spread.
 *
 *   x, y         [N, T, H, W, C] bf16, device; y may not overlap x.
 *   gamma, beta  [C] fp32, device.
 *   groups       divides C; C % 8 == 0; C <= 2048; (C/groups) % 8 == 0 or 8 % (C/groups) == 0.
 *   eps          > 0.
 *   ws           >= wan_workspace_size(WAN_OP_GN_SILU, N, T, H, W, C, 0, groups) bytes.
 * Values are supported for |x| < 2^60 (the squares of deviations stay finite in fp32).
 */
wan_status wan_gn_silu(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta,
                       int N, int T, int H, int W, int C, int groups, float eps,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * wan_gn_silu_clip: wan_gn_silu with the statistics of each (n, group) taken over the whole clip,
 * all T frames of n together (the GroupNorm of an N C T H W video as PyTorch computes it), where
 * wan_gn_silu takes them per frame.
 *   Same arguments, workspace and limits as wan_gn_silu, and H * W * C / groups < 2^24 (else
 *   WAN_ERR_UNSUPPORTED_SHAPE).
 *   Unlike the per-frame norm, the result depends on every frame of the clip, so a video split
 *   into chunks does not give the bits of one call over the whole video.
 */
wan_status wan_gn_silu_clip(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta,
                            int N, int T, int H, int W, int C, int groups, float eps,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * wan_gn_silu for callers that cannot allocate device memory. (The pages have no counterpart:
 * this is an interface of this library only.)
 *
 * Some hosts give a library only the tensors it works on: an application that has reserved all
 * device memory for its own pool and offers plug-ins no allocator, or a latency-bound loop that
 * may not call cudaMalloc and cannot hand over a workspace either. This call computes exactly
 * what wan_gn_silu computes, with the same kernels, but takes no workspace: its scratch is a
 * fixed 4 MiB array in the library's device memory, which every GPU that loads the library holds
 * until the process exits. The call allocates nothing.
 *   - Sizes whose scratch exceeds 4 MiB are refused with WAN_ERR_WORKSPACE (nothing is
 *     launched). The scratch needed is wan_workspace_size(WAN_OP_GN_SILU, ...); for example
 *     [1, 4, 88, 156, 512] with 32 groups needs about 0.45 MiB.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current, and keeps it for the life of the process; make that first call
 *     before any stream capture. After cudaDeviceReset() of a device the kept address is stale:
 *     do not call this entry point on that device again in the same process.
 *   - All calls share the one array: calls that may overlap on the GPU (on different streams,
 *     or from different threads without ordering) race on it and must be serialised by the
 *     caller. Each call clears, on its stream, the one scratch word that must start at zero
 *     (a grid-barrier counter) and writes every other word before reading it, so the array
 *     needs no clearing by the caller between calls.
 * Arguments and their conditions are those of wan_gn_silu.
 */
wan_status wan_gn_silu_noalloc(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta,
                               int N, int T, int H, int W, int C, int groups, float eps,
                               void* stream);

/*
 * Causal 3x3x3 convolution with a carried two-frame temporal cache (implicit GEMM on the
 * tcgen05 tensor cores, bf16 operands, fp32 accumulation, one rounding to bf16).
 *
 * Source: binding.cpp, `Decoder::conv` (the padded input is the cache frames followed by the
 * chunk; the cache then keeps the last two frames of that padded input) and `Decoder::resnet`.
 *     P = [cache_in (2 frames, or zeros if cache_in == NULL); a]   along T, per batch item,
 *     y[n,t,h,w,co] = bias[co] + residual[n,t,h,w,co]
 *                   + sum_{kt,kh,kw,ci} w[co,kt,kh,kw,ci] * P[n, t+kt, h+kh-1, w+kw-1, ci]
 * with P zero outside the frame in H and W (padding 1). Tap kt = 2 is the current frame.
 * cache_out (if not NULL) receives the last two frames of P, bit-for-bit: calling this on
 * consecutive chunks of a video with cache_out of one call passed as cache_in of the next
 * gives the same bits as one call on the whole video.
 *
 *   a          [N, T, H, W, Cin] bf16.
 *   cache_in   [N, 2, H, W, Cin] bf16 or NULL (zero history: the first chunk).
 *   cache_out  [N, 2, H, W, Cin] bf16 or NULL; MAY alias cache_in (updated after the conv
 *              has read it); must not overlap a or y.
 *   w          [Cout, 3, 3, 3, Cin] bf16 (taps kt, kh, kw; Cin innermost).
 *   bias       [Cout] bf16 or NULL.   residual  [N, T, H, W, Cout] bf16 or NULL (may not
 *              overlap y).
 *   y          [N, T, H, W, Cout] bf16.
 *   Cin % 64 == 0; 1 <= Cout; Cout % 2 == 0.
 *   ws         unused by this version of the library (wan_workspace_size returns 0); may be NULL.
 */
wan_status wan_causal_conv3d(const wan_bf16* a, const wan_bf16* cache_in, wan_bf16* cache_out,
                             const wan_bf16* w, const wan_bf16* bias, const wan_bf16* residual,
                             wan_bf16* y, int N, int T, int H, int W, int Cin, int Cout,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * wan_causal_conv3d that also emits the GroupNorm statistics of its output y, so that the
 * GroupNorm + SiLU which follows it (wan_gn_silu_from_stats) needs no pass over y of its own.
 * The pages have no such call: their decoder reads the conv output again for its norm
 * (binding.cpp, `Decoder::resnet`); fusing the statistics into the producing conv is the
 * cross-op fusion the scope lists after the hot path itself.
 *
 * y and the cache are exactly those of wan_causal_conv3d with the same arguments. stats receives,
 * per (frame, group, 32-pixel quarter of a 128-pixel tile of the frame), the float-float sums of
 * d and d^2 of d = y - s over the quarter's pixels and the group's channels, s being one value of
 * the group there, with s and the count, and a header with the number of such parts; its exact layout is private to this library: pass it
 * unchanged to wan_gn_silu_from_stats or wan_gn_silu_coefficients_from_stats with the same N, T,
 * H, W, C = Cout and groups.
 *
 *   groups     GroupNorm groups of the following norm; Cout % 256 == 0, groups divides Cout and
 *              the channels per group are a power of two from 4 to 64 (else
 *              WAN_ERR_UNSUPPORTED_SHAPE).
 *   stats      device buffer of >= wan_workspace_size(WAN_OP_GN_STATS, N, T, H, W, Cin, Cout,
 *              groups) bytes, 16-byte aligned, owned by the caller; must not overlap the tensors.
 *   Other arguments as wan_causal_conv3d (its 12-channel head path does not emit statistics).
 */
wan_status wan_causal_conv3d_gn_stats(const wan_bf16* a, const wan_bf16* cache_in, wan_bf16* cache_out,
                                      const wan_bf16* w, const wan_bf16* bias, const wan_bf16* residual,
                                      wan_bf16* y, int N, int T, int H, int W, int Cin, int Cout,
                                      int groups, void* stats, size_t stats_bytes, void* stream);

/*
 * GroupNorm + SiLU of x (the definition of wan_gn_silu, per (n, t, group)) using the statistics
 * that wan_causal_conv3d_gn_stats (or wan_causal_conv3d_gn_input_stats) emitted when it wrote x:
 * the per-part sums are moved to one shift and added as float-float pairs in a fixed part order,
 * so the result depends only on x's frames (the same bits in any chunking of the video). y is
 * within one bf16 ulp of the exact (fp64, rounded once) GroupNorm + SiLU, like wan_gn_silu's.
 * A stats buffer not written for these sizes is reported by wan_device_status.
 *
 *   x, y, gamma, beta, groups, eps, ws  as wan_gn_silu (ws >= wan_workspace_size(WAN_OP_GN_SILU,
 *              N, T, H, W, C, 0, groups)).
 *   stats      the buffer filled by wan_causal_conv3d_gn_stats, wan_causal_conv3d_gn_input_stats or
 *              wan_causal_conv3d_winograd_stats for this x (Cout = C, same groups); stats_bytes at
 *              least the size that call required. Below the smallest size any of them writes for
 *              these sizes the call returns WAN_ERR_INVALID_ARG; a buffer whose header names more
 *              records than stats_bytes holds is reported by wan_device_status.
 */
wan_status wan_gn_silu_from_stats(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta,
                                  int N, int T, int H, int W, int C, int groups, float eps,
                                  const void* stats, size_t stats_bytes, void* ws, size_t ws_bytes,
                                  void* stream);

/*
 * The per-(frame, channel) coefficients of x's GroupNorm (those wan_gn_silu_coefficients computes
 * with a pass over x) from the statistics a conv emitted when it wrote x, for a following
 * wan_causal_conv3d_gn_input: the norm then reads nothing of x beyond what its conv reads. Per
 * (frame, group) the parts are moved to one shift and added as float-float pairs in a fixed
 * order (so the result depends only on x's frames), then the mean and variance follow in fp64 as
 * in wan_gn_silu. The coefficients are those of wan_gn_silu_coefficients up to the rounding of
 * the sums (a few units in the 24th bit).
 *
 *   stats, stats_bytes  as wan_gn_silu_from_stats (C, groups: the conv's Cout and groups).
 *   gamma, beta, eps    as wan_gn_silu.
 *   coef       N*T*C*16 bytes, 16-byte aligned, caller-owned: the coefficients, in the layout
 *              wan_gn_silu_coefficients writes.
 * A stats buffer not written for these sizes is reported by wan_device_status.
 */
wan_status wan_gn_silu_coefficients_from_stats(const void* stats, size_t stats_bytes, const float* gamma,
                                               const float* beta, int N, int T, int H, int W, int C, int groups,
                                               float eps, void* coef, void* stream);

/*
 * GroupNorm + SiLU feeding a causal conv, the pair that every ResBlock of the decoder runs twice:
 *     a = silu(group_norm(x));  y = conv(a; cache_in) + bias + residual;
 *     cache_out = the last two frames of [cache_in or zeros; a]
 * Source: binding.cpp, `Decoder::conv` (its input is either the producer's "prepared" edge or
 * `norm_pad`: norm + SiLU + causal padding from the cache, which then keeps the last frames of
 * that padded input) and `Decoder::resnet`. The definitions are wan_gn_silu's,
 * wan_causal_conv3d's and wan_cache_update's; y and cache_out are bit for bit what those three
 * calls return.
 * For Cout >= 256 a is never stored: the norm's pass over x writes per-(frame, channel)
 * coefficients only, the conv normalises each operand tile of x in shared memory as it arrives,
 * and the last two frames of a are written once into cache_out: by the conv itself when
 * cache_out is a buffer apart from cache_in, else by a pass after the conv.
 *
 *   x          [N, T, H, W, Cin] bf16 (the norm's input); gamma, beta, groups, eps as wan_gn_silu.
 *   cache_in   NULL (zero history) or [N, 2, H, W, Cin] bf16, already activated (a previous
 *              chunk's cache_out).
 *   cache_out  NULL or [N, 2, H, W, Cin] bf16 receiving the new history; may equal cache_in.
 *   w, bias, residual, y, Cout  as wan_causal_conv3d.
 *   ws         >= wan_workspace_size(WAN_OP_GN_SILU_CONV3D, N, T, H, W, Cin, Cout, groups)
 *              bytes, 16-byte aligned.
 * Errors as wan_gn_silu and wan_causal_conv3d; x, y and the caches may not overlap (except
 * cache_in == cache_out).
 */
wan_status wan_gn_silu_causal_conv3d(const wan_bf16* x, const float* gamma, const float* beta, int groups,
                                     float eps, const wan_bf16* cache_in, wan_bf16* cache_out,
                                     const wan_bf16* w, const wan_bf16* bias, const wan_bf16* residual,
                                     wan_bf16* y, int N, int T, int H, int W, int Cin, int Cout, void* ws,
                                     size_t ws_bytes, void* stream);

/*
 * The three steps of wan_gn_silu_causal_conv3d for Cout >= 256, as separate calls (a norm whose
 * output feeds more than one consumer computes its coefficients once):
 *   1. wan_gn_silu_coefficients: the per-(frame, channel) scale S and shift B of x's GroupNorm
 *      (gamma, beta, groups and eps folded in), so that silu(x S + B) is wan_gn_silu's output.
 *   2. wan_causal_conv3d_gn_input: y = conv(silu(x S + B); cache_in) + bias + residual, the
 *      normalisation applied to the conv's operand tiles as they arrive.
 *   3. wan_gn_silu_cache_update: cache_out = the last two frames of [cache_in or zeros;
 *      silu(x S + B)].
 * coef holds N*T*C*16 bytes (16-byte aligned, caller-owned) in a layout private to the library:
 * pass it unchanged between the calls with the same x, N, T, H, W and C. Each result is bit for
 * bit what the corresponding step of wan_gn_silu_causal_conv3d writes. C (Cin) % 64 == 0.
 *
 *   wan_gn_silu_coefficients  x, gamma, beta, groups, eps, ws as wan_gn_silu (ws >=
 *                             wan_workspace_size(WAN_OP_GN_SILU, ...)).
 *   wan_causal_conv3d_gn_input  cache_in (activated history, or NULL), w, bias, residual, y as
 *                             wan_causal_conv3d; Cout < 256 gives WAN_ERR_UNSUPPORTED_SHAPE.
 *                             cache_out (NULL, or [N, 2, H, W, Cin]) receives step 3's result: a
 *                             buffer apart from cache_in is written by the conv's operand
 *                             prologue from its normalised tiles (no pass of its own); cache_out
 *                             == cache_in is updated after the conv, as step 3 does.
 *   wan_gn_silu_cache_update  cache_out may equal cache_in; must not overlap x or coef.
 */
wan_status wan_gn_silu_coefficients(const wan_bf16* x, const float* gamma, const float* beta, int N, int T,
                                    int H, int W, int C, int groups, float eps, void* coef, void* ws,
                                    size_t ws_bytes, void* stream);
wan_status wan_causal_conv3d_gn_input(const wan_bf16* x, const void* coef, const wan_bf16* cache_in,
                                      wan_bf16* cache_out, const wan_bf16* w, const wan_bf16* bias,
                                      const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W, int Cin,
                                      int Cout, void* stream);
wan_status wan_gn_silu_cache_update(const wan_bf16* x, const void* coef, const wan_bf16* cache_in,
                                    wan_bf16* cache_out, int N, int T, int H, int W, int C, void* stream);

/*
 * wan_causal_conv3d_gn_input that also emits the GroupNorm statistics of its output y (as
 * wan_causal_conv3d_gn_stats does for wan_causal_conv3d), so that the norm of the next ResBlock
 * step gets its coefficients from wan_gn_silu_coefficients_from_stats without a pass over y.
 * y and cache_out are bit for bit those of wan_causal_conv3d_gn_input.
 *
 *   groups, stats, stats_bytes  as wan_causal_conv3d_gn_stats (Cout % 256 == 0, channels per
 *              group a power of two from 4 to 64; stats_bytes >= wan_workspace_size(
 *              WAN_OP_GN_STATS, N, T, H, W, Cin, Cout, groups)); stats must not overlap the other
 *              buffers.
 *   Other arguments as wan_causal_conv3d_gn_input.
 */
wan_status wan_causal_conv3d_gn_input_stats(const wan_bf16* x, const void* coef, const wan_bf16* cache_in,
                                            wan_bf16* cache_out, const wan_bf16* w, const wan_bf16* bias,
                                            const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W,
                                            int Cin, int Cout, int groups, void* stats, size_t stats_bytes,
                                            void* stream);

/*
 * Temporal-cache update (the cache manager of the causal convolutions), on its own.
 *
 * Source: binding.cpp, `Decoder::conv` (`cache[idx] = last_frames(p, ...)`: after a chunk the
 * cache keeps the last two frames of the conv's padded input P = [cache_in; a]):
 *     cache_out[n, j] = P[n, T + j],  j = 0, 1   (bit-for-bit copies; zeros where P comes
 *                                                from a NULL cache_in)
 * wan_causal_conv3d does this itself when given cache_out; this call is the same copy for
 * callers that schedule it separately (it must run after every reader of cache_in).
 *
 *   a          [N, T, H, W, C] bf16.      cache_in  [N, 2, H, W, C] bf16 or NULL.
 *   cache_out  [N, 2, H, W, C] bf16; MAY alias cache_in; must not overlap a.
 *   C % 8 == 0.
 */
wan_status wan_cache_update(const wan_bf16* a, const wan_bf16* cache_in, wan_bf16* cache_out,
                            int N, int T, int H, int W, int C, void* stream);

/*
 * Phase-weight transform of the nearest-x2 upsampler.
 *
 * Source: binding.cpp, `prepare()` (nearest-x2 + 3x3 equals four 2x2 low-resolution phases;
 * sums formed in fp32, stored in bf16). For output parity (a, b), phase p = 2a + b, and phase
 * tap (u, v):
 *     wp[p, co, u, v, ci] = bf16( sum over r in R(a,u), c in R(b,v) of fp32(w3[co, r, c, ci]) )
 * where R(a, u) = { r in 0..2 : floor((a + r - 1) / 2) == u + a - 1 }, added in the order r
 * outer, c inner, starting from zero, rounded once to nearest even.
 *
 *   w3  [Cout, 3, 3, Cin] bf16.    wp  [4, Cout, 2, 2, Cin] bf16 (may not overlap w3).
 */
wan_status wan_upsample_phase_weights(const wan_bf16* w3, wan_bf16* wp, int Cin, int Cout,
                                      void* stream);

/*
 * Nearest-x2 spatial upsample followed by a 3x3 convolution (padding 1), executed as four 2x2
 * phase convolutions on the low-resolution input, written interleaved into the output.
 *
 * Source: binding.cpp, `Decoder::up` (the four phase convolutions of the resampler) with the
 * weights of wan_upsample_phase_weights:
 *     y[n, t, 2i+a, 2j+b, co] = bias[co]
 *         + sum_{u,v,ci} wp[2a+b, co, u, v, ci] * x[n, t, i+a-1+u, j+b-1+v, ci]
 * with x zero outside the frame. bf16 operands, fp32 accumulation, one rounding.
 *
 *   x     [N, T, H, W, Cin] bf16.       wp  [4, Cout, 2, 2, Cin] bf16.
 *   bias  [Cout] bf16 or NULL.          y   [N, T, 2H, 2W, Cout] bf16.
 *   Cin % 64 == 0; Cout % 2 == 0.
 */
wan_status wan_upsample_phase_conv(const wan_bf16* x, const wan_bf16* wp, const wan_bf16* bias,
                                   wan_bf16* y, int N, int T, int H, int W, int Cin, int Cout,
                                   void* stream);

/* Parameters of one causal ResBlock (C -> C). All device pointers. */
typedef struct wan_resblock_params {
  const float* gamma1;   /* [C] fp32, GroupNorm 1 scale */
  const float* beta1;    /* [C] fp32, GroupNorm 1 shift */
  const wan_bf16* w1;    /* [C, 3, 3, 3, C] bf16, conv 1 */
  const wan_bf16* b1;    /* [C] bf16 or NULL */
  const float* gamma2;   /* [C] fp32 */
  const float* beta2;    /* [C] fp32 */
  const wan_bf16* w2;    /* [C, 3, 3, 3, C] bf16, conv 2 */
  const wan_bf16* b2;    /* [C] bf16 or NULL */
  int groups;            /* GroupNorm groups, divides C */
  float eps;             /* GroupNorm eps, > 0 */
} wan_resblock_params;

/*
 * One causal ResBlock on one chunk of frames:
 *     a1 = silu(gn1(x));  h = conv1(a1; cache1) + b1;
 *     a2 = silu(gn2(h));  out = conv2(a2; cache2) + b2 + x
 * Source: binding.cpp, `Decoder::resnet` (residual x, each conv with its own cache of its
 * activated input). a1, h and a2 are rounded to bf16 as the standalone calls round them.
 *
 *   x, out       [N, T, H, W, C] bf16; out may not overlap x.
 *   cache1/2     [N, 2, H, W, C] bf16, in/out (the history of conv 1 / conv 2's input).
 *   cache_valid  0: the caches' contents are ignored (zero history, the first chunk) and
 *                overwritten; 1: they hold the history left by the previous chunk.
 *   C % 64 == 0 and the GroupNorm conditions of wan_gn_silu.
 *   ws           >= wan_workspace_size(WAN_OP_RESBLOCK, N, T, H, W, C, C, groups) bytes.
 * Cost of the in/out caches: with cache_valid = 1 a conv must read the old history before the
 * new one replaces it, so each conv is followed by a pass that normalises its input's last two
 * frames into the cache again (about 5% of a C = 256 conv at 176 x 312). Where the caller keeps
 * two buffers per cache and swaps them, the steps of this call (wan_gn_silu_coefficients,
 * wan_causal_conv3d_gn_input with cache_out apart from cache_in) let the conv write the new
 * history itself, and the result is the same bits.
 */
wan_status wan_resblock(const wan_bf16* x, wan_bf16* out, const wan_resblock_params* p,
                        wan_bf16* cache1, wan_bf16* cache2, int cache_valid,
                        int N, int T, int H, int W, int C, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * The decoder steps next to the ResBlock (binding.cpp, `Decoder::up` and `Decoder::resnet`).
 *
 * wan_time_upsample: the causal 3x1x1 time convolution that doubles the frame rate, written
 * frame-interleaved. With start = 1 when `first` (the first chunk of a video: its first frame
 * passes through unchanged and is no part of the time conv's history) and 0 otherwise, the
 * frames x[:, start:] are padded in front with the two history frames (cache_in, zeros if NULL)
 * and convolved over time to 2C channels:
 *     z[n, t] = bias + sum_kt w[:, kt, :] . [history; x[:, start:]][n, t + kt]
 * and output frame start + 2t + i holds channels [iC, (i + 1)C) of z[n, t] (i = 0, 1).
 * Source: `Decoder::up` (the narrow to frames start.., norm_pad's copy-only padding with the
 * cache, last_frames, time_upsample writing the x2 frames interleaved); the channel-half order is
 * the plainest reading of "frame-interleaved", as no source of time_upsample is on the pages.
 *   x          [N, T, H, W, C] bf16, C % 256 == 0.
 *   w, bias    [2C, 3, C] (taps kt = 0..2 meet frames t-2..t) and [2C] (or NULL), bf16.
 *   y          [N, start + 2 (T - start), H, W, C] bf16.
 *   cache_in   NULL or [N, 2, H, W, C]; cache_out NULL or the same shape (may equal cache_in):
 *              the last two frames of [cache_in or zeros; x[:, start:]].
 *
 * wan_conv1x1: y = x . w^T per pixel (w [Cout, Cin] bf16, no bias), rounded once: the 1x1x1
 * shortcut of a channel-changing block. Cin % 64 == 0, Cout >= 256 and even.
 *
 * wan_fold_bias: out = b2 + b_shortcut (C values, bf16), rounded once: the shortcut's bias folded
 * into the block's second conv at prepare time (binding.cpp, prepare()), so the shortcut tensor
 * needs no bias pass of its own.
 *
 * wan_resblock_shortcut: the ResBlock whose output has Cout != Cin channels:
 *     h = conv1(silu(gn1(x)); cache1) + b1                       (Cin -> Cout)
 *     out = conv2(silu(gn2(h)); cache2) + p->b2 + conv1x1(x, w_sc)  (one rounding)
 * with p->b2 already folded (wan_fold_bias(b2, b_shortcut)). gamma1/beta1 have Cin values,
 * gamma2/beta2 Cout; w1 [Cout, 3, 3, 3, Cin], w2 [Cout, 3, 3, 3, Cout]; cache1 [N, 2, H, W, Cin],
 * cache2 [N, 2, H, W, Cout]. Cout >= 256. ws >= wan_workspace_size(WAN_OP_RESBLOCK_SHORTCUT, N,
 * T, H, W, Cin, Cout, groups). Source: `Decoder::resnet` (change = true: skip = conv(x,
 * shortcut) without bias).
 */
wan_status wan_time_upsample(const wan_bf16* x, const wan_bf16* cache_in, wan_bf16* cache_out,
                             const wan_bf16* w, const wan_bf16* bias, wan_bf16* y, int N, int T,
                             int H, int W, int C, int first, void* stream);
wan_status wan_conv1x1(const wan_bf16* x, const wan_bf16* w, wan_bf16* y, int N, int T, int H, int W,
                       int Cin, int Cout, void* stream);
wan_status wan_fold_bias(const wan_bf16* b2, const wan_bf16* b_shortcut, wan_bf16* out, int C,
                         void* stream);
wan_status wan_resblock_shortcut(const wan_bf16* x, wan_bf16* out, const wan_resblock_params* p,
                                 const wan_bf16* w_sc, wan_bf16* cache1, wan_bf16* cache2,
                                 int cache_valid, int N, int T, int H, int W, int Cin, int Cout,
                                 void* ws, size_t ws_bytes, void* stream);

/*
 * The causal 3x3x3 convolution with its spatial 3x3 taps through Winograd F(2x2, 3x3), fp16
 * transformed operands, fp32 accumulation, one rounding to bf16.
 *
 * Source: binding.cpp, `prepare()` (the Winograd weights G g G^T, each component keeping the
 * causal 3-tap temporal convolution, summed in fp32) and `Decoder::conv` (only the spatial 3x3
 * convolutions use Winograd: the padded input transformed once, one convolution per component,
 * an epilogue applying the output transform with bias and residual). Transforms: Lavin and Gray
 * (2016), Y = A^T [(G g G^T) . (B^T d B)] A. The pages run F(4x4, 3x3) with bf16 operands; this
 * library runs F(2x2, 3x3) with fp16 operands, whose error equals the direct conv's (F(4x4) with
 * bf16 operands has about 15 times it). The result is that of wan_causal_conv3d within the conv
 * tolerance, not bit for bit; it does not depend on the chunking of the frames.
 *
 * wan_winograd_weights: u[xy][co][kt][ci] (component xy = 4 x + y of 16) = fp16 of
 *     sum over (r, c) with G[x][r] G[y][c] != 0 of G[x][r] G[y][c] w[co][kt][r][c][ci],
 *   G = [[1,0,0],[1/2,1/2,1/2],[1/2,-1/2,1/2],[0,0,1]], summed in fp32 in the order r outer, c inner,
 *   from zero (each product is exact), rounded once to nearest even. Once per weight set.
 *     w  [Cout, 3, 3, 3, Cin] bf16.   u  [16, Cout, 3, Cin] fp16 (16 * Cout * 3 * Cin values).
 *     Cin % 64 == 0, Cout % 256 == 0.
 *
 * wan_causal_conv3d_winograd: y = conv(A; cache_in) + bias + residual with the definition of
 *   wan_causal_conv3d, where A = silu(a S + B) if `coef` is given (the coefficients of a from
 *   wan_gn_silu_coefficients: the GroupNorm + SiLU applied to the conv's input as it is
 *   transformed) and A = a otherwise; cache_in holds already-activated frames (or NULL: zeros).
 *   cache_out (NULL or [N, 2, H, W, Cin], may equal cache_in) receives the last two frames of
 *   [cache_in or zeros; A] bit for bit as wan_gn_silu_cache_update / wan_cache_update write them
 *   (apart from cache_in it is written by the input transform, in place by a pass after the conv).
 *     u     from wan_winograd_weights.   Cin % 64 == 0, Cin <= 2048, Cout % 256 == 0.
 *     ws    >= wan_workspace_size(WAN_OP_WINOGRAD_CONV3D, N, T, H, W, Cin, Cout, 0) bytes: the
 *           transformed input (16 N (T + 2) ceil(H/2) ceil(W/2) Cin fp16) and the component
 *           products (16 N T ceil(H/2) ceil(W/2) Cout fp32); may not overlap the tensors.
 *   Values: the transformed input and weights must fit fp16 (|values| below about 16000 at the
 *   input, which GroupNorm + SiLU outputs are for any gamma, beta of moderate size).
 *
 * wan_causal_conv3d_winograd_stats: wan_causal_conv3d_winograd (y and cache_out bit for bit the
 *   same) whose output transform also writes the GroupNorm statistics of y for `groups` groups:
 *   per (frame, group, 2x2 output tile) the float-float sums of d and d^2 of d = y - s over the
 *   tile's pixels and the group's channels, s being one value of the group there, with s and the
 *   count, and a header with the number of tiles. As with wan_causal_conv3d_gn_stats the layout
 *   is private: pass the buffer to wan_gn_silu_from_stats or wan_gn_silu_coefficients_from_stats
 *   with the same N, T, H, W, C = Cout and groups.
 *     groups  divides Cout; the channels per group are a power of two from 4 to 64 (else
 *             WAN_ERR_UNSUPPORTED_SHAPE).
 *     stats   >= wan_workspace_size(WAN_OP_GN_STATS_WINOGRAD, N, T, H, W, Cin, Cout, groups) bytes,
 *             16-byte aligned, caller-owned; it may not overlap the tensors, coef or ws.
 *
 * wan_resblock_winograd: wan_resblock with both convolutions through Winograd (u1, u2 from
 *   wan_winograd_weights of w1, w2; p->w1 and p->w2 are not read). Same definition, caches and
 *   conditions as wan_resblock, and C % 256 == 0. The second norm's coefficients come from the
 *   statistics conv 1 writes with h (as wan_gn_silu_coefficients_from_stats computes them) when
 *   C / groups is a power of two from 4 to 64, else from a pass over h.
 *     ws  >= wan_workspace_size(WAN_OP_RESBLOCK_WINOGRAD, N, T, H, W, C, C, groups) bytes.
 */
wan_status wan_winograd_weights(const wan_bf16* w, wan_fp16* u, int Cin, int Cout, void* stream);
wan_status wan_causal_conv3d_winograd(const wan_bf16* a, const void* coef, const wan_bf16* cache_in,
                                      wan_bf16* cache_out, const wan_fp16* u, const wan_bf16* bias,
                                      const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W,
                                      int Cin, int Cout, void* ws, size_t ws_bytes, void* stream);
wan_status wan_causal_conv3d_winograd_stats(const wan_bf16* a, const void* coef, const wan_bf16* cache_in,
                                            wan_bf16* cache_out, const wan_fp16* u, const wan_bf16* bias,
                                            const wan_bf16* residual, wan_bf16* y, int N, int T, int H, int W,
                                            int Cin, int Cout, int groups, void* stats, size_t stats_bytes,
                                            void* ws, size_t ws_bytes, void* stream);
wan_status wan_resblock_winograd(const wan_bf16* x, wan_bf16* out, const wan_resblock_params* p,
                                 const wan_fp16* u1, const wan_fp16* u2, wan_bf16* cache1, wan_bf16* cache2,
                                 int cache_valid, int N, int T, int H, int W, int C, void* ws,
                                 size_t ws_bytes, void* stream);

/*
 * Self-test of the failure detection of the bounded device waits (the pages have no counterpart:
 * the waits and their error word belong to this library). It makes a wait run out on purpose, with
 * a short bound, so that a caller can check that the kernel gives up, winds down and reports
 * WAN_ERR_TIMEOUT through wan_device_status(), and that the next calls work normally.
 *   which = 0  wan_gn_silu's cooperative kernel on the given tensors, with its first grid
 *              barrier set one arrival beyond what the grid can give: every CTA waits
 *              `wait_cycles` SM cycles, records the timeout and returns; y is not written.
 *              The other arguments, their checks and errors are wan_gn_silu's.
 *   which = 1  one thread waits on an mbarrier (the tensor-core pipelines' wait) that never
 *              completes; the tensor and workspace arguments are ignored (may be NULL).
 *   wait_cycles  the bound, 1e3 .. 1e8 SM cycles (at most ~50 ms), else WAN_ERR_INVALID_ARG.
 * Nothing faults and nothing waits without bound.
 */
wan_status wan_selftest_wait_timeout(int which, long long wait_cycles, const wan_bf16* x, wan_bf16* y,
                                     const float* gamma, const float* beta, int N, int T, int H, int W,
                                     int C, int groups, float eps, void* ws, size_t ws_bytes, void* stream);

/*
 * Synchronises `stream`, then reads and clears the library's device error word on the
 * current device. Returns WAN_ERR_TIMEOUT if a kernel gave up a bounded wait since the last
 * call, else WAN_ERR_INVALID_ARG if a statistics buffer given to wan_gn_silu_from_stats or
 * wan_gn_silu_coefficients_from_stats did not hold statistics of the call's sizes (the
 * coefficients were then not written), WAN_ERR_CUDA if the synchronisation failed, else WAN_OK.
 */
wan_status wan_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* WAN_H */
