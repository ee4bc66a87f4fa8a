"""fp64 numpy oracle of the causal video-VAE decoder hot path (test infrastructure only).

Tensor conventions (the pages' channels-last video layout, NDHWC):
  activations  [N, T, H, W, C]       bf16 bit patterns (uint16) at the boundary
  conv weights [Cout, 3, 3, 3, Cin]  (kt, kh, kw) taps, bf16 bits
  GN gamma/beta [C]                  fp32
  conv bias    [Cout]                bf16 bits
  3x3 weights  [Cout, 3, 3, Cin]     bf16 bits (the spatial conv of the upsampler)
  phase weights [4, Cout, 2, 2, Cin] bf16 bits, phase p = 2a + b for output row parity a and
                                     column parity b
Inside each operation the oracle computes in fp64 and rounds once, directly from fp64 to bf16
(round to nearest, ties to even), wherever the library writes a bf16 tensor.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "round_to_bf16", "bf16_to_f64", "bf16_to_f32", "ulp_distance_bf16",
    "silu_f64", "gn_silu_f64", "gn_silu",
    "causal_conv3d_f64", "causal_conv3d", "causal_conv3d_products_f64", "conv_at_points_f64",
    "resblock", "conv1x1", "fold_bias", "resblock_shortcut",
    "time_upsample_f64", "time_upsample",
    "phase_tap_sources", "phase_weights", "phase_weights_f64",
    "phase_conv_f64", "phase_conv", "upsample_nearest_conv_f64", "upsample_nearest_conv",
    "f32_to_f16_bits", "f16_to_f64", "winograd_weights", "winograd_weights_f64", "winograd_causal_conv3d_f64",
]

_BF16_OVERFLOW = 2.0 ** 128  # |value| rounded to 2^128 or above is out of bf16 range


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def round_to_bf16(x) -> np.ndarray:
    """fp64 -> bf16 bits with ONE rounding (nearest, ties to even), not via fp32.

    bf16 keeps 8 significant bits and fp32's exponent range: a finite x = m 2^e (0.5 <= |m| < 1)
    is rounded to a multiple of 2^(e-8), or of 2^-133 (the subnormal spacing) below 2^-126.
    Results of magnitude 2^128 or more become infinities; NaN becomes the quiet NaN 0x7FC0."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    step = np.maximum(e - 8, -133)
    q = np.round(np.ldexp(x, -step))          # exact scaling by a power of two, then RNE
    val = np.ldexp(q, step)
    val = np.where(np.abs(val) >= _BF16_OVERFLOW, np.copysign(np.inf, x), val)
    with np.errstate(over="ignore", invalid="ignore"):
        f32 = val.astype(np.float32)            # exact: val has <= 8 significant bits
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return np.where(np.isnan(x), np.uint16(0x7FC0), bits)


def ulp_distance_bf16(a_bits, b_bits) -> np.ndarray:
    """Distance in bf16 units in the last place between two bf16 bit arrays: both are mapped to
    integers ordered like the reals (negative values mirrored, +0 and -0 equal)."""
    def ordered(bits):
        b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(ordered(a_bits) - ordered(b_bits))


# ----------------------------------------------------------------------------------------------
# GroupNorm + SiLU  (WanGP group_norm_silu.py: module docstring, `_group_stats`, `_apply_kernel`)
# ----------------------------------------------------------------------------------------------

def silu_f64(z) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + e^-z); written as z e^z / (1 + e^z) for z < 0 so that e^-z
    cannot overflow."""
    z = np.asarray(z, dtype=np.float64)
    ez = np.exp(-np.abs(z))
    return np.where(z >= 0, z / (1.0 + ez), z * ez / (1.0 + ez))


def gn_silu_f64(x, gamma, beta, groups: int, eps: float, whole_clip: bool = False) -> np.ndarray:
    """silu(group_norm(x)) in fp64, x float [N, T, H, W, C].

    Statistics are taken per (n, t, group) over the group's C/groups channels of all H*W pixels
    of one frame (the per-image GroupNorm of the pages applied to every frame); with whole_clip,
    per (n, group) over all T frames as well (GroupNorm of the whole N C T H W tensor). Two
    passes: m = sum(x)/L, var = sum((x - m)^2)/L (population variance, divided by the length L
    as the pages do), z = (x - m)/sqrt(var + eps) * gamma_c + beta_c, output silu(z)."""
    x = np.asarray(x, dtype=np.float64)
    N, T, H, W, C = x.shape
    assert C % groups == 0
    cg = C // groups
    L = H * W * cg * (T if whole_clip else 1)
    xg = x.reshape(N, T, H * W, groups, cg)
    axes = (1, 2, 4) if whole_clip else (2, 4)
    mean = xg.sum(axis=axes, keepdims=True) / L
    d = xg - mean
    var = (d * d).sum(axis=axes, keepdims=True) / L
    rstd = 1.0 / np.sqrt(var + float(eps))
    g = np.asarray(gamma, dtype=np.float64).reshape(groups, cg)
    b = np.asarray(beta, dtype=np.float64).reshape(groups, cg)
    z = d * rstd * g + b
    return silu_f64(z).reshape(N, T, H, W, C)


def gn_silu(x_bits, gamma, beta, groups: int, eps: float, whole_clip: bool = False) -> np.ndarray:
    """bf16 in, bf16 out: silu(group_norm(x)) rounded once."""
    return round_to_bf16(gn_silu_f64(bf16_to_f64(x_bits), gamma, beta, groups, eps, whole_clip))


# ----------------------------------------------------------------------------------------------
# Causal 3x3x3 convolution with the carried temporal cache  (binding.cpp, `Decoder::conv`)
# ----------------------------------------------------------------------------------------------

def _padded_input(a, cache):
    """P = [cache (2 frames, zeros if absent); a] along T, zero-padded by one pixel in H and W."""
    N, T, H, W, C = a.shape
    if cache is None:
        cache = np.zeros((N, 2, H, W, C), dtype=np.float64)
    p = np.concatenate([cache, a], axis=1)
    return np.pad(p, ((0, 0), (0, 0), (1, 1), (1, 1), (0, 0)))


def causal_conv3d_f64(a, w, bias=None, residual=None, cache=None) -> np.ndarray:
    """y[n,t,h,w,co] = bias[co] + residual[n,t,h,w,co]
                      + sum_{kt,kh,kw,ci} w[co,kt,kh,kw,ci] * P[n, t+kt, h+kh, w+kw, ci]
    with P from `_padded_input`: tap kt = 0 meets frame t-2 of the sequence, kt = 2 frame t
    (the conv of the front-padded input, as the decoder pads two history frames in front)."""
    a = np.asarray(a, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    N, T, H, W, _ = a.shape
    Co = w.shape[0]
    P = _padded_input(a, None if cache is None else np.asarray(cache, dtype=np.float64))
    y = np.zeros((N, T, H, W, Co), dtype=np.float64)
    for kt in range(3):
        for kh in range(3):
            for kw in range(3):
                win = P[:, kt:kt + T, kh:kh + H, kw:kw + W, :]
                y += win @ w[:, kt, kh, kw, :].T
    if bias is not None:
        y += np.asarray(bias, dtype=np.float64)
    if residual is not None:
        y += np.asarray(residual, dtype=np.float64)
    return y


def causal_conv3d(a_bits, w_bits, bias_bits=None, residual_bits=None, cache_bits=None):
    """bf16 causal conv: returns (y bits rounded once, cache_out bits).

    cache_out holds the last two frames of [cache_in; a] (the conv's padded input history that
    the next chunk continues from), bit-for-bit copies."""
    a = bf16_to_f64(a_bits)
    cache = None if cache_bits is None else bf16_to_f64(cache_bits)
    y = causal_conv3d_f64(a, bf16_to_f64(w_bits),
                          None if bias_bits is None else bf16_to_f64(bias_bits),
                          None if residual_bits is None else bf16_to_f64(residual_bits),
                          cache)
    N, T, H, W, C = np.asarray(a_bits).shape
    prev = np.zeros((N, 2, H, W, C), np.uint16) if cache_bits is None else np.asarray(cache_bits)
    cache_out = np.concatenate([prev, np.asarray(a_bits, dtype=np.uint16)], axis=1)[:, -2:]
    return round_to_bf16(y), np.ascontiguousarray(cache_out)


def causal_conv3d_products_f64(a, w, bias=None, residual=None, cache=None) -> np.ndarray:
    """The sum of causal_conv3d_f64 grouped by input frame, for convolutions with few output
    channels: every frame tau of the padded input P is contracted ONCE with the weights of all 27
    taps,
        Q_tau[h, w, (kt, kh, kw), co] = sum_ci P[n, tau, h, w, ci] * w[co, kt, kh, kw, ci],
    and each output adds its 27 shifted products in the definition's tap order,
        y[n, t, h, w, co] = sum_{kt, kh, kw} Q_{t+kt}[h+kh, w+kw, (kt, kh, kw), co] (+ bias + residual).
    The products and the order of the 27-term sum are those of the definition; only the contraction
    is one matrix product per frame with 27 * Cout columns instead of 27 with Cout."""
    a = np.asarray(a, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    N, T, H, W, Ci = a.shape
    Co = w.shape[0]
    P = _padded_input(a, None if cache is None else np.asarray(cache, dtype=np.float64))
    w_all = w.reshape(Co, 27, Ci).transpose(1, 0, 2).reshape(27 * Co, Ci)  # row tap * Co + co
    y = np.zeros((N, T, H, W, Co), dtype=np.float64)
    for n in range(N):
        Q = {}
        for tau in range(T + 2):
            Q[tau] = (P[n, tau].reshape(-1, Ci) @ w_all.T).reshape(H + 2, W + 2, 27, Co)
            t = tau - 2  # the output frame whose last input frame is tau
            if t < 0:
                continue
            for kt in range(3):
                for kh in range(3):
                    for kw in range(3):
                        tap = (kt * 3 + kh) * 3 + kw
                        y[n, t] += Q[t + kt][kh:kh + H, kw:kw + W, tap, :]
            del Q[t]
    if bias is not None:
        y += np.asarray(bias, dtype=np.float64)
    if residual is not None:
        y += np.asarray(residual, dtype=np.float64)
    return y


def conv_at_points_f64(patches, w, bias=None, residual=None) -> np.ndarray:
    """The same sum at isolated output points: patches [P, 3, 3, 3, Cin] are the padded-input
    neighbourhoods P[t:t+3, h:h+3, w:w+3] of each point; returns [P, Cout] in fp64."""
    patches = np.asarray(patches, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    y = patches.reshape(patches.shape[0], -1) @ w.reshape(w.shape[0], -1).T
    if bias is not None:
        y += np.asarray(bias, dtype=np.float64)
    if residual is not None:
        y += np.asarray(residual, dtype=np.float64)
    return y


# ----------------------------------------------------------------------------------------------
# Causal ResBlock  (binding.cpp, `Decoder::resnet`)
# ----------------------------------------------------------------------------------------------

def resblock(x_bits, p: dict, groups: int, eps: float, cache1=None, cache2=None):
    """out = conv2(silu(gn2(h))) + x with h = conv1(silu(gn1(x))); each conv carries its own
    cache of its activated input. Every tensor the library writes in bf16 (the two activations,
    h and out) is rounded once here too. Returns (out, cache1_out, cache2_out)."""
    a1 = gn_silu(x_bits, p["gamma1"], p["beta1"], groups, eps)
    h, c1 = causal_conv3d(a1, p["w1"], p["b1"], None, cache1)
    a2 = gn_silu(h, p["gamma2"], p["beta2"], groups, eps)
    out, c2 = causal_conv3d(a2, p["w2"], p["b2"], x_bits, cache2)
    return out, c1, c2


# ----------------------------------------------------------------------------------------------
# Channel-changing ResBlock: the 1x1x1 shortcut with its bias folded into conv2's bias
# (binding.cpp, `prepare()`: the shortcut bias folded into the second conv's bias;
# `Decoder::resnet`: skip = conv(x, shortcut) without bias when the block changes channels)
# ----------------------------------------------------------------------------------------------

def conv1x1(x_bits, w_bits) -> np.ndarray:
    """skip[n,t,h,w,co] = sum_ci w[co,ci] x[n,t,h,w,ci], rounded once (the shortcut carries no
    bias of its own: it is folded into the second conv's)."""
    x = bf16_to_f64(x_bits)
    w = bf16_to_f64(w_bits)
    return round_to_bf16(x @ w.T)


def fold_bias(b2_bits, bsc_bits) -> np.ndarray:
    """b2 + b_shortcut, one bf16 rounding of the sum (prepare-time)."""
    return round_to_bf16(bf16_to_f64(b2_bits) + bf16_to_f64(bsc_bits))


def resblock_shortcut(x_bits, p: dict, w_sc, b_sc, groups: int, eps: float, cache1=None, cache2=None):
    """out = conv2(silu(gn2(h))) + b2' + skip with h = conv1(silu(gn1(x))) (Cin -> Cout),
    skip = conv1x1(x, w_sc) and b2' = fold_bias(b2, b_sc): the output is one rounding of
    acc2 + b2' + skip. Returns (out, cache1_out, cache2_out)."""
    a1 = gn_silu(x_bits, p["gamma1"], p["beta1"], groups, eps)
    h, c1 = causal_conv3d(a1, p["w1"], p["b1"], None, cache1)
    a2 = gn_silu(h, p["gamma2"], p["beta2"], groups, eps)
    skip = conv1x1(x_bits, w_sc)
    out, c2 = causal_conv3d(a2, p["w2"], fold_bias(p["b2"], b_sc), skip, cache2)
    return out, c1, c2


# ----------------------------------------------------------------------------------------------
# Causal 3x1x1 time upsample with frame-interleaved output (binding.cpp, `Decoder::up`: the
# frames after the first of the first chunk are padded in front with the cache (norm_pad's
# copy-only mode), the cache keeps the last two padded frames (`last_frames`), and
# time_upsample writes the x2 frames interleaved)
# ----------------------------------------------------------------------------------------------

def time_upsample_f64(x, w, bias=None, cache=None, first: bool = False) -> np.ndarray:
    """x [N, T, H, W, C], w [2C, 3, C] (kt, Cin), bias [2C]. With start = 1 if `first` (the
    first frame of the first chunk passes through) else 0, a = x[:, start:] (nf frames) and
    P = [cache (2 frames, zeros if absent); a]:
        z[n, t] = bias + sum_kt w[:, kt, :] . P[n, t + kt]      (2C channels, t < nf)
    and output frame start + 2t + i holds channels [i C, (i + 1) C) of z[n, t] (i = 0, 1).
    Returns out [N, start + 2 nf, H, W, C] in fp64."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    N, T, H, W, C = x.shape
    start = 1 if first else 0
    nf = T - start
    cache = np.zeros((N, 2, H, W, C)) if cache is None else np.asarray(cache, dtype=np.float64)
    P = np.concatenate([cache, x[:, start:]], axis=1)
    z = np.zeros((N, nf, H, W, 2 * C))
    for kt in range(3):
        z += P[:, kt:kt + nf] @ w[:, kt, :].T
    if bias is not None:
        z += np.asarray(bias, dtype=np.float64)
    out = np.zeros((N, start + 2 * nf, H, W, C))
    if first:
        out[:, 0] = x[:, 0]
    out[:, start::2] = z[..., :C]
    out[:, start + 1::2] = z[..., C:]
    return out


def time_upsample(x_bits, w_bits, bias_bits=None, cache_bits=None, first: bool = False):
    """bf16 time upsample: returns (out bits, rounded once; the passed-through frame is a copy,
    cache_out bits = the last two frames of P, copies)."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    out = time_upsample_f64(bf16_to_f64(x_bits), bf16_to_f64(w_bits),
                            None if bias_bits is None else bf16_to_f64(bias_bits),
                            None if cache_bits is None else bf16_to_f64(cache_bits), first)
    N, T, H, W, C = x_bits.shape
    start = 1 if first else 0
    prev = np.zeros((N, 2, H, W, C), np.uint16) if cache_bits is None else np.asarray(cache_bits, np.uint16)
    cache_out = np.concatenate([prev, x_bits[:, start:]], axis=1)[:, -2:]
    return round_to_bf16(out), np.ascontiguousarray(cache_out)


# ----------------------------------------------------------------------------------------------
# Nearest-x2 + 3x3 as four 2x2 phase convolutions  (binding.cpp, `prepare()` phase transform,
# and `Decoder::up` / resample_upsample)
# ----------------------------------------------------------------------------------------------

def phase_tap_sources(a: int, u: int) -> list:
    """The 3x3 kernel rows r that land on low-resolution offset u of output parity a.

    Output row 2i + a of the nearest-x2 image reads high-resolution row 2i + a + r - 1, which is
    low-resolution row i + floor((a + r - 1)/2) (the pages write the floor as -1 for a negative
    dy and dy/2 otherwise). Tap u of phase a sits at low-resolution offset u + a - 1, so it
    collects the rows r with floor((a + r - 1)/2) == u + a - 1. Columns follow the same rule."""
    out = []
    for r in range(3):
        dy = a + r - 1
        iy = -1 if dy < 0 else dy // 2
        if iy == u + a - 1:
            out.append(r)
    return out


def phase_weights(w3_bits) -> np.ndarray:
    """[Cout, 3, 3, Cin] bf16 -> [4, Cout, 2, 2, Cin] bf16: each phase tap is the fp32 sum of its
    source taps, added in the order the pages loop (r outer, c inner, starting from zero), then
    rounded once to bf16."""
    w = bf16_to_f32(w3_bits)
    Co, _, _, Ci = w.shape
    out = np.zeros((4, Co, 2, 2, Ci), dtype=np.float32)
    for a in range(2):
        for b in range(2):
            for u in range(2):
                for v in range(2):
                    s = np.zeros((Co, Ci), dtype=np.float32)
                    for r in phase_tap_sources(a, u):
                        for c in phase_tap_sources(b, v):
                            s = (s + w[:, r, c, :]).astype(np.float32)
                    out[2 * a + b, :, u, v, :] = s
    return round_to_bf16(out.astype(np.float64))


def phase_weights_f64(w3) -> np.ndarray:
    """The same transform with exact (fp64) sums, for the fp64 identity with the definition."""
    w = np.asarray(w3, dtype=np.float64)
    Co, _, _, Ci = w.shape
    out = np.zeros((4, Co, 2, 2, Ci), dtype=np.float64)
    for a in range(2):
        for b in range(2):
            for u in range(2):
                for v in range(2):
                    for r in phase_tap_sources(a, u):
                        for c in phase_tap_sources(b, v):
                            out[2 * a + b, :, u, v, :] += w[:, r, c, :]
    return out


def phase_conv_f64(x, wp, bias=None) -> np.ndarray:
    """y[n, t, 2i+a, 2j+b, co] = bias[co] + sum_{u,v,ci} wp[2a+b, co, u, v, ci]
                                  * x[n, t, i+a-1+u, j+b-1+v, ci]   (x zero outside the frame)."""
    x = np.asarray(x, dtype=np.float64)
    wp = np.asarray(wp, dtype=np.float64)
    N, T, H, W, _ = x.shape
    Co = wp.shape[1]
    xp = np.pad(x, ((0, 0), (0, 0), (1, 1), (1, 1), (0, 0)))
    y = np.zeros((N, T, 2 * H, 2 * W, Co), dtype=np.float64)
    for a in range(2):
        for b in range(2):
            acc = np.zeros((N, T, H, W, Co), dtype=np.float64)
            for u in range(2):
                for v in range(2):
                    # padded index (i + a - 1 + u) + 1
                    win = xp[:, :, a + u:a + u + H, b + v:b + v + W, :]
                    acc += win @ wp[2 * a + b, :, u, v, :].T
            y[:, :, a::2, b::2, :] = acc
    if bias is not None:
        y += np.asarray(bias, dtype=np.float64)
    return y


def phase_conv(x_bits, wp_bits, bias_bits=None) -> np.ndarray:
    return round_to_bf16(phase_conv_f64(bf16_to_f64(x_bits), bf16_to_f64(wp_bits),
                                        None if bias_bits is None else bf16_to_f64(bias_bits)))


def upsample_nearest_conv_f64(x, w3, bias=None) -> np.ndarray:
    """The definition: nearest-neighbour x2 in H and W, then a 3x3 convolution, zero padding 1."""
    x = np.asarray(x, dtype=np.float64)
    w3 = np.asarray(w3, dtype=np.float64)
    N, T, H, W, _ = x.shape
    Co = w3.shape[0]
    x2 = np.repeat(np.repeat(x, 2, axis=2), 2, axis=3)
    xp = np.pad(x2, ((0, 0), (0, 0), (1, 1), (1, 1), (0, 0)))
    y = np.zeros((N, T, 2 * H, 2 * W, Co), dtype=np.float64)
    for r in range(3):
        for c in range(3):
            y += xp[:, :, r:r + 2 * H, c:c + 2 * W, :] @ w3[:, r, c, :].T
    if bias is not None:
        y += np.asarray(bias, dtype=np.float64)
    return y


def upsample_nearest_conv(x_bits, w3_bits, bias_bits=None) -> np.ndarray:
    return round_to_bf16(upsample_nearest_conv_f64(bf16_to_f64(x_bits), bf16_to_f64(w3_bits),
                                                   None if bias_bits is None else bf16_to_f64(bias_bits)))


# ----------------------------------------------------------------------------------------------
# Winograd F(2x2, 3x3) variant of the spatial taps  (binding.cpp, `prepare()`: the Winograd weights
# of the up blocks, each component keeping the causal 3-tap temporal conv; `Decoder::conv`: only the
# spatial 3x3 convolutions use Winograd, the transformed input, one conv per component, and the
# epilogue that applies the output transform). Transform matrices: Lavin and Gray, "Fast
# Algorithms for Convolutional Neural Networks" (2016), F(2x2, 3x3):
#   Y = A^T [ (G g G^T) . (B^T d B) ] A  for a 4x4 input tile d and a 3x3 kernel g.
# ----------------------------------------------------------------------------------------------

WINO_BT = np.array([[1, 0, -1, 0], [0, 1, 1, 0], [0, -1, 1, 0], [0, 1, 0, -1]], dtype=np.float64)
WINO_G = np.array([[1, 0, 0], [0.5, 0.5, 0.5], [0.5, -0.5, 0.5], [0, 0, 1]], dtype=np.float64)
WINO_AT = np.array([[1, 1, 1, 0], [0, 1, -1, -1]], dtype=np.float64)


def f32_to_f16_bits(x) -> np.ndarray:
    """fp32 -> IEEE half bits, round to nearest even (numpy's conversion)."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_to_f64(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def winograd_weights(w_bits) -> np.ndarray:
    """[Cout, 3, 3, 3, Cin] bf16 -> [16, Cout, 3, Cin] fp16 bits: component (x, y) = 4 x + y of
    G g G^T for every temporal tap kt, i.e. the sum over the spatial taps (r, c) with a non-zero
    coefficient G[x, r] G[y, c] of coefficient * w[:, kt, r, c, :], formed in fp32 in the pages'
    order (r outer, c inner, from zero), then rounded once to fp16. The coefficients are 1, 1/2,
    1/4 with signs, so each product is exact and only the fp32 sums and the final rounding round."""
    w = bf16_to_f32(w_bits)
    Co, _, _, _, Ci = w.shape
    out = np.zeros((16, Co, 3, Ci), dtype=np.float32)
    for x in range(4):
        for y in range(4):
            s = np.zeros((Co, 3, Ci), dtype=np.float32)
            for r in range(3):
                for c in range(3):
                    k = WINO_G[x, r] * WINO_G[y, c]
                    if k != 0:
                        s = (s + np.float32(k) * w[:, :, r, c, :]).astype(np.float32)
            out[4 * x + y] = s
    return f32_to_f16_bits(out)


def winograd_weights_f64(w) -> np.ndarray:
    """The same transform with exact sums: [16, Cout, 3, Cin] fp64."""
    w = np.asarray(w, dtype=np.float64)
    return np.einsum("xr,oarci,yc->xyoai", WINO_G, w, WINO_G).reshape(16, w.shape[0], 3, w.shape[4])


def winograd_causal_conv3d_f64(a, u, bias=None, residual=None, cache=None, store=None) -> np.ndarray:
    """The causal 3x3x3 convolution through F(2x2, 3x3) on the spatial taps, with transformed
    weights u [16, Cout, 3, Cin] (fp64 values): per frame tau of P = [cache or zeros; a] and 2x2
    output tile (i, j), the 4x4 input tile d = P[tau, 2i-1 .. 2i+2, 2j-1 .. 2j+2] (zero outside the
    frame) is transformed to V = B^T d B (then passed through `store`, e.g. a rounding to fp16, if
    given); per component the products are summed over the temporal taps and channels,
        M[t, tile, xy, co] = sum_{kt, ci} u[xy, co, kt, ci] V[t + kt, tile, xy, ci],
    and Y = A^T M A gives the 2x2 outputs, + bias + residual, in fp64."""
    a = np.asarray(a, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    N, T, H, W, Ci = a.shape
    Co = u.shape[1]
    Ht, Wt = (H + 1) // 2, (W + 1) // 2
    cache = np.zeros((N, 2, H, W, Ci)) if cache is None else np.asarray(cache, dtype=np.float64)
    P = np.concatenate([cache, a], axis=1)
    Pp = np.zeros((N, T + 2, 2 * Ht + 2, 2 * Wt + 2, Ci))
    Pp[:, :, 1:H + 1, 1:W + 1] = P
    # d[n, tau, i, j, r, c, ci] = Pp[n, tau, 2i + r, 2j + c, ci]
    d = np.stack([np.stack([Pp[:, :, r:r + 2 * Ht:2, c:c + 2 * Wt:2] for c in range(4)], axis=4)
                  for r in range(4)], axis=4)
    V = np.einsum("xr,ntijrcz,yc->ntijxyz", WINO_BT, d, WINO_BT)
    if store is not None:
        V = store(V)
    V = V.reshape(N, T + 2, Ht, Wt, 16, Ci)
    M = np.zeros((N, T, Ht, Wt, 16, Co))
    for kt in range(3):
        M += np.einsum("ntijkz,koz->ntijko", V[:, kt:kt + T], u[:, :, kt, :])
    Y = np.einsum("ax,ntijxyo,by->ntiajbo", WINO_AT, M.reshape(N, T, Ht, Wt, 4, 4, Co), WINO_AT)
    y = Y.reshape(N, T, 2 * Ht, 2 * Wt, Co)[:, :, :H, :W]
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)
    if residual is not None:
        y = y + np.asarray(residual, dtype=np.float64)
    return y
