"""Pins of the oracle's causal 3x3x3 convolution, cache and ResBlock."""
import numpy as np
import torch

from oracle import (causal_conv3d, causal_conv3d_f64, causal_conv3d_products_f64, conv_at_points_f64,
                    resblock, bf16_to_f64, round_to_bf16)
from video_vae_decoder_gb300 import synth


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).normal(0, scale, size=shape)


def test_matches_torch_conv3d_on_front_padded_input():
    N, T, H, W, Ci, Co = 1, 4, 5, 6, 8, 12
    a = _rand((N, T, H, W, Ci), 1)
    cache = _rand((N, 2, H, W, Ci), 2)
    w = _rand((Co, 3, 3, 3, Ci), 3, 0.1)
    bias = _rand((Co,), 4)
    res = _rand((N, T, H, W, Co), 5)
    ours = causal_conv3d_f64(a, w, bias, res, cache)
    seq = np.concatenate([cache, a], axis=1)                       # [N, T+2, H, W, Ci]
    xt = torch.from_numpy(seq).permute(0, 4, 1, 2, 3)               # NCDHW
    wt = torch.from_numpy(w).permute(0, 4, 1, 2, 3)                 # [Co, Ci, 3, 3, 3]
    ref = torch.nn.functional.conv3d(xt, wt, torch.from_numpy(bias), padding=(0, 1, 1))
    ref = ref.permute(0, 2, 3, 4, 1).numpy() + res
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)


def test_brute_force_points():
    N, T, H, W, Ci, Co = 1, 3, 4, 4, 3, 2
    a = _rand((N, T, H, W, Ci), 6)
    w = _rand((Co, 3, 3, 3, Ci), 7)
    ours = causal_conv3d_f64(a, w)
    for (t, h, x, co) in [(0, 0, 0, 0), (2, 3, 3, 1), (1, 2, 0, 1), (2, 0, 3, 0)]:
        s = 0.0
        for kt in range(3):
            for kh in range(3):
                for kw in range(3):
                    tt, hh, ww = t + kt - 2, h + kh - 1, x + kw - 1
                    if tt < 0 or not (0 <= hh < H) or not (0 <= ww < W):
                        continue      # zero cache in front, zero padding around the frame
                    for ci in range(Ci):
                        s += w[co, kt, kh, kw, ci] * a[0, tt, hh, ww, ci]
        assert abs(ours[0, t, h, x, co] - s) < 1e-12


def test_identity_and_causal_taps():
    N, T, H, W, C = 1, 3, 4, 5, 4
    a = _rand((N, T, H, W, C), 8)
    cache = _rand((N, 2, H, W, C), 9)
    w = np.zeros((C, 3, 3, 3, C))
    w[:, 2, 1, 1, :] = np.eye(C)          # current frame, centre pixel
    np.testing.assert_array_equal(causal_conv3d_f64(a, w, cache=cache), a)
    w = np.zeros((C, 3, 3, 3, C))
    w[:, 0, 1, 1, :] = np.eye(C)          # two frames back: the cache for t = 0, 1
    y = causal_conv3d_f64(a, w, cache=cache)
    np.testing.assert_array_equal(y[:, 0], cache[:, 0])
    np.testing.assert_array_equal(y[:, 1], cache[:, 1])
    np.testing.assert_array_equal(y[:, 2], a[:, 0])
    w = np.zeros((C, 3, 3, 3, C))
    w[:, 2, 0, 2, :] = np.eye(C)          # up one row, right one column, zero outside
    y = causal_conv3d_f64(a, w)
    np.testing.assert_array_equal(y[:, :, 1:, :-1], a[:, :, :-1, 1:])
    assert not y[:, :, 0, :].any() and not y[:, :, :, -1].any()


def test_linearity():
    a1 = _rand((1, 2, 3, 3, 4), 10)
    a2 = _rand((1, 2, 3, 3, 4), 11)
    w = _rand((5, 3, 3, 3, 4), 12)
    lhs = causal_conv3d_f64(2.0 * a1 - 3.0 * a2, w)
    rhs = 2.0 * causal_conv3d_f64(a1, w) - 3.0 * causal_conv3d_f64(a2, w)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


def test_points_match_full():
    N, T, H, W, Ci, Co = 1, 3, 4, 5, 6, 7
    a = _rand((N, T, H, W, Ci), 13)
    cache = _rand((N, 2, H, W, Ci), 14)
    w = _rand((Co, 3, 3, 3, Ci), 15)
    b = _rand((Co,), 16)
    full = causal_conv3d_f64(a, w, b, cache=cache)
    P = np.pad(np.concatenate([cache, a], 1), ((0, 0), (0, 0), (1, 1), (1, 1), (0, 0)))
    pts = [(0, 0, 0), (2, 3, 4), (1, 1, 2)]
    patches = np.stack([P[0, t:t + 3, h:h + 3, x:x + 3] for t, h, x in pts])
    got = conv_at_points_f64(patches, w, b)
    for i, (t, h, x) in enumerate(pts):
        np.testing.assert_allclose(got[i], full[0, t, h, x], rtol=1e-12, atol=1e-12)


def test_chunked_equals_unchunked_conv():
    # The history crosses chunks in the cache, so the result does not depend on the chunk size.
    N, T, H, W, C = 1, 6, 4, 4, 8
    ab = synth.normal_bf16((N, T, H, W, C), 0, "t/chunk/a")
    wb = synth.normal_bf16((C, 3, 3, 3, C), 0, "t/chunk/w", 0, 0.1)
    full, cache_full = causal_conv3d(ab, wb)
    parts, cache = [], None
    for s in (0, 2, 3, 5):           # ragged chunks: 2, 1, 2, 1 frames
        e = {0: 2, 2: 3, 3: 5, 5: 6}[s]
        y, cache = causal_conv3d(ab[:, s:e], wb, cache_bits=cache)
        parts.append(y)
    np.testing.assert_array_equal(np.concatenate(parts, axis=1), full)
    np.testing.assert_array_equal(cache, cache_full)
    np.testing.assert_array_equal(cache_full, ab[:, -2:])


def test_chunked_equals_unchunked_resblock():
    C, G = 16, 8
    p = synth.resblock_params(C, 0, "t/rb")
    x = synth.normal_bf16((1, 6, 4, 5, C), 0, "t/rb/x")
    full, c1f, c2f = resblock(x, p, G, 1e-6)
    outs, c1, c2 = [], None, None
    for s, e in ((0, 3), (3, 4), (4, 6)):
        o, c1, c2 = resblock(x[:, s:e], p, G, 1e-6, c1, c2)
        outs.append(o)
    np.testing.assert_array_equal(np.concatenate(outs, 1), full)
    np.testing.assert_array_equal(c1, c1f)
    np.testing.assert_array_equal(c2, c2f)


def test_cache_out_is_last_two_padded_input_frames_t1():
    C = 4
    a = synth.normal_bf16((1, 1, 2, 2, C), 0, "t/c1/a")
    cache = synth.normal_bf16((1, 2, 2, 2, C), 0, "t/c1/c")
    w = synth.normal_bf16((C, 3, 3, 3, C), 0, "t/c1/w")
    _, out = causal_conv3d(a, w, cache_bits=cache)
    np.testing.assert_array_equal(out[:, 0], cache[:, 1])
    np.testing.assert_array_equal(out[:, 1], a[:, 0])


def test_residual_and_bias_rounded_once():
    a = synth.normal_bf16((1, 1, 2, 2, 4), 0, "t/r/a")
    w = synth.normal_bf16((4, 3, 3, 3, 4), 0, "t/r/w")
    b = synth.normal_bf16((4,), 0, "t/r/b")
    r = synth.normal_bf16((1, 1, 2, 2, 4), 0, "t/r/r")
    y, _ = causal_conv3d(a, w, b, r)
    exact = causal_conv3d_f64(bf16_to_f64(a), bf16_to_f64(w), bf16_to_f64(b), bf16_to_f64(r))
    np.testing.assert_array_equal(y, round_to_bf16(exact))


def test_products_form_matches_torch_conv3d():
    # The frame-grouped form against torch's conv3d (fp64) on the front-padded input: batch 2,
    # 12 output channels, a cache, bias and residual; asymmetric random weights, so a transposed
    # tap index (kh <-> kw) or a reversed temporal tap would show.
    N, T, H, W, Ci, Co = 2, 5, 6, 7, 16, 12
    a = _rand((N, T, H, W, Ci), 11)
    cache = _rand((N, 2, H, W, Ci), 12)
    w = _rand((Co, 3, 3, 3, Ci), 13, 0.1)
    bias = _rand((Co,), 14)
    res = _rand((N, T, H, W, Co), 15)
    ours = causal_conv3d_products_f64(a, w, bias, res, cache)
    seq = np.concatenate([cache, a], axis=1)
    xt = torch.from_numpy(seq).permute(0, 4, 1, 2, 3)
    wt = torch.from_numpy(w).permute(0, 4, 1, 2, 3)
    ref = torch.nn.functional.conv3d(xt, wt, torch.from_numpy(bias), padding=(0, 1, 1))
    ref = ref.permute(0, 2, 3, 4, 1).numpy() + res
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)
    # without a cache the history is zero
    ref0 = torch.nn.functional.conv3d(torch.from_numpy(np.concatenate([np.zeros_like(cache), a], 1))
                                      .permute(0, 4, 1, 2, 3), wt, padding=(0, 1, 1)).permute(0, 2, 3, 4, 1).numpy()
    np.testing.assert_allclose(causal_conv3d_products_f64(a, w), ref0, rtol=1e-12, atol=1e-12)


def test_products_form_brute_force_points():
    N, T, H, W, Ci, Co = 1, 3, 4, 5, 3, 2
    a = _rand((N, T, H, W, Ci), 16)
    w = _rand((Co, 3, 3, 3, Ci), 17)
    ours = causal_conv3d_products_f64(a, w)
    for (t, h, x, co) in [(0, 0, 0, 0), (2, 3, 4, 1), (1, 2, 0, 1), (2, 0, 3, 0)]:
        s = 0.0
        for kt in range(3):
            for kh in range(3):
                for kw in range(3):
                    tt, hh, ww = t + kt - 2, h + kh - 1, x + kw - 1
                    if tt < 0 or not (0 <= hh < H) or not (0 <= ww < W):
                        continue
                    for ci in range(Ci):
                        s += w[co, kt, kh, kw, ci] * a[0, tt, hh, ww, ci]
        assert abs(ours[0, t, h, x, co] - s) < 1e-12


def test_conv_rows_depend_only_on_neighbouring_input_rows():
    # Output rows [r0, r1) read input rows [r0 - 1, r1 + 1) only (zero padding at the frame's
    # edge): the conv of that band of the input, minus its first and last row where they are halo,
    # is those rows of the full output. The full-size tests split a frame into such bands.
    N, T, H, W, Ci, Co = 1, 3, 11, 6, 8, 5
    a = _rand((N, T, H, W, Ci), 18)
    w = _rand((Co, 3, 3, 3, Ci), 19, 0.2)
    full = causal_conv3d_products_f64(a, w)
    for r0, r1 in ((0, 4), (4, 8), (8, 11), (3, 4)):
        lo, hi = max(r0 - 1, 0), min(r1 + 1, H)
        band = causal_conv3d_products_f64(a[:, :, lo:hi], w)
        np.testing.assert_allclose(band[:, :, r0 - lo:r0 - lo + (r1 - r0)], full[:, :, r0:r1], rtol=1e-13, atol=1e-13)
