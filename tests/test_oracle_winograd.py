"""Pins of the oracle's Winograd F(2x2, 3x3) variant of the causal conv: the transform identity
against the direct convolution and torch, the weight transform's fp32 sums against scalar brute
force, and closed forms of the corner components."""
import numpy as np
import torch

import oracle
from video_vae_decoder_gb300 import synth


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).normal(0, scale, size=shape)


def test_winograd_identity_equals_direct_and_torch():
    # Exact transforms (fp64, no rounding) reproduce the causal conv: odd and even H, W, batch 2,
    # history, bias, residual; asymmetric weights so a transposed tap or component shows.
    for (N, T, H, W) in ((2, 3, 5, 7), (1, 4, 6, 4), (1, 1, 1, 3)):
        Ci, Co = 8, 6
        a = _rand((N, T, H, W, Ci), 1)
        c = _rand((N, 2, H, W, Ci), 2)
        w = _rand((Co, 3, 3, 3, Ci), 3, 0.1)
        b = _rand((Co,), 4)
        r = _rand((N, T, H, W, Co), 5)
        y = oracle.winograd_causal_conv3d_f64(a, oracle.winograd_weights_f64(w), b, r, c)
        np.testing.assert_allclose(y, oracle.causal_conv3d_f64(a, w, b, r, c), rtol=1e-12, atol=1e-12)
        seq = torch.from_numpy(np.concatenate([c, a], 1)).permute(0, 4, 1, 2, 3)
        ref = torch.nn.functional.conv3d(seq, torch.from_numpy(w).permute(0, 4, 1, 2, 3), torch.from_numpy(b),
                                         padding=(0, 1, 1)).permute(0, 2, 3, 4, 1).numpy() + r
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
        # without history the two leading frames are zeros
        np.testing.assert_allclose(oracle.winograd_causal_conv3d_f64(a, oracle.winograd_weights_f64(w)),
                                   oracle.causal_conv3d_f64(a, w), rtol=1e-12, atol=1e-12)


def test_winograd_weights_fp32_sums_brute_force():
    w = synth.normal_bf16((3, 3, 3, 3, 5), 0, "wino/pin/w", 0.0, 0.3)
    got = oracle.winograd_weights(w)
    assert got.shape == (16, 3, 3, 5) and got.dtype == np.uint16
    wf = oracle.bf16_to_f32(w)
    G = [[1.0, 0.0, 0.0], [0.5, 0.5, 0.5], [0.5, -0.5, 0.5], [0.0, 0.0, 1.0]]
    for xy in range(16):
        x, y = divmod(xy, 4)
        for co in range(3):
            for kt in range(3):
                for ci in range(5):
                    s = np.float32(0.0)
                    for r in range(3):
                        for c in range(3):
                            k = G[x][r] * G[y][c]
                            if k != 0:
                                s = np.float32(s + np.float32(k) * wf[co, kt, r, c, ci])
                    assert np.float16(s).view(np.uint16) == got[xy, co, kt, ci]


def test_winograd_weights_corner_components_and_rounding():
    w = synth.normal_bf16((4, 3, 3, 3, 8), 0, "wino/pin/w2", 0.0, 0.2)
    u = oracle.winograd_weights(w)
    wf = oracle.bf16_to_f64(w)
    # G's first row is (1, 0, 0) and its last (0, 0, 1): components (0, 0), (0, 3), (3, 0), (3, 3)
    # are single taps of the kernel, rounded to fp16 once.
    for xy, (r, c) in ((0, (0, 0)), (3, (0, 2)), (12, (2, 0)), (15, (2, 2))):
        assert np.array_equal(u[xy], oracle.f32_to_f16_bits(wf[:, :, r, c, :].astype(np.float32)))
    # every component within half an fp16 step (plus fp32 sum error) of the exact transform
    exact = oracle.winograd_weights_f64(wf)
    got = oracle.f16_to_f64(u)
    assert np.all(np.abs(got - exact) <= np.abs(exact) * (2.0 ** -11 + 2.0 ** -22) + 2.0 ** -25)


def test_fp16_winograd_operands_keep_the_conv_criterion():
    # The variant with both transformed operands stored in fp16 stays within the conv criterion
    # (relative L2 4e-3, max 2^-7 max|ref|) of the exact conv on a decoder-like case.
    N, T, H, W, Ci, Co = 1, 2, 9, 10, 64, 32
    a = oracle.bf16_to_f64(synth.normal_bf16((N, T, H, W, Ci), 0, "wino/pin/a"))
    w = synth.normal_bf16((Co, 3, 3, 3, Ci), 0, "wino/pin/w3", 0.0, float(np.sqrt(1.0 / (27 * Ci))))
    to16 = lambda v: np.asarray(v, np.float16).astype(np.float64)  # noqa: E731
    y = oracle.winograd_causal_conv3d_f64(a, oracle.f16_to_f64(oracle.winograd_weights(w)), store=to16)
    ref = oracle.causal_conv3d_f64(a, oracle.bf16_to_f64(w))
    yb = oracle.bf16_to_f64(oracle.round_to_bf16(y))
    rel = np.linalg.norm(yb - ref) / np.linalg.norm(ref)
    assert rel <= 4e-3 and np.abs(yb - ref).max() <= 2.0 ** -7 * np.abs(ref).max()
