"""Pins of the oracle's GroupNorm + SiLU (per-frame statistics, population variance)."""
import math

import numpy as np
import torch

from oracle import gn_silu, gn_silu_f64, silu_f64, bf16_to_f64
from video_vae_decoder_gb300 import synth


def test_brute_force_tiny():
    # Element-by-element loops (a different formulation from the vectorised oracle).
    rng = np.random.default_rng(3)
    N, T, H, W, C, G = 1, 2, 2, 3, 8, 4
    x = rng.normal(0.3, 1.7, size=(N, T, H, W, C))
    gamma = rng.normal(1, 0.1, size=C)
    beta = rng.normal(0, 0.1, size=C)
    eps = 1e-6
    got = gn_silu_f64(x, gamma, beta, G, eps)
    cg = C // G
    for n in range(N):
        for t in range(T):
            for g in range(G):
                vals = [x[n, t, h, w, c] for h in range(H) for w in range(W)
                        for c in range(g * cg, (g + 1) * cg)]
                m = math.fsum(vals) / len(vals)
                v = math.fsum((u - m) ** 2 for u in vals) / len(vals)
                for h in range(H):
                    for w in range(W):
                        for c in range(g * cg, (g + 1) * cg):
                            z = (x[n, t, h, w, c] - m) / math.sqrt(v + eps) * gamma[c] + beta[c]
                            s = z / (1 + math.exp(-z))
                            assert abs(got[n, t, h, w, c] - s) <= 1e-13 * max(1.0, abs(s))


def test_matches_torch_group_norm_per_frame():
    # PyTorch's group_norm on each frame as an image (N*T images, NCHW), fp64.
    N, T, H, W, C, G = 2, 3, 5, 7, 64, 32
    x = synth.normal_f32((N, T, H, W, C), 0, "t/gn/x", 0.5, np.sqrt(2.0)).astype(np.float64)
    gamma = synth.normal_f32((C,), 0, "t/gn/g", 1, 0.1)
    beta = synth.normal_f32((C,), 0, "t/gn/b", 0, 0.1)
    eps = float(np.float32(1e-6))
    ours = gn_silu_f64(x, gamma, beta, G, eps)
    xt = torch.from_numpy(x).permute(0, 1, 4, 2, 3).reshape(N * T, C, H, W)
    ref = torch.nn.functional.group_norm(xt, G, torch.from_numpy(gamma.astype(np.float64)),
                                         torch.from_numpy(beta.astype(np.float64)), eps)
    ref = torch.nn.functional.silu(ref).reshape(N, T, C, H, W).permute(0, 1, 3, 4, 2).numpy()
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-14)


def test_mean_shift_invariance():
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, size=(1, 2, 6, 6, 16))
    g = rng.normal(1, 0.1, size=16)
    b = rng.normal(0, 0.1, size=16)
    base = gn_silu_f64(x, g, b, 8, 1e-6)
    shifted = gn_silu_f64(x + 1e3, g, b, 8, 1e-6)
    np.testing.assert_allclose(shifted, base, rtol=1e-10, atol=1e-12)


def test_zero_variance_closed_form():
    # Every value of a group equal: x - m = 0 exactly, z = beta, output silu(beta).
    x = np.full((1, 1, 4, 4, 8), 1000.0)
    g = np.linspace(0.5, 1.5, 8)
    b = np.linspace(-0.3, 0.4, 8)
    out = gn_silu_f64(x, g, b, 4, 1e-6)
    np.testing.assert_array_equal(out, np.broadcast_to(silu_f64(b), out.shape))


def test_normalised_moments():
    # With beta = 0 the pre-activation divided by gamma has group mean 0 and variance
    # var/(var+eps). gamma = 0.1 keeps z inside (-1, 1), where silu is increasing and can be
    # inverted by bisection.
    rng = np.random.default_rng(7)
    x = rng.normal(2.0, 0.01, size=(1, 1, 8, 8, 4))
    eps = 1e-4
    cg, gain = 2, 0.1
    out = gn_silu_f64(x, np.full(4, gain), np.zeros(4), 2, eps)
    lo, hi = np.full(out.shape, -1.2), np.full(out.shape, 2.0)
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        up = silu_f64(mid) < out
        lo = np.where(up, mid, lo)
        hi = np.where(up, hi, mid)
    z = 0.5 * (lo + hi) / gain
    for g in range(2):
        zs = z[..., g * cg:(g + 1) * cg].ravel()
        xs = x[..., g * cg:(g + 1) * cg].ravel()
        var = xs.var()
        assert abs(zs.mean()) < 1e-9
        assert abs(zs.var() - var / (var + eps)) < 1e-9


def test_frames_are_independent():
    rng = np.random.default_rng(9)
    x = rng.normal(0, 1, size=(1, 3, 4, 4, 8))
    g, b = np.ones(8), np.zeros(8)
    base = gn_silu_f64(x, g, b, 4, 1e-6)
    x2 = x.copy()
    x2[:, 1] *= 7.0
    x2[:, 1] += 3.0
    out = gn_silu_f64(x2, g, b, 4, 1e-6)
    np.testing.assert_array_equal(out[:, 0], base[:, 0])
    np.testing.assert_array_equal(out[:, 2], base[:, 2])


def test_silu_large_negative_no_overflow():
    z = np.array([-800.0, -100.0, -1.0, 0.0, 1.0, 800.0])
    s = silu_f64(z)
    assert np.all(np.isfinite(s))
    assert s[0] == -0.0 or s[0] == 0.0
    assert abs(s[1] - (-100.0 * math.exp(-100.0) / (1 + math.exp(-100.0)))) < 1e-50
    assert s[5] == 800.0


def test_bf16_wrapper_rounds_once():
    rng = np.random.default_rng(11)
    xb = synth.f32_to_bf16_bits(rng.normal(0, 1, size=(1, 2, 4, 4, 8)).astype(np.float32))
    g = np.ones(8, np.float32)
    b = np.zeros(8, np.float32)
    out = gn_silu(xb, g, b, 4, 1e-6)
    f = gn_silu_f64(bf16_to_f64(xb), g, b, 4, 1e-6)
    # the rounded value is the nearest bf16: within half a bf16 step of the fp64 value
    back = bf16_to_f64(out)
    step = np.ldexp(1.0, np.frexp(f)[1] - 8)
    assert np.all(np.abs(back - f) <= 0.5 * step + 1e-300)


def test_whole_clip_brute_force_tiny():
    # Whole-clip statistics (per (n, group) over every frame) by element-by-element loops.
    rng = np.random.default_rng(5)
    N, T, H, W, C, G = 2, 3, 2, 2, 8, 2
    x = rng.normal(-0.4, 1.3, size=(N, T, H, W, C))
    gamma = rng.normal(1, 0.1, size=C)
    beta = rng.normal(0, 0.1, size=C)
    eps = 1e-6
    got = gn_silu_f64(x, gamma, beta, G, eps, whole_clip=True)
    cg = C // G
    for n in range(N):
        for g in range(G):
            vals = [x[n, t, h, w, c] for t in range(T) for h in range(H) for w in range(W)
                    for c in range(g * cg, (g + 1) * cg)]
            m = math.fsum(vals) / len(vals)
            v = math.fsum((u - m) ** 2 for u in vals) / len(vals)
            for t in range(T):
                for h in range(H):
                    for w in range(W):
                        for c in range(g * cg, (g + 1) * cg):
                            z = (x[n, t, h, w, c] - m) / math.sqrt(v + eps) * gamma[c] + beta[c]
                            s = z / (1 + math.exp(-z))
                            assert abs(got[n, t, h, w, c] - s) <= 1e-13 * max(1.0, abs(s))


def test_whole_clip_matches_torch_group_norm_5d():
    # PyTorch's group_norm on the N C T H W video (its statistics span the whole clip), fp64.
    N, T, H, W, C, G = 2, 3, 4, 5, 64, 32
    x = synth.normal_f32((N, T, H, W, C), 0, "t/gnc/x", 0.5, np.sqrt(2.0)).astype(np.float64)
    gamma = synth.normal_f32((C,), 0, "t/gnc/g", 1, 0.1)
    beta = synth.normal_f32((C,), 0, "t/gnc/b", 0, 0.1)
    ref = torch.nn.functional.group_norm(torch.from_numpy(x).permute(0, 4, 1, 2, 3), G,
                                         torch.from_numpy(gamma.astype(np.float64)),
                                         torch.from_numpy(beta.astype(np.float64)), 1e-6)
    ref = torch.nn.functional.silu(ref).permute(0, 2, 3, 4, 1).numpy()
    got = gn_silu_f64(x, gamma, beta, G, 1e-6, whole_clip=True)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_whole_clip_of_one_frame_is_per_frame():
    x = synth.normal_f32((2, 1, 3, 5, 32), 0, "t/gnc1/x").astype(np.float64)
    g = np.ones(32)
    b = np.zeros(32)
    assert np.array_equal(gn_silu_f64(x, g, b, 8, 1e-6, whole_clip=True), gn_silu_f64(x, g, b, 8, 1e-6))
