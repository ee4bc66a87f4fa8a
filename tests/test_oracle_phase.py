"""Pins of the oracle's phase-weight transform and phase convolution."""
import os

import numpy as np

from oracle import (phase_tap_sources, phase_weights, phase_weights_f64, phase_conv_f64,
                    upsample_nearest_conv_f64, bf16_to_f32, round_to_bf16)
from video_vae_decoder_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "phase_taps.txt")


def test_tap_sources_match_golden_table():
    table = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if line:
            a, u, *rows = map(int, line)
            table[(a, u)] = rows
    assert len(table) == 4
    for (a, u), rows in table.items():
        assert phase_tap_sources(a, u) == rows


def test_every_tap_used_once_per_phase():
    w3 = np.random.default_rng(1).normal(size=(3, 3, 3, 2))
    wp = phase_weights_f64(w3)
    for p in range(4):
        np.testing.assert_allclose(wp[p].sum(axis=(1, 2)), w3.sum(axis=(1, 2)), rtol=1e-13)


def test_phase_form_equals_definition_fp64():
    # Nearest-x2 then 3x3 (pad 1) equals the four 2x2 phase convolutions, exactly up to rounding.
    rng = np.random.default_rng(2)
    x = rng.normal(size=(1, 2, 5, 7, 6))
    w3 = rng.normal(size=(4, 3, 3, 6))
    b = rng.normal(size=4)
    ref = upsample_nearest_conv_f64(x, w3, b)
    got = phase_conv_f64(x, phase_weights_f64(w3), b)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_definition_brute_force_point():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(1, 1, 3, 4, 2))
    w3 = rng.normal(size=(2, 3, 3, 2))
    y = upsample_nearest_conv_f64(x, w3)
    H, W = 3, 4
    for (Y, X, co) in [(0, 0, 0), (5, 7, 1), (2, 3, 0), (4, 0, 1)]:
        s = 0.0
        for r in range(3):
            for c in range(3):
                yy, xx = Y + r - 1, X + c - 1
                if 0 <= yy < 2 * H and 0 <= xx < 2 * W:
                    s += float(np.dot(w3[co, r, c], x[0, 0, yy // 2, xx // 2]))
        assert abs(y[0, 0, Y, X, co] - s) < 1e-12


def test_bf16_phase_weights_brute_force():
    w3 = synth.normal_bf16((3, 3, 3, 4), 0, "t/ph/w3", 0, 0.05)
    wf = bf16_to_f32(w3)
    got = phase_weights(w3)
    for a in range(2):
        for b in range(2):
            for u in range(2):
                for v in range(2):
                    for co in range(3):
                        for ci in range(4):
                            s = np.float32(0.0)
                            for r in phase_tap_sources(a, u):
                                for c in phase_tap_sources(b, v):
                                    s = np.float32(s + wf[co, r, c, ci])
                            want = round_to_bf16(np.array([float(s)]))[0]
                            assert got[2 * a + b, co, u, v, ci] == want


def test_definition_matches_torch_nearest_and_conv2d():
    # The definition against PyTorch: nearest-x2 interpolation, then conv2d with padding 1 (fp64).
    import torch
    x = synth.normal_f32((1, 2, 5, 7, 16), 0, "t/up/torch/x").astype(np.float64)
    w3 = synth.normal_f32((24, 3, 3, 16), 0, "t/up/torch/w", 0.0, 0.2).astype(np.float64)
    b = synth.normal_f32((24,), 0, "t/up/torch/b", 0.0, 0.1).astype(np.float64)
    got = upsample_nearest_conv_f64(x, w3, b)
    xt = torch.from_numpy(x).reshape(2, 5, 7, 16).permute(0, 3, 1, 2)      # frames as images, NCHW
    up = torch.nn.functional.interpolate(xt, scale_factor=2, mode="nearest")
    ref = torch.nn.functional.conv2d(up, torch.from_numpy(w3).permute(0, 3, 1, 2), torch.from_numpy(b), padding=1)
    ref = ref.permute(0, 2, 3, 1).reshape(1, 2, 10, 14, 24).numpy()
    assert np.max(np.abs(got - ref)) < 1e-12
