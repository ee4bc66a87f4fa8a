"""GroupNorm + SiLU on the GPU against the oracle: every element within one bf16 ulp."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, f32_dev, bits
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))


def run_case(wan, shape, groups, mean, std, name, seed=0):
    x = synth.normal_bf16(shape, seed, f"{name}/x", mean, std)
    C = shape[-1]
    g = synth.normal_f32((C,), seed, f"{name}/gamma", 1.0, 0.1)
    b = synth.normal_f32((C,), seed, f"{name}/beta", 0.0, 0.1)
    y = wan.wan_gn_silu(to_dev(x), f32_dev(g), f32_dev(b), groups, EPS)
    got = bits(y)
    ref = oracle.gn_silu(x, g, b, groups, EPS)
    ulp = oracle.ulp_distance_bf16(got, ref)
    assert wan.wan_device_status() == 0
    return int(ulp.max()), got, (x, g, b)


@pytest.mark.parametrize("shape,groups", [
    ((1, 3, 16, 16, 64), 32),      # 2 channels per group (4 groups per 16-byte vector)
    ((1, 3, 7, 13, 256), 32),      # 8 per group, ragged spans
    ((2, 2, 5, 9, 128), 16),       # batch of 2, 8 per group
    ((1, 2, 9, 11, 32), 32),       # 1 channel per group
    ((1, 2, 10, 10, 64), 16),      # 4 per group
    ((1, 1, 1, 1, 512), 32),       # a single pixel
    ((1, 2, 33, 47, 1024), 32),    # 32 per group
    ((1, 2, 9, 13, 2048), 32),     # the widest C supported: 64 per group
    ((1, 1, 5, 7, 2048), 256),     # the widest C in 256 groups of 8
])
def test_gn_small(wan, shape, groups):
    mx, _, _ = run_case(wan, shape, groups, 0.5, np.sqrt(2.0), f"gn/{shape}")
    assert mx <= 1


def test_gn_decode_mid_full_size(wan):
    # [1, C=512, T=4, H=88, W=156] stored channels-last, x ~ N(0.5, variance 2)
    mx, got, _ = run_case(wan, (1, 4, 88, 156, 512), 32, 0.5, np.sqrt(2.0), "gn/cfg2")
    assert mx <= 1


def test_gn_stress_degenerate_mean_1e3(wan):
    # mean 1e3, std 1e-2: every bf16 value rounds to 1000 (ulp 4 there), variance 0, so the
    # output is silu(beta) per channel exactly.
    mx, got, (x, g, b) = run_case(wan, (1, 4, 88, 156, 512), 32, 1e3, 1e-2, "gn/stress")
    assert np.all(x == x.flat[0])
    assert mx <= 1


def test_gn_stress_large_mean_small_spread(wan):
    # mean 1e4 with a spread of about one bf16 ulp: naive E[x^2] - E[x]^2 in fp32 fails here.
    mx, _, _ = run_case(wan, (1, 2, 44, 78, 512), 32, 1e4, 64.0, "gn/stress2")
    assert mx <= 1


def test_gn_deterministic(wan):
    x = to_dev(synth.normal_bf16((1, 4, 30, 40, 256), 1, "gn/det/x"))
    g = f32_dev(np.ones(256))
    b = f32_dev(np.zeros(256))
    y1 = bits(wan.wan_gn_silu(x, g, b, 32, EPS))
    y2 = bits(wan.wan_gn_silu(x, g, b, 32, EPS))
    assert np.array_equal(y1, y2)


def test_gn_very_negative_z(wan):
    # One outlier per group and large gammas put z in [-100, -80], where e^-|z| is subnormal in
    # fp32 but z*sigmoid(z) is still a representable (tiny) bf16: the exact-range path.
    N, T, H, W, C, G = 1, 2, 8, 8, 64, 32
    x = synth.normal_f32((N, T, H, W, C), 0, "gn/negz/x")
    x[:, :, 0, 0, :] = -30.0
    xb = synth.f32_to_bf16_bits(x)
    g = np.linspace(6.0, 11.0, C).astype(np.float32)
    b = np.zeros(C, np.float32)
    y = wan.wan_gn_silu(to_dev(xb), f32_dev(g), f32_dev(b), G, EPS)
    ref = oracle.gn_silu(xb, g, b, G, EPS)
    got = bits(y)
    assert int(oracle.ulp_distance_bf16(got, ref).max()) <= 1
    tiny = oracle.bf16_to_f64(ref[:, :, 0, 0, :])
    assert np.any((tiny < 0) & (tiny > -1e-30)), "the case must reach the tiny-output range"


@pytest.mark.parametrize("shape,groups,mean,std", [
    ((1, 3, 16, 16, 64), 32, 0.5, np.sqrt(2.0)),     # 2 channels per group
    ((2, 4, 9, 14, 128), 16, 0.5, np.sqrt(2.0)),     # batch of 2: one clip each
    ((1, 1, 7, 9, 256), 32, 0.5, np.sqrt(2.0)),      # one frame: the per-frame statistics
    ((1, 4, 88, 156, 512), 32, 0.5, np.sqrt(2.0)),   # the decode-mid size
    ((1, 2, 44, 78, 512), 32, 1e4, 64.0),            # large mean, spread of about one ulp
])
def test_gn_whole_clip(wan, shape, groups, mean, std):
    # Statistics per (n, group) over all frames (wan_gn_silu_clip), within one ulp of the oracle.
    name = f"gnclip/{shape}"
    x = synth.normal_bf16(shape, 0, f"{name}/x", mean, std)
    C = shape[-1]
    g = synth.normal_f32((C,), 0, f"{name}/gamma", 1.0, 0.1)
    b = synth.normal_f32((C,), 0, f"{name}/beta", 0.0, 0.1)
    got = bits(wan.wan_gn_silu(to_dev(x), f32_dev(g), f32_dev(b), groups, EPS, whole_clip=True))
    assert wan.wan_device_status() == 0
    ref = oracle.gn_silu(x, g, b, groups, EPS, whole_clip=True)
    assert int(oracle.ulp_distance_bf16(got, ref).max()) <= 1
    if shape[1] == 1:  # one frame: the same bits as the per-frame call
        assert np.array_equal(got, bits(wan.wan_gn_silu(to_dev(x), f32_dev(g), f32_dev(b), groups, EPS)))
