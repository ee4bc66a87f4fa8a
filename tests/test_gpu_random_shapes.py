"""Seeded random small shapes through the CTA-pair conv (plain and with the GroupNorm prologue), the
output head, the phase-conv upsample and the time upsample, against the oracle.

The shapes are drawn so that tile counts, ragged edges, batch items, history and the scheduling of
the last round (whole items or 128-channel halves) vary from case to case."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, f32_dev, bits, conv_close
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))


def _cases():
    rng = np.random.default_rng(2024)
    out = []
    for i in range(10):
        Cin = int(rng.choice([64, 128, 256]))
        Cout = int(rng.choice([256, 320, 512, 768]))
        N, T = int(rng.integers(1, 3)), int(rng.integers(1, 6))
        H, W = int(rng.integers(1, 20)), int(rng.integers(1, 40))
        while N * T * H * W * Cin * Cout * 27 > 4e9:
            W, H = max(1, W // 2), max(1, H - 3)
        out.append(("conv", (N, T, H, W, Cin), Cout, tuple(bool(v) for v in rng.integers(0, 2, 3)), bool(i % 2)))
    for i in range(5):
        Cin = int(rng.choice([64, 128, 192, 256]))
        shape = (int(rng.integers(1, 3)), int(rng.integers(1, 10)), int(rng.integers(1, 14)), int(rng.integers(1, 280)), Cin)
        out.append(("head", shape, 12, tuple(bool(v) for v in rng.integers(0, 2, 3)), False))
    for i in range(3):
        shape = (1, int(rng.integers(1, 3)), int(rng.integers(1, 12)), int(rng.integers(1, 24)), int(rng.choice([64, 128])))
        out.append(("up", shape, int(rng.choice([256, 512])), (bool(rng.integers(2)), False, False), False))
    for i in range(3):
        shape = (1, int(rng.integers(1, 5)), int(rng.integers(1, 10)), int(rng.integers(1, 20)), int(rng.choice([256, 512])))
        out.append(("tup", shape, 2 * shape[-1], (bool(rng.integers(2)), bool(rng.integers(2)), False), False))
    return out


def f64(x):
    return None if x is None else oracle.bf16_to_f64(x)


@pytest.mark.parametrize("kind,shape,Cout,flags,norm", _cases())
def test_random_shape(wan, kind, shape, Cout, flags, norm):
    name = f"rand/{kind}/{shape}/{Cout}/{flags}/{norm}"
    N, T, H, W, Cin = shape
    if kind in ("conv", "head"):
        bias, residual, cache = flags
        a = synth.normal_bf16(shape, 0, f"{name}/a")
        w = synth.normal_bf16((Cout, 3, 3, 3, Cin), 0, f"{name}/w", 0.0, float(np.sqrt(1.0 / (27 * Cin))))
        b = synth.normal_bf16((Cout,), 0, f"{name}/b", 0.0, 0.01) if bias else None
        r = synth.normal_bf16((N, T, H, W, Cout), 0, f"{name}/r") if residual else None
        c = synth.normal_bf16((N, 2, H, W, Cin), 0, f"{name}/c") if cache else None
        d = [None if v is None else to_dev(v) for v in (b, r, c)]
        if norm:
            gam = synth.normal_f32((Cin,), 0, f"{name}/g", 1.0, 0.1)
            bet = synth.normal_f32((Cin,), 0, f"{name}/be", 0.0, 0.1)
            y = wan.wan_gn_silu_causal_conv3d(to_dev(a), f32_dev(gam), f32_dev(bet), 32, EPS, to_dev(w), *d)
            act = oracle.gn_silu(a, gam, bet, 32, EPS)
            ref = oracle.causal_conv3d_f64(f64(act), f64(w), f64(b), f64(r), f64(c))
        else:
            y = wan.wan_causal_conv3d(to_dev(a), to_dev(w), *d)
            ref = oracle.causal_conv3d_f64(f64(a), f64(w), f64(b), f64(r), f64(c))
    elif kind == "up":
        bias = flags[0]
        x = synth.normal_bf16(shape, 0, f"{name}/x")
        w3 = synth.normal_bf16((Cout, 3, 3, Cin), 0, f"{name}/w", 0.0, float(np.sqrt(1.0 / (9 * Cin))))
        b = synth.normal_bf16((Cout,), 0, f"{name}/b", 0.0, 0.01) if bias else None
        y = wan.wan_upsample_phase_conv(to_dev(x), wan.wan_upsample_phase_weights(to_dev(w3)),
                                        None if b is None else to_dev(b))
        ref = oracle.upsample_nearest_conv_f64(f64(x), f64(w3), f64(b))
    else:
        first, history = flags[0], flags[1]
        x = synth.normal_bf16(shape, 0, f"{name}/x")
        w = synth.normal_bf16((Cout, 3, Cin), 0, f"{name}/w", 0.0, float(np.sqrt(1.0 / (3 * Cin))))
        b = synth.normal_bf16((Cout,), 0, f"{name}/b", 0.0, 0.01)
        c = synth.normal_bf16((N, 2, H, W, Cin), 0, f"{name}/c") if history else None
        y = wan.wan_time_upsample(to_dev(x), to_dev(w), to_dev(b), first, None if c is None else to_dev(c))
        ref = oracle.time_upsample_f64(f64(x), f64(w), f64(b), f64(c), first)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    got = bits(y)
    assert got.shape == ref.shape
    conv_close(got, ref, name)
