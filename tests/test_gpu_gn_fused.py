"""GroupNorm + SiLU from the statistics that the CTA-pair conv emits with its output, on the GPU.
Emitting them leaves the conv's output unchanged bit for bit; the norm computed from them is
within one bf16 ulp of the oracle's GroupNorm + SiLU of that output; and it does not depend on
how the frames are chunked."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, f32_dev, bits
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))


def conv_inputs(shape, Cout, name, bias_mean=0.0, cache=False):
    N, T, H, W, Cin = shape
    a = synth.normal_bf16(shape, 0, f"{name}/a")
    w = synth.normal_bf16((Cout, 3, 3, 3, Cin), 0, f"{name}/w", 0.0, float(np.sqrt(1.0 / (27 * Cin))))
    b = synth.normal_bf16((Cout,), 0, f"{name}/b", bias_mean, 0.01)
    c = synth.normal_bf16((N, 2, H, W, Cin), 0, f"{name}/c") if cache else None
    return a, w, b, c


def norm_params(C, name):
    return synth.normal_f32((C,), 0, f"{name}/gamma", 1.0, 0.1), synth.normal_f32((C,), 0, f"{name}/beta", 0.0, 0.1)


def dev(t):
    return None if t is None else to_dev(t)


@pytest.mark.parametrize("shape,Cout,groups,bias_mean,cache", [
    ((1, 3, 19, 37, 64), 256, 32, 0.0, True),      # 8 channels per group, ragged tiles
    ((2, 2, 12, 33, 64), 512, 32, 0.0, False),     # 16 per group, batch 2, no history, two N blocks
    ((1, 2, 10, 20, 64), 1024, 32, 0.0, True),     # 32 per group: a group spans two 16-channel chunks
    ((1, 2, 9, 17, 64), 256, 64, 0.0, False),      # 4 per group
    ((1, 2, 11, 21, 64), 256, 32, 1000.0, True),   # mean 1000 against a spread of ~1: the shifts matter
])
def test_gn_from_conv_statistics(wan, shape, Cout, groups, bias_mean, cache):
    name = f"gnfused/{shape}/{Cout}/{groups}/{bias_mean}"
    a, w, b, c = conv_inputs(shape, Cout, name, bias_mean, cache)
    y_plain = wan.wan_causal_conv3d(dev(a), dev(w), dev(b), None, dev(c))
    y, st = wan.wan_causal_conv3d_gn_stats(dev(a), dev(w), groups, dev(b), None, dev(c))
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_plain.view(torch.int16))
    g, be = norm_params(Cout, name)
    out = wan.wan_gn_silu_from_stats(y, f32_dev(g), f32_dev(be), groups, EPS, st)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    ref = oracle.gn_silu(bits(y), g, be, groups, EPS)
    assert int(oracle.ulp_distance_bf16(bits(out), ref).max()) <= 1


def test_gn_from_conv_statistics_chunked_equals_unchunked(wan):
    shape, Cout, groups = (1, 8, 10, 30, 64), 256, 32
    a, w, b, _ = conv_inputs(shape, Cout, "gnfused/chunks")
    g, be = norm_params(Cout, "gnfused/chunks")
    ad, wd, bd, gd, bed = to_dev(a), to_dev(w), to_dev(b), f32_dev(g), f32_dev(be)
    y, st = wan.wan_causal_conv3d_gn_stats(ad, wd, groups, bd)
    full = wan.wan_gn_silu_from_stats(y, gd, bed, groups, EPS, st)
    cache = torch.empty((1, 2, 10, 30, 64), dtype=torch.bfloat16, device="cuda")
    parts = []
    for s0 in range(0, 8, 4):
        yc, stc = wan.wan_causal_conv3d_gn_stats(ad[:, s0:s0 + 4].contiguous(), wd, groups, bd, None,
                                                 None if s0 == 0 else cache, cache)
        parts.append(wan.wan_gn_silu_from_stats(yc, gd, bed, groups, EPS, stc))
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    assert torch.equal(torch.cat(parts, 1).view(torch.int16), full.view(torch.int16))
