"""GroupNorm + SiLU into a causal conv (wan_gn_silu_causal_conv3d) on the GPU.

For Cout >= 256 the conv normalises its operand tiles in shared memory and the activation is never
stored; for smaller Cout it is materialised. Either way y and the new cache must be bit for bit
what the unfused calls return (wan_gn_silu, then wan_causal_conv3d with its cache update), the
pair must match the oracle, and chunking the frames must not change a bit."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, f32_dev, bits, conv_close
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))
G = 32


def inputs(shape, Cout, name):
    N, T, H, W, Cin = shape
    x = synth.normal_bf16(shape, 0, f"{name}/x", 0.3, 1.5)
    g = synth.normal_f32((Cin,), 0, f"{name}/gamma", 1.0, 0.1)
    be = synth.normal_f32((Cin,), 0, f"{name}/beta", 0.0, 0.1)
    w = synth.normal_bf16((Cout, 3, 3, 3, Cin), 0, f"{name}/w", 0.0, float(np.sqrt(1.0 / (27 * Cin))))
    b = synth.normal_bf16((Cout,), 0, f"{name}/b", 0.0, 0.01)
    c = synth.normal_bf16((N, 2, H, W, Cin), 0, f"{name}/c", 0.0, 0.5)
    r = synth.normal_bf16((N, T, H, W, Cout), 0, f"{name}/r")
    return x, g, be, w, b, c, r


def unfused(wan, x, g, be, w, b, r, c_in):
    a = wan.wan_gn_silu(x, g, be, G, EPS)
    c_out = torch.empty((x.shape[0], 2) + tuple(x.shape[2:]), dtype=torch.bfloat16, device="cuda")
    y = wan.wan_causal_conv3d(a, w, b, r, c_in, c_out)
    return y, c_out


def same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("shape,Cout,history,residual", [
    ((1, 4, 19, 37, 64), 256, True, False),    # prologue path, ragged tiles, 2 channels per group
    ((2, 3, 12, 33, 128), 256, False, True),   # batch 2, no history, residual
    ((1, 1, 10, 20, 256), 512, True, False),   # one frame: the history shifts by one; two N blocks
    ((1, 2, 9, 17, 256), 256, True, True),     # two frames: the new history is all of a
    ((1, 3, 16, 16, 64), 64, True, False),     # Cout < 256: the activation is materialised
])
def test_fused_equals_unfused(wan, shape, Cout, history, residual):
    x, g, be, w, b, c, r = inputs(shape, Cout, f"gnconv/{shape}/{Cout}")
    xd, gd, bed, wd, bd = to_dev(x), f32_dev(g), f32_dev(be), to_dev(w), to_dev(b)
    cd = to_dev(c) if history else None
    rd = to_dev(r) if residual else None
    y_ref, c_ref = unfused(wan, xd, gd, bed, wd, bd, rd, cd)
    c_out = torch.empty_like(c_ref)
    y = wan.wan_gn_silu_causal_conv3d(xd, gd, bed, G, EPS, wd, bd, rd, cd, c_out)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    assert same(y, y_ref)
    assert same(c_out, c_ref)
    if history:  # the cache updated in place gives the same bits
        c_io = cd.clone()
        y2 = wan.wan_gn_silu_causal_conv3d(xd, gd, bed, G, EPS, wd, bd, rd, c_io, c_io)
        torch.cuda.synchronize()
        assert same(y2, y_ref)
        assert same(c_io, c_ref)


@pytest.mark.parametrize("shape,Cout", [
    ((1, 3, 11, 21, 64), 256),
    ((1, 2, 9, 17, 256), 256),     # 8 channels per group
    ((1, 2, 9, 17, 1024), 1024),   # the widest stage's Cin: 16 K blocks per tap, 32 channels per group
    ((1, 3, 8, 20, 1024), 256),
    ((1, 2, 1, 1, 64), 256),       # 1 x 1 frames: each group of a frame holds 2 values
    ((1, 2, 1, 9, 256), 256),      # one-pixel-high frames: the tiles' boxes mostly zero padding
    ((1, 2, 9, 1, 256), 256),      # one-pixel-wide frames
    ((1, 2, 5, 9, 2048), 256),     # the widest Cin the norm takes: 32 K blocks per tap
])
def test_fused_matches_oracle(wan, shape, Cout):
    x, g, be, w, b, c, _ = inputs(shape, Cout, f"gnconv/oracle/{shape}/{Cout}")
    N, T, H, W, Cin = shape
    c_out = torch.empty((N, 2, H, W, Cin), dtype=torch.bfloat16, device="cuda")
    y = wan.wan_gn_silu_causal_conv3d(to_dev(x), f32_dev(g), f32_dev(be), G, EPS, to_dev(w), to_dev(b), None,
                                      to_dev(c), c_out)
    torch.cuda.synchronize()
    a_ref = oracle.gn_silu(x, g, be, G, EPS)
    y_ref, c_ref = oracle.causal_conv3d(a_ref, w, b, None, c)
    conv_close(bits(y), y_ref, "norm into conv")
    assert int(oracle.ulp_distance_bf16(bits(c_out), c_ref).max()) <= 1


def test_fused_chunked_equals_unchunked(wan):
    shape, Cout = (1, 8, 14, 40, 128), 256
    x, g, be, w, b, _, _ = inputs(shape, Cout, "gnconv/chunks")
    xd, gd, bed, wd, bd = to_dev(x), f32_dev(g), f32_dev(be), to_dev(w), to_dev(b)
    c_full = torch.empty((1, 2, 14, 40, 128), dtype=torch.bfloat16, device="cuda")
    full = wan.wan_gn_silu_causal_conv3d(xd, gd, bed, G, EPS, wd, bd, None, None, c_full)
    cache = torch.empty_like(c_full)
    parts = []
    for i, s0 in enumerate(range(0, 8, 3)):  # chunks of 3, 3 and 2 frames
        parts.append(wan.wan_gn_silu_causal_conv3d(xd[:, s0:s0 + 3].contiguous(), gd, bed, G, EPS, wd, bd, None,
                                                   cache if i else None, cache))
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    assert same(torch.cat(parts, 1), full)
    assert same(cache, c_full)


def test_fused_equals_unfused_decode_size(wan):
    # The C=256 decoder stage's chunk [1, 4, 176, 312, 256] with history, as the ResBlock runs it.
    shape = (1, 4, 176, 312, 256)
    xd = synth.normal_torch(shape, 0, "gnconv/big/x", 0.3, 1.5, device="cuda", dtype=torch.bfloat16)
    gd = synth.normal_torch((256,), 0, "gnconv/big/g", 1.0, 0.1, device="cuda", dtype=torch.float32)
    bed = synth.normal_torch((256,), 0, "gnconv/big/be", 0.0, 0.1, device="cuda", dtype=torch.float32)
    wd = synth.normal_torch((256, 3, 3, 3, 256), 0, "gnconv/big/w", 0.0, float(np.sqrt(1.0 / (27 * 256))),
                            device="cuda", dtype=torch.bfloat16)
    bd = synth.normal_torch((256,), 0, "gnconv/big/b", 0.0, 0.01, device="cuda", dtype=torch.bfloat16)
    cd = synth.normal_torch((1, 2, 176, 312, 256), 0, "gnconv/big/c", 0.0, 0.5, device="cuda", dtype=torch.bfloat16)
    y_ref, c_ref = unfused(wan, xd, gd, bed, wd, bd, xd, cd)
    c_out = torch.empty_like(c_ref)
    y = wan.wan_gn_silu_causal_conv3d(xd, gd, bed, G, EPS, wd, bd, xd, cd, c_out)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    assert same(y, y_ref)
    assert same(c_out, c_ref)


@pytest.mark.parametrize("shape,history,in_place", [
    ((1, 4, 12, 20, 128), True, False),
    ((2, 1, 9, 17, 64), True, True),     # one frame: the history shifts by a strided copy, in place
    ((1, 1, 9, 17, 64), False, False),   # one frame, no history: zeros move in
])
def test_steps_equal_fused(wan, shape, history, in_place):
    Cout = 256
    x, g, be, w, b, c, r = inputs(shape, Cout, f"gnconv/steps/{shape}")
    xd, gd, bed, wd, bd, rd = to_dev(x), f32_dev(g), f32_dev(be), to_dev(w), to_dev(b), to_dev(r)
    cd = to_dev(c) if history else None
    c_f = torch.empty((shape[0], 2) + shape[2:], dtype=torch.bfloat16, device="cuda")
    y_f = wan.wan_gn_silu_causal_conv3d(xd, gd, bed, G, EPS, wd, bd, rd, cd, c_f)
    coef = wan.wan_gn_silu_coefficients(xd, gd, bed, G, EPS)
    # the conv writing the new history itself (a cache_out apart from the history it reads)
    c_d = torch.empty_like(c_f)
    y_d = wan.wan_causal_conv3d_gn_input(xd, coef, wd, bd, rd, cd, cache_out=c_d)
    y = wan.wan_causal_conv3d_gn_input(xd, coef, wd, bd, rd, cd)
    if in_place:
        c_s = cd.clone()
        wan.wan_gn_silu_cache_update(xd, coef, c_s, c_s)
    else:
        c_s = torch.empty_like(c_f)
        wan.wan_gn_silu_cache_update(xd, coef, c_s, cd)
    torch.cuda.synchronize()
    assert same(y_d, y_f) and same(c_d, c_f)
    assert wan.wan_device_status() == 0
    assert same(y, y_f)
    assert same(c_s, c_f)


@pytest.mark.parametrize("shape", [(1, 4, 176, 312, 256), (1, 2, 44, 78, 1024)])
def test_history_written_by_the_conv_equals_the_pass_after_it(wan, shape):
    # At the decoder's sizes: the conv storing the normalised last two frames from its operand
    # prologue (cache_out apart from cache_in) writes the bits that the pass after the conv writes
    # (cache_out == cache_in), and the same y.
    N, T, H, W, C = shape
    x = synth.normal_torch(shape, 0, f"gnconv/hist/{C}/x", device="cuda", dtype=torch.bfloat16)
    g = f32_dev(synth.normal_f32((C,), 0, f"gnconv/hist/{C}/g", 1.0, 0.1))
    be = f32_dev(synth.normal_f32((C,), 0, f"gnconv/hist/{C}/b", 0.0, 0.1))
    w = synth.normal_torch((C, 3, 3, 3, C), 0, f"gnconv/hist/{C}/w", 0.0, float(np.sqrt(1.0 / (27 * C))),
                           device="cuda", dtype=torch.bfloat16)
    hist = synth.normal_torch((N, 2, H, W, C), 0, f"gnconv/hist/{C}/c", 0.1, 0.6, device="cuda", dtype=torch.bfloat16)
    coef = wan.wan_gn_silu_coefficients(x, g, be, G, EPS)
    c_direct = torch.empty_like(hist)
    y_direct = wan.wan_causal_conv3d_gn_input(x, coef, w, None, None, hist, cache_out=c_direct)
    c_place = hist.clone()
    y_place = wan.wan_causal_conv3d_gn_input(x, coef, w, None, None, c_place, cache_out=c_place)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    assert same(y_direct, y_place)
    assert same(c_direct, c_place)
