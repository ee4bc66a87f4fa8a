"""The Winograd F(2x2, 3x3) causal conv on the GPU (fp16 transformed operands, tcgen05 kind::f16):

  * the weight transform bit for bit against the oracle's fp32 sums (binding.cpp, `prepare()`);
  * the conv against the definition (the direct fp64 conv) under the conv criterion, and against
    the oracle's Winograd algorithm with the same fp16 operands (the kernel's own arithmetic,
    within one bf16 step);
  * with the GroupNorm + SiLU coefficients applied to its input, with history, bias, residual,
    batch 2, odd frame sizes and a single frame;
  * chunked == unchunked bit for bit, and the ResBlock built on it against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from util import REL_L2_MAX, to_dev, f32_dev, bits, conv_close, cache2_close
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))
G = 32


def u_dev(u_bits):
    return torch.from_numpy(np.ascontiguousarray(u_bits).view(np.int16).copy()).view(torch.float16).cuda()


def fp16_store(v):
    return np.asarray(v, np.float16).astype(np.float64)


@pytest.mark.parametrize("Cout,Cin", [(256, 64), (512, 128), (256, 1024)])
def test_winograd_weights_bit_exact(wan, Cout, Cin):
    w = synth.normal_bf16((Cout, 3, 3, 3, Cin), 0, f"wino/w/{Cout}/{Cin}", 0.0, float(np.sqrt(1.0 / (27 * Cin))))
    u = wan.wan_winograd_weights(to_dev(w))
    torch.cuda.synchronize()
    got = u.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.winograd_weights(w))


def make(shape, Cout, name, coef, cache, bias, residual):
    N, T, H, W, Cin = shape
    x = synth.normal_bf16(shape, 0, f"{name}/x", 0.2, 1.2)
    w = synth.normal_bf16((Cout, 3, 3, 3, Cin), 0, f"{name}/w", 0.0, float(np.sqrt(1.0 / (27 * Cin))))
    g = synth.normal_f32((Cin,), 0, f"{name}/g", 1.0, 0.1) if coef else None
    be = synth.normal_f32((Cin,), 0, f"{name}/be", 0.0, 0.1) if coef else None
    c = synth.normal_bf16((N, 2, H, W, Cin), 0, f"{name}/c", 0.1, 0.6) if cache else None
    b = synth.normal_bf16((Cout,), 0, f"{name}/b", 0.0, 0.01) if bias else None
    r = synth.normal_bf16((N, T, H, W, Cout), 0, f"{name}/r") if residual else None
    return x, w, g, be, c, b, r


def run_wino(wan, x, w, g, be, c, b, r, cache_out=True):
    N, T, H, W, Cin = x.shape
    xd = to_dev(x)
    coef = wan.wan_gn_silu_coefficients(xd, f32_dev(g), f32_dev(be), G, EPS) if g is not None else None
    cout = torch.empty((N, 2, H, W, Cin), dtype=torch.bfloat16, device="cuda") if cache_out else None
    u = wan.wan_winograd_weights(to_dev(w))
    y = wan.wan_causal_conv3d_winograd(xd, u, coef, None if b is None else to_dev(b), None if r is None else to_dev(r),
                                       None if c is None else to_dev(c), cout)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    return bits(y), (bits(cout) if cache_out else None)


@pytest.mark.parametrize("shape,Cout,coef,cache,bias,residual", [
    ((1, 3, 9, 11, 64), 256, False, False, True, False),     # odd H and W: half-empty edge tiles
    ((1, 4, 8, 16, 128), 256, True, True, False, True),      # the norm applied to the input, history, residual
    ((2, 2, 5, 7, 64), 512, False, True, True, True),        # batch 2 (a pair tile crosses batch items), 2 N blocks
    ((1, 1, 6, 6, 64), 256, True, True, True, False),        # one frame: both history frames from the cache
    ((1, 5, 20, 40, 256), 256, True, False, True, False),    # 1000 rows: 4 pair tiles, the last partial
    ((1, 2, 7, 9, 1024), 256, True, True, True, True),       # 16 K blocks per tap
    ((1, 2, 11, 91, 64), 256, True, True, False, False),     # 46 tiles wide: two column blocks of the transform
    ((1, 2, 1, 1, 64), 256, True, True, True, True),         # a 1 x 1 frame: one tile, 3 of its outputs outside
    ((1, 3, 1, 3, 64), 256, True, False, True, False),       # one-pixel-high frames
    ((1, 2, 3, 1, 128), 256, False, True, False, True),      # one-pixel-wide frames
    ((1, 2, 5, 7, 2048), 256, True, True, True, True),       # the widest Cin with the norm applied
])
def test_winograd_conv_matches_oracle(wan, shape, Cout, coef, cache, bias, residual):
    name = f"wino/conv/{shape}/{Cout}"
    x, w, g, be, c, b, r = make(shape, Cout, name, coef, cache, bias, residual)
    got, cout = run_wino(wan, x, w, g, be, c, b, r)
    f = oracle.bf16_to_f64
    a = oracle.gn_silu(x, g, be, G, EPS) if coef else x
    bb, rr, cc = (None if v is None else f(v) for v in (b, r, c))
    # the definition: the direct conv in fp64
    conv_close(got, oracle.causal_conv3d_f64(f(a), f(w), bb, rr, cc), "winograd vs the direct conv")
    # the same algorithm with the same fp16 operands: within one bf16 step at the largest magnitude
    ref = oracle.winograd_causal_conv3d_f64(f(a), oracle.f16_to_f64(oracle.winograd_weights(w)), bb, rr, cc,
                                            store=fp16_store)
    ref_b = oracle.bf16_to_f64(oracle.round_to_bf16(ref))
    diff = oracle.bf16_to_f64(got) - ref_b
    assert np.linalg.norm(diff) <= 0.25 * REL_L2_MAX * np.linalg.norm(ref_b)
    assert np.abs(diff).max() <= 2.0 ** -8 * np.abs(ref_b).max()
    # the new history: the last two frames of [cache; activated input], as the other paths write them
    prev = np.zeros_like(x[:, :2]) if c is None else c
    want = np.concatenate([prev, a], 1)[:, -2:]
    assert int(oracle.ulp_distance_bf16(cout, want).max()) <= (1 if coef else 0)


def test_winograd_chunked_equals_unchunked(wan):
    shape = (1, 8, 12, 20, 256)
    x, w, g, be, _, b, _ = make(shape, 256, "wino/chunks", True, False, True, False)
    xd, gd, bed, bd = to_dev(x), f32_dev(g), f32_dev(be), to_dev(b)
    u = wan.wan_winograd_weights(to_dev(w))

    def call(xs, cin, cout):
        coef = wan.wan_gn_silu_coefficients(xs, gd, bed, G, EPS)
        return wan.wan_causal_conv3d_winograd(xs, u, coef, bd, None, cin, cout)
    full_cache = torch.empty((1, 2, 12, 20, 256), dtype=torch.bfloat16, device="cuda")
    full = call(xd, None, full_cache)
    cache = torch.empty_like(full_cache)
    parts = []
    for s in range(0, 8, 4):
        parts.append(call(xd[:, s:s + 4].contiguous(), None if s == 0 else cache, cache))
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts, 1).view(torch.int16), full.view(torch.int16))
    assert torch.equal(cache.view(torch.int16), full_cache.view(torch.int16))
    assert wan.wan_device_status() == 0


def test_resblock_winograd_matches_oracle(wan):
    # Two chunks (2 + 2 frames) of a C=256 ResBlock with both convs through Winograd.
    x = synth.normal_bf16((1, 4, 12, 20, 256), 0, "wino/rb/x")
    p = synth.resblock_params(256, 0, "wino/rb")
    pd = {k: (f32_dev(v) if v.dtype == np.float32 else to_dev(v)) for k, v in p.items()}
    u1, u2 = wan.wan_winograd_weights(pd["w1"]), wan.wan_winograd_weights(pd["w2"])
    c1 = torch.zeros((1, 2, 12, 20, 256), dtype=torch.bfloat16, device="cuda")
    c2 = torch.zeros_like(c1)
    outs = [wan.wan_resblock_winograd(to_dev(np.ascontiguousarray(x[:, s:s + 2])), pd, u1, u2, c1, c2, s > 0, G, EPS)
            for s in (0, 2)]
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    r_a, r1, r2 = oracle.resblock(x[:, :2], p, G, EPS)
    r_b, r1, r2 = oracle.resblock(x[:, 2:], p, G, EPS, r1, r2)
    conv_close(np.concatenate([bits(o) for o in outs], 1), np.concatenate([r_a, r_b], 1), "winograd resblock")
    assert int(oracle.ulp_distance_bf16(bits(c1), r1).max()) <= 1
    cache2_close(bits(c2), r2, "winograd resblock cache 2")
