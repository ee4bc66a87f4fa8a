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


@pytest.mark.parametrize("groups", [
    32,    # 8 channels per group: the second norm from conv 1's statistics
    64,    # 4 per group: the statistics with one lane per group
    128,   # 2 per group: no statistics at this width, the second norm from a pass over h
])
def test_resblock_winograd_matches_oracle(wan, groups):
    # Two chunks (2 + 2 frames) of a C=256 ResBlock with both convs through Winograd.
    x = synth.normal_bf16((1, 4, 12, 20, 256), 0, "wino/rb/x")
    p = synth.resblock_params(256, 0, "wino/rb")
    pd = {k: (f32_dev(v) if v.dtype == np.float32 else to_dev(v)) for k, v in p.items()}
    u1, u2 = wan.wan_winograd_weights(pd["w1"]), wan.wan_winograd_weights(pd["w2"])
    c1 = torch.zeros((1, 2, 12, 20, 256), dtype=torch.bfloat16, device="cuda")
    c2 = torch.zeros_like(c1)
    outs = [wan.wan_resblock_winograd(to_dev(np.ascontiguousarray(x[:, s:s + 2])), pd, u1, u2, c1, c2, s > 0, groups,
                                      EPS) for s in (0, 2)]
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    r_a, r1, r2 = oracle.resblock(x[:, :2], p, groups, EPS)
    r_b, r1, r2 = oracle.resblock(x[:, 2:], p, groups, EPS, r1, r2)
    conv_close(np.concatenate([bits(o) for o in outs], 1), np.concatenate([r_a, r_b], 1), "winograd resblock")
    assert int(oracle.ulp_distance_bf16(bits(c1), r1).max()) <= 1
    cache2_close(bits(c2), r2, "winograd resblock cache 2")


# ---- GroupNorm statistics from the output transform ----------------------------------------------

def _coef_values(coef):
    """The (S_hi, S_lo, B_hi, B_lo) quadruples as fp64 S = S_hi + S_lo, B = B_hi + B_lo."""
    q = coef.view(torch.float32).cpu().numpy().astype(np.float64).reshape(-1, 4)
    return q[:, 0] + q[:, 1], q[:, 2] + q[:, 3]


def _norm(C, name):
    return synth.normal_f32((C,), 0, f"{name}/gamma", 1.0, 0.1), synth.normal_f32((C,), 0, f"{name}/beta", 0.0, 0.1)


@pytest.mark.parametrize("shape,Cout,groups,coef,cache,residual", [
    ((1, 3, 9, 11, 64), 256, 32, True, True, False),      # odd H and W: tiles of 1 to 4 pixels; 8 per group
    ((2, 2, 5, 7, 64), 512, 32, False, False, True),      # batch 2, 16 channels per group, residual
    ((1, 2, 12, 20, 1024), 1024, 32, True, True, True),   # the widest stage's channels: 32 per group
    ((1, 2, 6, 10, 64), 256, 64, True, False, False),     # 4 per group: one lane per group
    ((1, 2, 6, 10, 64), 256, 4, True, False, False),      # 64 per group: 16 lanes per group
    ((1, 2, 1, 1, 64), 256, 32, True, True, False),       # 1 x 1 frames: one record per frame and group
    ((1, 1, 6, 10, 64), 256, 32, True, True, True),       # one frame with history and residual
])
def test_winograd_statistics(wan, shape, Cout, groups, coef, cache, residual):
    name = f"wino/stats/{shape}/{Cout}/{groups}"
    x, w, g, be, c, b, r = make(shape, Cout, name, coef, cache, True, residual)
    N, T, H, W, Cin = shape
    xd, u = to_dev(x), wan.wan_winograd_weights(to_dev(w))
    k1 = wan.wan_gn_silu_coefficients(xd, f32_dev(g), f32_dev(be), G, EPS) if coef else None
    cd, bd, rd = (None if v is None else to_dev(v) for v in (c, b, r))
    c_plain = torch.empty((N, 2, H, W, Cin), dtype=torch.bfloat16, device="cuda")
    c_st = torch.empty_like(c_plain)
    y_plain = wan.wan_causal_conv3d_winograd(xd, u, k1, bd, rd, cd, c_plain)
    y, st = wan.wan_causal_conv3d_winograd_stats(xd, u, groups, k1, bd, rd, cd, c_st)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    assert torch.equal(y.view(torch.int16), y_plain.view(torch.int16))  # the statistics change nothing
    assert torch.equal(c_st.view(torch.int16), c_plain.view(torch.int16))
    # the next norm's coefficients from them against its own pass over y
    g2, be2 = _norm(Cout, f"{name}/n2")
    k_st = wan.wan_gn_silu_coefficients_from_stats(st, f32_dev(g2), f32_dev(be2), y.shape, groups, EPS)
    k_pass = wan.wan_gn_silu_coefficients(y, f32_dev(g2), f32_dev(be2), groups, EPS)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    s_st, b_st = _coef_values(k_st)
    s_p, b_p = _coef_values(k_pass)
    assert np.max(np.abs(s_st - s_p) / np.abs(s_p)) < 1e-6
    assert np.max(np.abs(b_st - b_p) / (np.abs(b_p) + np.abs(s_p))) < 1e-6
    # the norm applied from them: within one bf16 ulp of the oracle's GroupNorm + SiLU of y
    out = wan.wan_gn_silu_from_stats(y, f32_dev(g2), f32_dev(be2), groups, EPS, st)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    ref = oracle.gn_silu(bits(y), g2, be2, groups, EPS)
    assert int(oracle.ulp_distance_bf16(bits(out), ref).max()) <= 1


def test_winograd_statistics_chunked_equals_unchunked(wan):
    shape, Cout, groups = (1, 6, 10, 14, 64), 256, 32
    x, w, g, be, _, b, _ = make(shape, Cout, "wino/stats/chunks", True, False, True, False)
    g2, be2 = _norm(Cout, "wino/stats/chunks/n2")
    xd, u, bd = to_dev(x), wan.wan_winograd_weights(to_dev(w)), to_dev(b)

    def call(xs, cin, cout):
        k = wan.wan_gn_silu_coefficients(xs, f32_dev(g), f32_dev(be), G, EPS)
        y, st = wan.wan_causal_conv3d_winograd_stats(xs, u, groups, k, bd, None, cin, cout)
        return wan.wan_gn_silu_coefficients_from_stats(st, f32_dev(g2), f32_dev(be2), y.shape, groups, EPS)
    full = call(xd, None, torch.empty((1, 2, 10, 14, 64), dtype=torch.bfloat16, device="cuda"))
    caches = [torch.empty((1, 2, 10, 14, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    parts = [call(xd[:, :3].contiguous(), None, caches[0]), call(xd[:, 3:].contiguous(), caches[0], caches[1])]
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    assert torch.equal(torch.cat(parts), full)


def test_winograd_statistics_of_other_sizes_are_refused(wan):
    # Statistics of 24 x 40 frames (240 tiles per frame and group) read as those of 12 x 20
    # frames: refused, the coefficients untouched.
    x, w, g, be, _, b, _ = make((1, 2, 24, 40, 64), 256, "wino/stats/other", False, False, True, False)
    _, st = wan.wan_causal_conv3d_winograd_stats(to_dev(x), wan.wan_winograd_weights(to_dev(w)), 32, None,
                                                 to_dev(b))
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    k = torch.full((1 * 2 * 256 * 16,), 7, dtype=torch.uint8, device="cuda")
    g2, be2 = _norm(256, "wino/stats/other/n2")
    wan.wan_gn_silu_coefficients_from_stats(st, f32_dev(g2), f32_dev(be2), (1, 2, 12, 20, 256), 32, EPS, k)
    assert wan.wan_device_status() == 1  # WAN_ERR_INVALID_ARG
    assert bool((k == 7).all())


def test_winograd_statistics_with_a_large_mean(wan):
    # Outputs around 1000 (a bias of mean 1000) against a spread of about one: the sums only stay
    # exact because every record is taken around a value of its own group and moved to one shift.
    shape, Cout, groups = (1, 2, 9, 11, 64), 256, 32
    x, w, g, be, c, _, _ = make(shape, Cout, "wino/stats/mean", True, True, False, False)
    b = synth.normal_bf16((Cout,), 0, "wino/stats/mean/b", 1000.0, 1.0)
    xd, u = to_dev(x), wan.wan_winograd_weights(to_dev(w))
    k1 = wan.wan_gn_silu_coefficients(xd, f32_dev(g), f32_dev(be), G, EPS)
    y, st = wan.wan_causal_conv3d_winograd_stats(xd, u, groups, k1, to_dev(b), None, to_dev(c))
    g2, be2 = _norm(Cout, "wino/stats/mean/n2")
    k_st = wan.wan_gn_silu_coefficients_from_stats(st, f32_dev(g2), f32_dev(be2), y.shape, groups, EPS)
    k_pass = wan.wan_gn_silu_coefficients(y, f32_dev(g2), f32_dev(be2), groups, EPS)
    out = wan.wan_gn_silu_from_stats(y, f32_dev(g2), f32_dev(be2), groups, EPS, st)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    assert float(oracle.bf16_to_f64(bits(y)).mean()) > 900.0
    s_st, b_st = _coef_values(k_st)
    s_p, b_p = _coef_values(k_pass)
    assert np.max(np.abs(s_st - s_p) / np.abs(s_p)) < 1e-6
    assert np.max(np.abs(b_st - b_p) / (np.abs(b_p) + np.abs(s_p))) < 1e-6
    ref = oracle.gn_silu(bits(y), g2, be2, groups, EPS)
    assert int(oracle.ulp_distance_bf16(bits(out), ref).max()) <= 1
