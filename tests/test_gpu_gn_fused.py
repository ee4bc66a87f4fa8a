"""GroupNorm + SiLU from the statistics that the CTA-pair conv emits with its output, on the GPU.
Emitting them leaves the conv's output unchanged bit for bit; the norm computed from them is
within one bf16 ulp of the oracle's GroupNorm + SiLU of that output; and it does not depend on
how the frames are chunked."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, f32_dev, bits, conv_close
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


# ---- the norm-prologue conv that emits the statistics of its own output --------------------------

def prologue_inputs(shape, Cout, name, cache=True):
    N, T, H, W, Cin = shape
    x = synth.normal_bf16(shape, 0, f"{name}/x", 0.2, 1.1)
    g, be = norm_params(Cin, f"{name}/n1")
    w = synth.normal_bf16((Cout, 3, 3, 3, Cin), 0, f"{name}/w", 0.0, float(np.sqrt(1.0 / (27 * Cin))))
    b = synth.normal_bf16((Cout,), 0, f"{name}/b", 0.0, 0.01)
    c = synth.normal_bf16((N, 2, H, W, Cin), 0, f"{name}/c", 0.1, 0.6) if cache else None
    return x, g, be, w, b, c


def coef_values(coef):
    """The (S_hi, S_lo, B_hi, B_lo) quadruples as fp64 S = S_hi + S_lo, B = B_hi + B_lo."""
    q = coef.view(torch.float32).cpu().numpy().astype(np.float64).reshape(-1, 4)
    return q[:, 0] + q[:, 1], q[:, 2] + q[:, 3]


@pytest.mark.parametrize("shape,Cout,groups,residual", [
    ((1, 3, 12, 20, 256), 256, 32, True),     # 16 x 8 tiles (3 per frame against 4), residual
    ((1, 2, 24, 40, 256), 256, 32, False),    # 8 x 16 tiles (9 per frame against 10)
    ((2, 2, 9, 17, 128), 512, 32, False),     # batch 2, two N blocks, 16 channels per group
    ((1, 1, 10, 20, 256), 256, 64, True),     # one frame, 4 channels per group
])
def test_gn_input_conv_statistics(wan, shape, Cout, groups, residual):
    name = f"gninst/{shape}/{Cout}/{groups}"
    x, g, be, w, b, c = prologue_inputs(shape, Cout, name)
    N, T, H, W, Cin = shape
    xd, wd, bd, cd = to_dev(x), to_dev(w), to_dev(b), to_dev(c)
    rd = to_dev(synth.normal_bf16((N, T, H, W, Cout), 0, f"{name}/r")) if residual else None
    coef = wan.wan_gn_silu_coefficients(xd, f32_dev(g), f32_dev(be), 32, EPS)
    c_plain, c_st = torch.empty_like(cd), torch.empty_like(cd)
    y_plain = wan.wan_causal_conv3d_gn_input(xd, coef, wd, bd, rd, cd, cache_out=c_plain)
    y, st = wan.wan_causal_conv3d_gn_input_stats(xd, coef, wd, groups, bd, rd, cd, cache_out=c_st)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y_plain.view(torch.int16))
    assert torch.equal(c_st.view(torch.int16), c_plain.view(torch.int16))
    # the next norm's coefficients from the statistics against its own pass over y
    g2, be2 = norm_params(Cout, f"{name}/n2")
    k_st = wan.wan_gn_silu_coefficients_from_stats(st, f32_dev(g2), f32_dev(be2), y.shape, groups, EPS)
    k_pass = wan.wan_gn_silu_coefficients(y, f32_dev(g2), f32_dev(be2), groups, EPS)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    s_st, b_st = coef_values(k_st)
    s_p, b_p = coef_values(k_pass)
    assert np.max(np.abs(s_st - s_p) / np.abs(s_p)) < 1e-6
    assert np.max(np.abs(b_st - b_p) / (np.abs(b_p) + np.abs(s_p))) < 1e-6
    # the norm applied from them: within one bf16 ulp of the oracle's GroupNorm + SiLU of y
    out = wan.wan_gn_silu_from_stats(y, f32_dev(g2), f32_dev(be2), groups, EPS, st)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    ref = oracle.gn_silu(bits(y), g2, be2, groups, EPS)
    assert int(oracle.ulp_distance_bf16(bits(out), ref).max()) <= 1


def test_gn_input_conv_statistics_chunked_equals_unchunked(wan):
    shape, Cout, groups = (1, 6, 12, 20, 256), 256, 32
    x, g, be, w, b, _ = prologue_inputs(shape, Cout, "gninst/chunks", cache=False)
    g2, be2 = norm_params(Cout, "gninst/chunks/n2")
    xd, wd, bd, gd, bed = to_dev(x), to_dev(w), to_dev(b), f32_dev(g), f32_dev(be)

    def call(xs, cin, cout):
        coef = wan.wan_gn_silu_coefficients(xs, gd, bed, 32, EPS)
        y, st = wan.wan_causal_conv3d_gn_input_stats(xs, coef, wd, groups, bd, None, cin, cache_out=cout)
        return wan.wan_gn_silu_coefficients_from_stats(st, f32_dev(g2), f32_dev(be2), y.shape, groups, EPS)
    full = call(xd, None, torch.empty((1, 2, 12, 20, 256), dtype=torch.bfloat16, device="cuda"))
    cache = torch.empty((1, 2, 12, 20, 256), dtype=torch.bfloat16, device="cuda")
    parts = [call(xd[:, s:s + 3].contiguous(), None if s == 0 else cache, cache) for s in (0, 3)]
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    assert torch.equal(torch.cat(parts), full)


def test_coefficients_from_a_buffer_without_statistics_are_refused(wan):
    # A zero-filled buffer has no record count: the call writes nothing and the device status says so.
    shape, groups = (1, 2, 12, 20, 256), 32
    st = torch.zeros(wan.wan_workspace_size(wan.WAN_OP_GN_STATS, *shape, 256, groups), dtype=torch.uint8, device="cuda")
    g, be = norm_params(256, "gninst/bad")
    coef = torch.full((1 * 2 * 256 * 16,), 7, dtype=torch.uint8, device="cuda")
    wan.wan_gn_silu_coefficients_from_stats(st, f32_dev(g), f32_dev(be), shape, groups, EPS, coef)
    assert wan.wan_device_status() == 1  # WAN_ERR_INVALID_ARG
    assert bool((coef == 7).all())
    assert wan.wan_device_status() == 0  # read and cleared


def test_resblock_chain_with_statistics_matches_oracle(wan):
    # Two C=256 ResBlocks over two 2-frame chunks as a decoder stage runs them with the statistics
    # passed along: block 0's first norm from its own pass, every later norm from the statistics
    # of the conv that wrote its input.
    shape, groups = (1, 4, 12, 20, 256), 32
    N, T, H, W, C = shape
    x = synth.normal_bf16(shape, 0, "gninst/chain/x")
    ps = [synth.resblock_params(C, 0, f"gninst/chain/block{i}") for i in range(2)]
    pd = [{k: (f32_dev(v) if v.dtype == np.float32 else to_dev(v)) for k, v in p.items()} for p in ps]
    caches = [[torch.zeros((N, 2, H, W, C), dtype=torch.bfloat16, device="cuda") for _ in range(2)] for _ in ps]
    alt = [[torch.zeros((N, 2, H, W, C), dtype=torch.bfloat16, device="cuda") for _ in range(2)] for _ in ps]
    outs = []
    for s in (0, 2):
        cur = to_dev(np.ascontiguousarray(x[:, s:s + 2]))
        st = None
        for i, p in enumerate(pd):
            c1 = wan.wan_gn_silu_coefficients(cur, p["gamma1"], p["beta1"], groups, EPS) if st is None else \
                wan.wan_gn_silu_coefficients_from_stats(st, p["gamma1"], p["beta1"], cur.shape, groups, EPS)
            h, st_h = wan.wan_causal_conv3d_gn_input_stats(cur, c1, p["w1"], groups, p["b1"], None, caches[i][0],
                                                          cache_out=alt[i][0])
            c2 = wan.wan_gn_silu_coefficients_from_stats(st_h, p["gamma2"], p["beta2"], h.shape, groups, EPS)
            cur, st = wan.wan_causal_conv3d_gn_input_stats(h, c2, p["w2"], groups, p["b2"], cur, caches[i][1],
                                                          cache_out=alt[i][1])
            caches[i], alt[i] = alt[i], caches[i]  # the new histories are read by the next chunk
        outs.append(bits(cur))
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    ref, state = [], [(None, None), (None, None)]
    for s in (0, 2):
        h = np.ascontiguousarray(x[:, s:s + 2])
        for i, p in enumerate(ps):
            h, c1o, c2o = oracle.resblock(h, p, groups, EPS, *state[i])
            state[i] = (c1o, c2o)
        ref.append(h)
    conv_close(np.concatenate(outs, 1), np.concatenate(ref, 1), "resblock chain with statistics")


def test_coefficients_from_statistics_of_other_sizes_are_refused(wan):
    # Statistics written for 24 x 40 frames (36 records per frame and group) read as those of
    # 12 x 20 frames (16 or 12): refused, the coefficients untouched.
    x, g, be, w, b, c = prologue_inputs((1, 2, 24, 40, 256), 256, "gninst/other")
    xd = to_dev(x)
    coef = wan.wan_gn_silu_coefficients(xd, f32_dev(g), f32_dev(be), 32, EPS)
    _, st = wan.wan_causal_conv3d_gn_input_stats(xd, coef, to_dev(w), 32, to_dev(b), None, to_dev(c))
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    k = torch.full((1 * 2 * 256 * 16,), 7, dtype=torch.uint8, device="cuda")
    g2, be2 = norm_params(256, "gninst/other/n2")
    wan.wan_gn_silu_coefficients_from_stats(st, f32_dev(g2), f32_dev(be2), (1, 2, 12, 20, 256), 32, EPS, k)
    assert wan.wan_device_status() == 1  # WAN_ERR_INVALID_ARG
    assert bool((k == 7).all())
