"""The decoder steps next to the ResBlock, on the GPU: the causal 3x1x1 time upsample with
frame-interleaved output, the 1x1x1 shortcut, the folded shortcut bias and the channel-changing
ResBlock; each against the oracle, with chunked == unchunked bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, f32_dev, bits, conv_close, cache2_close
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))


def tu_inputs(shape, name):
    N, T, H, W, C = shape
    x = synth.normal_bf16(shape, 0, f"{name}/x")
    w = synth.normal_bf16((2 * C, 3, C), 0, f"{name}/w", 0.0, float(np.sqrt(1.0 / (3 * C))))
    b = synth.normal_bf16((2 * C,), 0, f"{name}/b", 0.0, 0.01)
    c = synth.normal_bf16((N, 2, H, W, C), 0, f"{name}/c")
    return x, w, b, c


def same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("shape,first,history", [
    ((1, 3, 10, 20, 256), True, False),    # first chunk: frame 0 passes through, ragged tiles
    ((2, 4, 9, 17, 256), False, True),     # batch 2 with history
    ((1, 1, 8, 16, 256), False, True),     # one frame: the history shifts by one
    ((1, 1, 8, 16, 256), True, False),     # the first chunk of one frame: only the pass-through
    ((1, 2, 12, 33, 512), False, False),   # no history, two N blocks per channel half
    ((1, 2, 1, 1, 256), False, True),      # 1 x 1 frames with history
    ((1, 3, 1, 5, 256), True, False),      # one-pixel-high frames, first chunk
])
def test_time_upsample_matches_oracle(wan, shape, first, history):
    x, w, b, c = tu_inputs(shape, f"tu/{shape}/{first}/{history}")
    c_out = torch.empty((shape[0], 2) + shape[2:], dtype=torch.bfloat16, device="cuda")
    y = wan.wan_time_upsample(to_dev(x), to_dev(w), to_dev(b), first, to_dev(c) if history else None, c_out)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    ref, c_ref = oracle.time_upsample(x, w, b, c if history else None, first)
    got = bits(y)
    assert got.shape == ref.shape
    start = 1 if first else 0
    if first:
        assert np.array_equal(got[:, :1], ref[:, :1])  # the passed-through frame is a copy
    if got.shape[1] > start:
        conv_close(got[:, start:], ref[:, start:], "time upsample")
    assert np.array_equal(bits(c_out), c_ref)


def test_time_upsample_chunked_equals_unchunked(wan):
    x, w, b, _ = tu_inputs((1, 7, 12, 20, 256), "tu/chunks")
    xd, wd, bd = to_dev(x), to_dev(w), to_dev(b)
    c_full = torch.empty((1, 2, 12, 20, 256), dtype=torch.bfloat16, device="cuda")
    full = wan.wan_time_upsample(xd, wd, bd, True, None, c_full)
    cache = torch.empty_like(c_full)
    parts = []
    for i, (s0, s1) in enumerate(((0, 1), (1, 4), (4, 7))):  # a one-frame first chunk, then 3 + 3
        parts.append(wan.wan_time_upsample(xd[:, s0:s1].contiguous(), wd, bd, i == 0, cache if i else None, cache))
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    assert same(torch.cat(parts, 1), full)
    assert same(cache, c_full)


def test_time_upsample_decode_size_sampled(wan):
    # [1, 4, 44, 78, 512] with history, 512 -> 1024 channels: sampled outputs against the oracle's sum.
    shape = (1, 4, 44, 78, 512)
    x, w, b, c = tu_inputs(shape, "tu/big")
    y = wan.wan_time_upsample(to_dev(x), to_dev(w), to_dev(b), False, to_dev(c))
    torch.cuda.synchronize()
    got = oracle.bf16_to_f64(bits(y))
    xf, wf, bf, cf = (oracle.bf16_to_f64(a) for a in (x, w, b, c))
    P = np.concatenate([cf, xf], axis=1)
    rng = np.random.default_rng(1)
    pts = np.stack([rng.integers(0, 4, 400), rng.integers(0, 44, 400), rng.integers(0, 78, 400)], 1)
    ref = np.stack([bf + sum(wf[:, kt] @ P[0, t + kt, h, ww] for kt in range(3)) for t, h, ww in pts])
    out = np.stack([np.concatenate([got[0, 2 * t, h, ww], got[0, 2 * t + 1, h, ww]]) for t, h, ww in pts])
    conv_close(oracle.round_to_bf16(out), ref, "time upsample, sampled")


def test_time_upsample_bench_size_every_element(wan):
    # The adjacent-step shape bench.py times, [1, 4, 44, 78, 1024] -> [1, 8, 44, 78, 1024] with
    # history: every output element against the oracle (its two frames per CTA, the split last round).
    shape = (1, 4, 44, 78, 1024)
    x, w, b, c = tu_inputs(shape, "tu/bench")
    c_out = torch.empty((1, 2, 44, 78, 1024), dtype=torch.bfloat16, device="cuda")
    y = wan.wan_time_upsample(to_dev(x), to_dev(w), to_dev(b), False, to_dev(c), c_out)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    ref, c_ref = oracle.time_upsample(x, w, b, c, False)
    conv_close(bits(y), ref, "time upsample, bench size")
    assert np.array_equal(bits(c_out), c_ref)


@pytest.mark.parametrize("shape,Cout", [((1, 2, 12, 33, 128), 256), ((2, 3, 9, 17, 256), 512),
                                        ((1, 2, 7, 19, 192), 256)])  # an odd count of 64-channel blocks
def test_conv1x1_matches_oracle(wan, shape, Cout):
    x = synth.normal_bf16(shape, 0, f"c11/{shape}/x")
    w = synth.normal_bf16((Cout, shape[-1]), 0, f"c11/{shape}/w", 0.0, float(np.sqrt(1.0 / shape[-1])))
    y = wan.wan_conv1x1(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    conv_close(bits(y), oracle.conv1x1(x, w), "1x1x1")


def test_fold_bias_bit_exact(wan):
    b2 = synth.normal_bf16((1024,), 0, "fold/b2")
    bs = synth.normal_bf16((1024,), 0, "fold/bs", 0.0, 0.3)
    # ties of round-to-nearest-even and a large exponent gap
    b2[:3] = oracle.round_to_bf16(np.array([1.0, 1.0, 1.0]))
    bs[:3] = oracle.round_to_bf16(np.array([2.0 ** -8, 1.5 * 2.0 ** -8, 2.0 ** -30]))
    got = wan.wan_fold_bias(to_dev(b2), to_dev(bs))
    torch.cuda.synchronize()
    assert np.array_equal(bits(got), oracle.fold_bias(b2, bs))


def _shortcut_params(Cin, Cout, name):
    p = synth.resblock_params(Cout, 0, name)
    p["gamma1"] = synth.normal_f32((Cin,), 0, f"{name}/g1in", 1.0, 0.1)
    p["beta1"] = synth.normal_f32((Cin,), 0, f"{name}/b1in", 0.0, 0.1)
    p["w1"] = synth.normal_bf16((Cout, 3, 3, 3, Cin), 0, f"{name}/w1in", 0.0, float(np.sqrt(1.0 / (27 * Cin))))
    w_sc = synth.normal_bf16((Cout, Cin), 0, f"{name}/wsc", 0.0, float(np.sqrt(1.0 / Cin)))
    b_sc = synth.normal_bf16((Cout,), 0, f"{name}/bsc", 0.0, 0.01)
    return p, w_sc, b_sc


def _dev(p):
    return {k: (f32_dev(v) if v.dtype == np.float32 else to_dev(v)) for k, v in p.items()}


def _run_shortcut(wan, x_dev, pd, w_sc_dev, Cin, Cout, chunk):
    N, T, H, W, _ = x_dev.shape
    c1 = torch.zeros((N, 2, H, W, Cin), dtype=torch.bfloat16, device="cuda")
    c2 = torch.zeros((N, 2, H, W, Cout), dtype=torch.bfloat16, device="cuda")
    outs = [wan.wan_resblock_shortcut(x_dev[:, s:s + chunk].contiguous(), pd, w_sc_dev, c1, c2, i > 0, 32, EPS)
            for i, s in enumerate(range(0, T, chunk))]
    torch.cuda.synchronize()
    return torch.cat(outs, 1), c1, c2


def test_resblock_shortcut_matches_oracle(wan):
    Cin, Cout = 128, 256
    x = synth.normal_bf16((1, 5, 12, 20, Cin), 0, "rbsc/x")
    p, w_sc, b_sc = _shortcut_params(Cin, Cout, "rbsc")
    pd = _dev(p)
    pd["b2"] = wan.wan_fold_bias(pd["b2"], to_dev(b_sc))  # prepare time
    out, c1, c2 = _run_shortcut(wan, to_dev(x), pd, to_dev(w_sc), Cin, Cout, 3)
    assert wan.wan_device_status() == 0
    r_a, r1, r2 = oracle.resblock_shortcut(x[:, :3], p, w_sc, b_sc, 32, EPS)
    r_b, r1, r2 = oracle.resblock_shortcut(x[:, 3:], p, w_sc, b_sc, 32, EPS, r1, r2)
    conv_close(bits(out), np.concatenate([r_a, r_b], 1), "channel-changing resblock")
    assert int(oracle.ulp_distance_bf16(bits(c1), r1).max()) <= 1
    cache2_close(bits(c2), r2, "cache 2")


def test_resblock_shortcut_chunked_equals_unchunked(wan):
    Cin, Cout = 256, 512
    x = to_dev(synth.normal_bf16((1, 8, 16, 24, Cin), 0, "rbsc/chunks/x"))
    p, w_sc, b_sc = _shortcut_params(Cin, Cout, "rbsc/chunks")
    pd = _dev(p)
    pd["b2"] = wan.wan_fold_bias(pd["b2"], to_dev(b_sc))
    full = _run_shortcut(wan, x, pd, to_dev(w_sc), Cin, Cout, 8)
    part = _run_shortcut(wan, x, pd, to_dev(w_sc), Cin, Cout, 4)
    assert wan.wan_device_status() == 0
    for a, b in zip(full, part):
        assert same(a, b)
