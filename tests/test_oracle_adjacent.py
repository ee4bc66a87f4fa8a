"""Pins of the oracle's adjacent decoder steps against facts other than its own formulas: brute
force on tiny inputs, closed forms (frame doubling, a one-frame shift), chunk invariance of the
causal time conv, and reductions to the already pinned causal conv and ResBlock."""
import itertools

import numpy as np

import oracle
from video_vae_decoder_gb300 import synth


def f64(bits):
    return oracle.bf16_to_f64(bits)


def bits_of(values):
    return oracle.round_to_bf16(np.asarray(values, dtype=np.float64))


# ---------------------------------------------------------------- time upsample (3x1x1, x2 frames)

def _time_upsample_loops(x, w, b, cache, first):
    """Pure-Python loops over every output element, independent of the vectorised oracle."""
    N, T, H, W, C = x.shape
    start = 1 if first else 0
    frames = [cache[:, j] if cache is not None else np.zeros((N, H, W, C)) for j in range(2)]
    frames += [x[:, t] for t in range(start, T)]
    nf = T - start
    out = np.zeros((N, start + 2 * nf, H, W, C))
    for n, h, ww in itertools.product(range(N), range(H), range(W)):
        if first:
            out[n, 0, h, ww] = x[n, 0, h, ww]
        for t in range(nf):
            for co in range(2 * C):
                acc = b[co]
                for kt in range(3):
                    for ci in range(C):
                        acc += w[co, kt, ci] * frames[t + kt][n, h, ww, ci]
                out[n, start + 2 * t + co // C, h, ww, co % C] = acc
    return out


def test_time_upsample_matches_loops():
    x = synth.normal_bf16((2, 3, 2, 3, 2), 0, "pin/tu/x")
    w = synth.normal_bf16((4, 3, 2), 0, "pin/tu/w")
    b = synth.normal_bf16((4,), 0, "pin/tu/b")
    c = synth.normal_bf16((2, 2, 2, 3, 2), 0, "pin/tu/c")
    for cache, first in ((None, True), (c, False), (None, False)):
        ref = _time_upsample_loops(f64(x), f64(w), f64(b), None if cache is None else f64(cache), first)
        got = oracle.time_upsample_f64(f64(x), f64(w), f64(b), None if cache is None else f64(cache), first)
        assert got.shape == ref.shape
        assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_time_upsample_frame_doubling_and_shift():
    # w[:, 2] = [I; I] (the current frame to both halves): every frame appears twice, in order.
    C = 3
    x = synth.normal_bf16((1, 4, 2, 2, C), 0, "pin/tu/dbl")
    w = np.zeros((2 * C, 3, C))
    w[:C, 2] = np.eye(C)
    w[C:, 2] = np.eye(C)
    out, _ = oracle.time_upsample(x, bits_of(w), None, None, first=True)
    xs = np.asarray(x)
    expect = np.concatenate([xs[:, :1]] + [np.repeat(xs[:, t:t + 1], 2, axis=1) for t in range(1, 4)], axis=1)
    assert np.array_equal(out, expect)
    # First half = the current frame, second half = the frame before (tap kt = 1): frames
    # x1, x0', x2, x1, x3, x2 where x0' is the zero history before the first chunk's
    # time-upsampled frames (its first frame passes through and is not part of that history).
    w = np.zeros((2 * C, 3, C))
    w[:C, 2] = np.eye(C)
    w[C:, 1] = np.eye(C)
    out, cache = oracle.time_upsample(x, bits_of(w), None, None, first=True)
    zero = np.zeros_like(xs[:, :1])
    expect = np.concatenate([xs[:, :1], xs[:, 1:2], zero, xs[:, 2:3], xs[:, 1:2], xs[:, 3:4], xs[:, 2:3]], axis=1)
    assert np.array_equal(out, expect)
    assert np.array_equal(cache, xs[:, 2:4])


def test_time_upsample_chunked_equals_unchunked():
    x = synth.normal_bf16((1, 7, 3, 2, 4), 0, "pin/tu/chunks")
    w = synth.normal_bf16((8, 3, 4), 0, "pin/tu/chunks/w", 0.0, 0.3)
    b = synth.normal_bf16((8,), 0, "pin/tu/chunks/b")
    full, c_full = oracle.time_upsample(x, w, b, None, first=True)
    parts, cache = [], None
    for i, (s0, s1) in enumerate(((0, 1), (1, 4), (4, 7))):  # a one-frame first chunk, then 3 + 3
        o, cache = oracle.time_upsample(np.ascontiguousarray(np.asarray(x)[:, s0:s1]), w, b, cache, first=(i == 0))
        parts.append(o)
    assert np.array_equal(np.concatenate(parts, axis=1), full)
    assert np.array_equal(cache, c_full)
    assert full.shape[1] == 1 + 2 * 6


# ---------------------------------------------------------------- 1x1x1 shortcut and bias folding

def test_conv1x1_matches_loops_and_the_centre_tap_conv():
    x = synth.normal_bf16((1, 2, 2, 3, 3), 0, "pin/sc/x")
    w = synth.normal_bf16((5, 3), 0, "pin/sc/w")
    got = oracle.conv1x1(x, w)
    xf, wf = f64(x), f64(w)
    loops = np.zeros((1, 2, 2, 3, 5))
    for t, h, ww, co in itertools.product(range(2), range(2), range(3), range(5)):
        loops[0, t, h, ww, co] = sum(wf[co, ci] * xf[0, t, h, ww, ci] for ci in range(3))
    assert np.array_equal(got, bits_of(loops))
    # the causal 3x3x3 conv whose only non-zero tap is the current frame's centre
    w3 = np.zeros((5, 3, 3, 3, 3), np.uint16)
    w3[:, 2, 1, 1, :] = np.asarray(w)
    y, _ = oracle.causal_conv3d(x, w3)
    assert np.array_equal(got, y)


def test_fold_bias_rounds_the_sum_once():
    one, half_ulp = bits_of([1.0]), bits_of([2.0 ** -8])
    assert oracle.bf16_to_f64(oracle.fold_bias(one, half_ulp))[0] == 1.0            # tie to even: 1
    three_q = bits_of([1.5 * 2.0 ** -8])
    assert oracle.bf16_to_f64(oracle.fold_bias(one, three_q))[0] == 1.0 + 2.0 ** -7  # above the tie
    a, b = bits_of([0.75]), bits_of([-0.25])
    assert oracle.bf16_to_f64(oracle.fold_bias(a, b))[0] == 0.5                     # exact sums stay


def test_resblock_shortcut_with_identity_equals_resblock():
    C = 64
    x = synth.normal_bf16((1, 2, 4, 4, C), 0, "pin/rbs/x")
    p = synth.resblock_params(C, 0, "pin/rbs")
    eye = bits_of(np.eye(C))
    zero = np.zeros(C, np.uint16)
    out_s, c1_s, c2_s = oracle.resblock_shortcut(x, p, eye, zero, 32, float(np.float32(1e-6)))
    out, c1, c2 = oracle.resblock(x, p, 32, float(np.float32(1e-6)))
    assert np.array_equal(out_s, out) and np.array_equal(c1_s, c1) and np.array_equal(c2_s, c2)


def test_time_upsample_matches_torch_conv3d():
    # The time conv against PyTorch's conv3d with a (3, 1, 1) kernel on [history; frames], fp64.
    import torch
    N, T, H, W, C = 2, 3, 3, 4, 8
    x = oracle.bf16_to_f64(synth.normal_bf16((N, T, H, W, C), 0, "t/tu/torch/x"))
    w = oracle.bf16_to_f64(synth.normal_bf16((2 * C, 3, C), 0, "t/tu/torch/w", 0.0, 0.2))
    b = oracle.bf16_to_f64(synth.normal_bf16((2 * C,), 0, "t/tu/torch/b", 0.0, 0.1))
    cache = oracle.bf16_to_f64(synth.normal_bf16((N, 2, H, W, C), 0, "t/tu/torch/c"))
    got = oracle.time_upsample_f64(x, w, b, cache, first=False)
    p = torch.from_numpy(np.concatenate([cache, x], 1)).permute(0, 4, 1, 2, 3)          # N C T H W
    z = torch.nn.functional.conv3d(p, torch.from_numpy(w).permute(0, 2, 1)[..., None, None], torch.from_numpy(b))
    z = z.permute(0, 2, 3, 4, 1).numpy()                                              # [N, T, H, W, 2C]
    ref = np.stack([z[..., :C], z[..., C:]], 2).reshape(N, 2 * T, H, W, C)            # half i -> frame 2t + i
    assert np.max(np.abs(got - ref)) < 1e-12
