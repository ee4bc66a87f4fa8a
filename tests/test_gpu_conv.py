"""Causal 3x3x3 convolution on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, bits, conv_close
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu


def make(shape, Cout, name, bias=True, residual=False, cache=False, seed=0):
    N, T, H, W, Cin = shape
    a = synth.normal_bf16(shape, seed, f"{name}/a")
    w = synth.normal_bf16((Cout, 3, 3, 3, Cin), seed, f"{name}/w", 0.0, float(np.sqrt(1.0 / (27 * Cin))))
    b = synth.normal_bf16((Cout,), seed, f"{name}/b", 0.0, 0.01) if bias else None
    r = synth.normal_bf16((N, T, H, W, Cout), seed, f"{name}/r") if residual else None
    c = synth.normal_bf16((N, 2, H, W, Cin), seed, f"{name}/c") if cache else None
    return a, w, b, r, c


def run(wan, a, w, b, r, c, with_cache_out=True):
    N, T, H, W, Cin = a.shape
    cout = torch.empty((N, 2, H, W, Cin), dtype=torch.bfloat16, device="cuda") if with_cache_out else None
    y = wan.wan_causal_conv3d(to_dev(a), to_dev(w), None if b is None else to_dev(b),
                              None if r is None else to_dev(r), None if c is None else to_dev(c), cout)
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    return bits(y), (bits(cout) if with_cache_out else None)


@pytest.mark.parametrize("shape,Cout,bias,residual,cache", [
    ((1, 3, 16, 16, 64), 64, True, False, False),     # the tiny ResBlock's conv
    ((1, 3, 16, 16, 64), 64, True, True, True),
    ((1, 5, 11, 21, 128), 96, True, False, True),     # ragged pixel tiles, N block wider than Cout
    ((2, 3, 9, 14, 64), 320, False, True, True),      # batch 2, two N blocks (second ragged)
    ((1, 4, 10, 24, 64), 12, False, False, False),    # head-like: 12 output channels
    ((1, 1, 8, 8, 64), 64, True, False, True),        # a single frame: both history frames from the cache
    ((1, 2, 5, 5, 192), 256, True, True, False),
    # CTA-pair path (Cout >= 256, 8 x 16-pixel tiles with their halo boxes):
    ((1, 3, 19, 37, 128), 256, True, True, False),    # ragged rows and columns, odd tile count, no history
    ((1, 4, 8, 16, 64), 512, False, False, True),     # exactly one tile per frame, two N blocks
    ((1, 1, 3, 50, 64), 256, True, False, False),     # one frame, fewer rows than a tile, 4 tiles wide
    ((2, 2, 12, 33, 64), 256, True, True, True),      # batch 2: tile pairs that cross batch items
    # degenerate frames: every tile mostly outside the frame, only some taps inside it
    ((1, 2, 1, 1, 64), 256, True, True, True),        # 1 x 1 frames on the CTA-pair path: the centre taps
    ((1, 3, 1, 9, 64), 256, True, False, True),       # one-pixel-high frames
    ((1, 2, 9, 1, 64), 256, False, True, True),       # one-pixel-wide frames
    ((1, 2, 1, 1, 64), 64, True, True, True),         # 1 x 1 frames on the one-CTA kernel
])
def test_conv_small(wan, shape, Cout, bias, residual, cache):
    a, w, b, r, c = make(shape, Cout, f"conv/{shape}/{Cout}", bias, residual, cache)
    got, cout = run(wan, a, w, b, r, c)
    ref, ref_cache = oracle.causal_conv3d(a, w, b, r, c)
    conv_close(got, oracle.causal_conv3d_f64(oracle.bf16_to_f64(a), oracle.bf16_to_f64(w),
                                             None if b is None else oracle.bf16_to_f64(b),
                                             None if r is None else oracle.bf16_to_f64(r),
                                             None if c is None else oracle.bf16_to_f64(c)), "conv")
    assert np.array_equal(cout, ref_cache)


def test_conv_chunked_equals_unchunked(wan):
    shape = (1, 12, 12, 20, 128)
    a, w, b, _, _ = make(shape, 128, "conv/chunks")
    full, full_cache = run(wan, a, w, b, None, None)
    parts, cache = [], None
    for s in range(0, 12, 4):
        y, cache = run(wan, a[:, s:s + 4], w, b, None, cache)
        parts.append(y)
    assert np.array_equal(np.concatenate(parts, 1), full)
    assert np.array_equal(cache, full_cache)


def test_conv_pair_chunked_equals_unchunked(wan):
    # The CTA-pair path: chunks of 4 frames give the same bits as one 8-frame call.
    shape = (1, 8, 10, 30, 64)
    a, w, b, _, _ = make(shape, 256, "conv/pair-chunks")
    full, full_cache = run(wan, a, w, b, None, None)
    parts, cache = [], None
    for s in range(0, 8, 4):
        y, cache = run(wan, a[:, s:s + 4], w, b, None, cache)
        parts.append(y)
    assert np.array_equal(np.concatenate(parts, 1), full)
    assert np.array_equal(cache, full_cache)


def test_conv_cache_aliasing_in_place(wan):
    # cache_out may be cache_in: it is updated after the convolution has read it (T = 1 and 3).
    for T in (1, 3):
        a, w, b, _, c = make((1, T, 6, 8, 64), 64, f"conv/alias{T}", cache=True)
        ref, ref_cache = oracle.causal_conv3d(a, w, b, None, c)
        cd = to_dev(c)
        y = wan.wan_causal_conv3d(to_dev(a), to_dev(w), to_dev(b), None, cd, cd)
        torch.cuda.synchronize()
        assert np.array_equal(bits(cd), ref_cache)
        conv_close(bits(y), ref, "alias")


def test_conv_c1024_split_last_round_equals_chunks(wan):
    # [1, 4, 44, 78, 1024]: 240 items (pixel-tile pairs x 4 blocks of 256 output channels). On 76
    # CTA pairs the last round holds 12 items, which run as 24 halves of 128 channels; two 2-frame
    # chunks (120 items, a last round of 44) run whole. Both must give the same bits.
    shape = (1, 4, 44, 78, 1024)
    a, w, b, _, _ = make(shape, 1024, "conv/split")
    full, full_cache = run(wan, a, w, b, None, None)
    parts, cache = [], None
    for s in range(0, 4, 2):
        y, cache = run(wan, a[:, s:s + 2], w, b, None, cache)
        parts.append(y)
    assert np.array_equal(np.concatenate(parts, 1), full)
    assert np.array_equal(cache, full_cache)
