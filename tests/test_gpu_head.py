"""The causal conv to 12 channels (the output head: temporal GEMM to 112 columns + 3x3 stencil in
the epilogue) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, bits, conv_close
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu


def make(shape, name, bias, residual, cache):
    N, T, H, W, Cin = shape
    a = synth.normal_bf16(shape, 0, f"{name}/a")
    w = synth.normal_bf16((12, 3, 3, 3, Cin), 0, f"{name}/w", 0.0, float(np.sqrt(1.0 / (27 * Cin))))
    b = synth.normal_bf16((12,), 0, f"{name}/b", 0.0, 0.01) if bias else None
    r = synth.normal_bf16((N, T, H, W, 12), 0, f"{name}/r") if residual else None
    c = synth.normal_bf16((N, 2, H, W, Cin), 0, f"{name}/c") if cache else None
    return a, w, b, r, c


def f64(x):
    return None if x is None else oracle.bf16_to_f64(x)


@pytest.mark.parametrize("shape,bias,residual,cache", [
    ((1, 4, 10, 24, 64), False, False, False),
    ((1, 5, 13, 300, 256), True, False, True),      # 3 strips (ragged), odd T (a lone last frame)
    ((2, 3, 7, 130, 128), True, True, False),       # batch 2, 2 strips, residual
    ((1, 1, 1, 5, 64), False, False, True),         # one row, one frame from the cache
    ((1, 2, 2, 127, 192), True, False, False),      # two rows; width just over one strip
    ((1, 6, 40, 60, 256), False, False, False),     # several row bands
    # rows issued by compile-time code: the first quad of a chunk without history (input frames
    # t..t+3) and quads with all six input frames, for 2, 3 and 1 blocks of 64 input channels
    ((1, 8, 9, 40, 128), True, False, False),
    ((1, 4, 6, 50, 192), False, False, True),
    ((1, 8, 5, 20, 64), False, True, True),
    ((1, 3, 1, 1, 64), True, False, True),          # 1 x 1 frames: only the centre stencil term
    ((1, 2, 7, 1, 128), False, True, False),        # one-pixel-wide frames
])
def test_head_small(wan, shape, bias, residual, cache):
    a, w, b, r, c = make(shape, f"head/{shape}", bias, residual, cache)
    y = wan.wan_causal_conv3d(to_dev(a), to_dev(w), None if b is None else to_dev(b),
                              None if r is None else to_dev(r), None if c is None else to_dev(c))
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    ref = oracle.causal_conv3d_f64(f64(a), f64(w), f64(b), f64(r), f64(c))
    conv_close(bits(y), ref, "head")


def test_head_chunked_equals_unchunked(wan):
    a, w, b, _, _ = make((1, 12, 20, 140, 256), "head/chunks", True, False, False)
    ad, wd, bd = to_dev(a), to_dev(w), to_dev(b)
    full = wan.wan_causal_conv3d(ad, wd, bd)
    cache = torch.empty((1, 2, 20, 140, 256), dtype=torch.bfloat16, device="cuda")
    parts = []
    for s in range(0, 12, 4):
        cin = None if s == 0 else cache
        parts.append(wan.wan_causal_conv3d(ad[:, s:s + 4].contiguous(), wd, bd, None, cin, cache))
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(parts, 1).view(torch.int16), full.view(torch.int16))
