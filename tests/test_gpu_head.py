"""The causal conv to 12 channels (the output head: temporal GEMM to 112 columns + 3x3 stencil in
the epilogue) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, bits, conv_close, sample_points
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


def test_head_full_size_sampled(wan):
    # [1, 16, 704, 1248, 256] ~ N(0,1) -> 12 channels, weights N(0, 1/(27*256)), zero history.
    shape = (1, 16, 704, 1248, 256)
    N, T, H, W, C = shape
    name = "head/full/x"
    x = synth.normal_torch(shape, 0, name, device="cuda", dtype=torch.bfloat16)
    w = synth.normal_bf16((12, 3, 3, 3, C), 0, "head/full/w", 0.0, float(np.sqrt(1.0 / (27 * C))))
    y = wan.wan_causal_conv3d(x, to_dev(w))
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    got_all = bits(y)
    rng = np.random.default_rng(1)
    pts = sample_points(rng, N, T, H, W, 96)
    patches, sel = [], []
    for n, t, h, ww in pts:
        patch = np.zeros((3, 3, 3, C))
        for kt in range(3):
            tau = t + kt - 2
            if tau < 0:
                continue
            for kh in range(3):
                hh = h + kh - 1
                if not 0 <= hh < H:
                    continue
                for kw in range(3):
                    wc = ww + kw - 1
                    if not 0 <= wc < W:
                        continue
                    base = (((n * T + tau) * H + hh) * W + wc) * C
                    vals = synth.f32_to_bf16_bits(
                        synth.standard_normal_at(0, name, np.arange(base, base + C)).astype(np.float32))
                    dev_vals = x[n, tau, hh, wc].view(torch.int16).cpu().numpy().view(np.uint16)
                    assert np.array_equal(vals, dev_vals), "device and host generators disagree"
                    patch[kt, kh, kw] = oracle.bf16_to_f64(vals)
        patches.append(patch)
        sel.append(got_all[n, t, h, ww])
    ref = oracle.conv_at_points_f64(np.stack(patches), oracle.bf16_to_f64(w))
    conv_close(np.stack(sel), ref, "head full size")
