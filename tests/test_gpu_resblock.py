"""Causal ResBlock on the GPU: oracle parity, cache chaining, chunked == unchunked bits."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, f32_dev, bits, conv_close, cache2_close
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))


def dev_params(p):
    return {k: (f32_dev(v) if v.dtype == np.float32 else to_dev(v)) for k, v in p.items()}


def check_caches(c1, c2, r1, r2):
    # cache 1 = last frames of silu(gn1(x)): within one bf16 ulp of the oracle. cache 2 = last
    # frames of silu(gn2(h)): h carries the convolution's error, so the conv criterion applies.
    assert int(oracle.ulp_distance_bf16(bits(c1), r1).max()) <= 1
    cache2_close(bits(c2), r2, "cache 2")


def run_chunks(wan, x_dev, params, G, chunk, caches=None):
    N, T, H, W, C = x_dev.shape
    c1 = torch.zeros((N, 2, H, W, C), dtype=torch.bfloat16, device="cuda")
    c2 = torch.zeros_like(c1)
    outs = []
    for i, s in enumerate(range(0, T, chunk)):
        outs.append(wan.wan_resblock(x_dev[:, s:s + chunk].contiguous(), params, c1, c2, i > 0, G, EPS))
    torch.cuda.synchronize()
    return torch.cat(outs, 1), c1, c2


def test_resblock_tiny_matches_oracle(wan):
    # [1, 3, 16, 16, 64], zero caches, GroupNorm 32 groups, eps 1e-6
    x = synth.normal_bf16((1, 3, 16, 16, 64), 0, "rb/tiny/x")
    p = synth.resblock_params(64, 0, "rb/tiny")
    out, c1, c2 = run_chunks(wan, to_dev(x), dev_params(p), 32, 3)
    ref, r1, r2 = oracle.resblock(x, p, 32, EPS)
    conv_close(bits(out), ref, "resblock")
    check_caches(c1, c2, r1, r2)
    assert wan.wan_device_status() == 0


def test_resblock_medium_with_history(wan):
    # Two chunks (3 + 2 frames) at C=256 with ragged pixel tiles, against the oracle run the same way.
    x = synth.normal_bf16((1, 5, 12, 20, 256), 0, "rb/med/x")
    p = synth.resblock_params(256, 0, "rb/med")
    out, c1, c2 = run_chunks(wan, to_dev(x), dev_params(p), 32, 3)
    r_a, r1, r2 = oracle.resblock(x[:, :3], p, 32, EPS)
    r_b, r1, r2 = oracle.resblock(x[:, 3:], p, 32, EPS, r1, r2)
    conv_close(bits(out), np.concatenate([r_a, r_b], 1), "resblock chunks")
    check_caches(c1, c2, r1, r2)


def test_resblock_c1024_small_with_history_matches_oracle(wan):
    # The widest stage's ResBlock (Cin = Cout = 1024: the norm applied in the conv's operand prologue
    # over 16 K blocks per tap) on small frames, two chunks (2 + 2 frames) carrying the caches.
    x = synth.normal_bf16((1, 4, 12, 20, 1024), 0, "rb/c1024s/x")
    p = synth.resblock_params(1024, 0, "rb/c1024s")
    out, c1, c2 = run_chunks(wan, to_dev(x), dev_params(p), 32, 2)
    r_a, r1, r2 = oracle.resblock(x[:, :2], p, 32, EPS)
    r_b, r1, r2 = oracle.resblock(x[:, 2:], p, 32, EPS, r1, r2)
    conv_close(bits(out), np.concatenate([r_a, r_b], 1), "resblock C=1024 chunks")
    check_caches(c1, c2, r1, r2)
    assert wan.wan_device_status() == 0


def test_resblock_chunked_equals_unchunked_small(wan):
    x = to_dev(synth.normal_bf16((1, 12, 24, 40, 256), 0, "rb/chunk/x"))
    params = dev_params(synth.resblock_params(256, 0, "rb/chunk"))
    full, f1, f2 = run_chunks(wan, x, params, 32, 12)
    part, p1, p2 = run_chunks(wan, x, params, 32, 4)
    assert torch.equal(full.view(torch.int16), part.view(torch.int16))
    assert torch.equal(f1.view(torch.int16), p1.view(torch.int16))
    assert torch.equal(f2.view(torch.int16), p2.view(torch.int16))


def test_decoder_stage_c256_chunked_equals_unchunked(wan):
    # Three ResBlocks on [1, 12, 176, 312, 256]: 3 chunks of 4 frames vs one 12-frame pass.
    x = synth.normal_torch((1, 12, 176, 312, 256), 0, "stage4/x", device="cuda", dtype=torch.bfloat16)
    blocks = [dev_params(synth.resblock_params(256, 0, f"stage4/block{i}")) for i in range(3)]
    N, T, H, W, C = x.shape

    def stage(chunk):
        caches = [(torch.zeros((1, 2, H, W, C), dtype=torch.bfloat16, device="cuda"),
                   torch.zeros((1, 2, H, W, C), dtype=torch.bfloat16, device="cuda")) for _ in range(3)]
        outs = []
        for i, s in enumerate(range(0, T, chunk)):
            h = x[:, s:s + chunk].contiguous()
            for blk, (c1, c2) in zip(blocks, caches):
                h = wan.wan_resblock(h, blk, c1, c2, i > 0, 32, EPS)
            outs.append(h)
        torch.cuda.synchronize()
        return torch.cat(outs, 1)
    a = stage(12)
    b = stage(4)
    assert torch.isfinite(a.float()).all()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert wan.wan_device_status() == 0


def test_resblock_c1024_chunked_equals_unchunked(wan):
    # The widest stage's ResBlock on [1, 4, 44, 78, 1024] (GroupNorm + SiLU in the convs' operand
    # prologue): one 4-frame call, whose convs split their last round into 128-channel halves,
    # against two 2-frame chunks, whose convs do not.
    x = synth.normal_torch((1, 4, 44, 78, 1024), 0, "rb/c1024/x", device="cuda", dtype=torch.bfloat16)
    params = dev_params(synth.resblock_params(1024, 0, "rb/c1024"))
    full, f1, f2 = run_chunks(wan, x, params, 32, 4)
    part, p1, p2 = run_chunks(wan, x, params, 32, 2)
    assert torch.isfinite(full.float()).all()
    assert torch.equal(full.view(torch.int16), part.view(torch.int16))
    assert torch.equal(f1.view(torch.int16), p1.view(torch.int16))
    assert torch.equal(f2.view(torch.int16), p2.view(torch.int16))
    assert wan.wan_device_status() == 0
