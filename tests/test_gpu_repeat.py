"""Repeated GPU runs give the same bits: every output's reduction runs in a fixed order, whatever
CTA pair computes it and however the items are scheduled (whole items or 128-channel halves)."""
import numpy as np
import pytest
import torch

from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))


def n(shape, name, std=1.0):
    return synth.normal_torch(shape, 0, name, 0.0, std, device="cuda", dtype=torch.bfloat16)


def same(f):
    a = f().clone()
    b = f().clone()
    torch.cuda.synchronize()
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_repeat_resblock_c256_chunk(wan):
    C = 256
    x = n((1, 4, 176, 312, C), "rep/x")
    p = {k: (torch.from_numpy(v).cuda() if v.dtype == np.float32 else
             torch.from_numpy(v.view(np.int16).copy()).view(torch.bfloat16).cuda())
         for k, v in synth.resblock_params(C, 0, "rep/block").items()}
    c = n((1, 2, 176, 312, C), "rep/c")

    def run():
        c1, c2 = c.clone(), c.clone()
        return wan.wan_resblock(x, p, c1, c2, True, 32, EPS)
    assert same(run)
    assert wan.wan_device_status() == 0


def test_repeat_resblock_winograd_c1024(wan):
    # The widest stage's block through Winograd, its second norm from conv 1's statistics.
    C = 1024
    x = n((1, 4, 44, 78, C), "rep/w/x")
    p = {k: (torch.from_numpy(v).cuda() if v.dtype == np.float32 else
             torch.from_numpy(v.view(np.int16).copy()).view(torch.bfloat16).cuda())
         for k, v in synth.resblock_params(C, 0, "rep/w/block").items()}
    u1, u2 = wan.wan_winograd_weights(p["w1"]), wan.wan_winograd_weights(p["w2"])
    c = n((1, 2, 44, 78, C), "rep/w/c")

    def run():
        c1, c2 = c.clone(), c.clone()
        return wan.wan_resblock_winograd(x, p, u1, u2, c1, c2, True, 32, EPS)
    assert same(run)
    assert wan.wan_device_status() == 0


def test_repeat_conv_c1024_split(wan):
    C = 1024
    x = n((1, 4, 44, 78, C), "rep/x5")
    w = n((C, 3, 3, 3, C), "rep/w5", (1.0 / (27 * C)) ** 0.5)
    b = n((C,), "rep/b5", 0.01)
    cache = n((1, 2, 44, 78, C), "rep/c5")
    assert same(lambda: wan.wan_causal_conv3d(x, w, b, None, cache))
    assert wan.wan_device_status() == 0


def test_repeat_head_and_upsample(wan):
    xh = n((1, 8, 96, 320, 256), "rep/xh")
    wh = n((12, 3, 3, 3, 256), "rep/wh", (1.0 / (27 * 256)) ** 0.5)
    assert same(lambda: wan.wan_causal_conv3d(xh, wh))
    xu = n((1, 4, 44, 78, 512), "rep/xu")
    wp = wan.wan_upsample_phase_weights(n((512, 3, 3, 512), "rep/w3", (1.0 / (9 * 512)) ** 0.5))
    assert same(lambda: wan.wan_upsample_phase_conv(xu, wp))
    assert wan.wan_device_status() == 0
