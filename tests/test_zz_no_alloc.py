"""wan_gn_silu_noalloc: GroupNorm + SiLU for callers that cannot allocate device memory (hosts that
give a library no allocator and no workspace, such as an application that keeps all device memory
in its own pool, or a loop that may not call cudaMalloc). It must give exactly what wan_gn_silu
gives, call after call, while its scratch is the library's fixed device array shared by every call.

This file is collected last on purpose: it runs after every other test in a full run, and also
passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from util import to_dev, f32_dev, bits
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))
WAN_ERR_WORKSPACE = 4


def _inputs(shape, name, mean, std):
    C = shape[-1]
    xb = synth.normal_bf16(shape, 0, f"{name}/x", mean, std)
    g = synth.normal_f32((C,), 0, f"{name}/g", 1.0, 0.1)
    b = synth.normal_f32((C,), 0, f"{name}/b", 0.0, 0.1)
    return xb, g, b


def _call_c_abi(x, g, b, groups, y):
    """Straight through the C ABI with raw device pointers (the call takes no workspace)."""
    from video_vae_decoder_gb300 import binding
    L = binding.lib()
    N, T, H, W, C = x.shape
    return L.wan_gn_silu_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                                 ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                                 N, T, H, W, C, groups, ctypes.c_float(EPS),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_two_calls_in_a_row(wan):
    # Two different problems back to back: the second call reuses the scratch the first left
    # (other partial counts, another barrier count), so stale scratch would show as a difference.
    cases = [((1, 4, 88, 156, 512), 32, "noalloc/a", 0.5, float(np.sqrt(2.0))),
             ((1, 3, 20, 36, 256), 32, "noalloc/b", 1e3, 1.0)]
    host, outs = [], []
    for shape, groups, name, mean, std in cases:
        xb, g, b = _inputs(shape, name, mean, std)
        x, gd, bd = to_dev(xb), f32_dev(g), f32_dev(b)
        y = torch.full_like(x, float("nan"))
        assert _call_c_abi(x, gd, bd, groups, y) == 0
        host.append((xb, g, b, groups))
        outs.append((x, gd, bd, groups, y))
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    for (xb, g, b, groups), (x, gd, bd, _, y) in zip(host, outs):
        ref = wan.wan_gn_silu(x, gd, bd, groups, EPS)
        torch.cuda.synchronize()
        # the same kernels with the same plan: the same bits as the call with a workspace ...
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        # ... and within one bf16 ulp of the fp64 oracle, rounded once
        ulp = oracle.ulp_distance_bf16(bits(y), oracle.gn_silu(xb, g, b, groups, EPS))
        assert int(ulp.max()) <= 1


def test_noalloc_refuses_a_size_beyond_its_scratch_and_writes_nothing(wan):
    # [1, 500, 4, 4, 512] with 32 groups needs 4.15 MiB of scratch, more than the 4 MiB array:
    # refused on the host with WAN_ERR_WORKSPACE, and y keeps its contents.
    shape = (1, 500, 4, 4, 512)
    assert wan.wan_workspace_size(wan.WAN_OP_GN_SILU, *shape, 0, 32) > 4 << 20
    xb, g, b = _inputs(shape, "noalloc/big", 0.0, 1.0)
    x, gd, bd = to_dev(xb), f32_dev(g), f32_dev(b)
    y = torch.full_like(x, 3.0)
    assert _call_c_abi(x, gd, bd, 32, y) == WAN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())
    assert wan.wan_device_status() == 0
