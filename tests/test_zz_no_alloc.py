"""wan_gn_silu_noalloc: GroupNorm + SiLU for callers that cannot allocate device memory (hosts that
give a library no allocator and no workspace). It must give what wan_gn_silu gives, call after
call, while its scratch is the library's fixed device array shared by every call.

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


def _inputs(shape, name, mean, std):
    C = shape[-1]
    x = to_dev(synth.normal_bf16(shape, 0, f"{name}/x", mean, std))
    g = f32_dev(synth.normal_f32((C,), 0, f"{name}/g", 1.0, 0.1))
    b = f32_dev(synth.normal_f32((C,), 0, f"{name}/b", 0.0, 0.1))
    return x, g, b


def _call_c_abi(x, g, b, groups, y):
    """Straight through the C ABI with raw device pointers (no workspace argument exists)."""
    from video_vae_decoder_gb300 import binding
    L = binding.lib()
    N, T, H, W, C = x.shape
    return L.wan_gn_silu_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                                 ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(b.data_ptr()),
                                 N, T, H, W, C, groups, ctypes.c_float(EPS),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_two_calls_in_a_row(wan):
    # Two different problems back to back: the second call reuses the scratch the first left.
    cases = [((1, 4, 88, 156, 512), 32, "noalloc/a", 0.5, float(np.sqrt(2.0))),
             ((1, 3, 20, 36, 256), 32, "noalloc/b", 1e3, 1.0)]
    outs = []
    for shape, groups, name, mean, std in cases:
        x, g, b = _inputs(shape, name, mean, std)
        y = torch.empty_like(x)
        assert _call_c_abi(x, g, b, groups, y) == 0
        outs.append((x, g, b, groups, y))
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0
    for x, g, b, groups, y in outs:
        ref = wan.wan_gn_silu(x, g, b, groups, EPS)
        torch.cuda.synchronize()
        ulp = oracle.ulp_distance_bf16(bits(y), bits(ref))
        assert int(ulp.max()) <= 1
