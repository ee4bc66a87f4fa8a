"""Failure detection of the bounded device waits: a wait made to run out on purpose (a short bound
and a wait nothing can complete) ends the kernel with WAN_ERR_TIMEOUT in the device error word, and
the next calls run normally. Nothing faults and nothing waits without bound."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, f32_dev, bits
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
EPS = float(np.float32(1e-6))
WAN_ERR_TIMEOUT = 6
SHORT = 1_000_000  # SM cycles (about 0.5 ms)


def _gn_case():
    xb = synth.normal_bf16((1, 2, 12, 20, 128), 0, "timeout/x", 0.5, 1.0)
    g = synth.normal_f32((128,), 0, "timeout/g", 1.0, 0.1)
    b = synth.normal_f32((128,), 0, "timeout/b", 0.0, 0.1)
    return xb, g, b


def test_mbarrier_wait_times_out_and_reports(wan):
    assert wan.wan_device_status() == 0
    assert wan.wan_selftest_wait_timeout(1, SHORT) == 0
    assert wan.wan_device_status() == WAN_ERR_TIMEOUT
    assert wan.wan_device_status() == 0  # read and cleared


def test_grid_barrier_times_out_then_the_norm_runs_normally(wan):
    xb, g, b = _gn_case()
    x, gd, bd = to_dev(xb), f32_dev(g), f32_dev(b)
    y = torch.full_like(x, 7.0)
    assert wan.wan_device_status() == 0
    assert wan.wan_selftest_wait_timeout(0, SHORT, x, gd, bd, 32, EPS, y) == 0
    assert wan.wan_device_status() == WAN_ERR_TIMEOUT
    # every CTA gave up at the first barrier, before the apply pass: y is untouched
    assert bool((y == 7.0).all())
    # the context is usable and the same kernel, called normally, is correct
    y2 = wan.wan_gn_silu(x, gd, bd, 32, EPS)
    assert wan.wan_device_status() == 0
    ulp = oracle.ulp_distance_bf16(bits(y2), oracle.gn_silu(xb, g, b, 32, EPS))
    assert int(ulp.max()) <= 1
