"""Phase-weight transform and nearest-x2 + 3x3 upsample on the GPU against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from util import to_dev, bits, conv_close
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu


def test_phase_weights_bit_exact(wan):
    w3 = synth.normal_bf16((512, 3, 3, 512), 0, "up/cfg3/w3", 0.0, float(np.sqrt(1.0 / (9 * 512))))
    wp = bits(wan.wan_upsample_phase_weights(to_dev(w3)))
    assert np.array_equal(wp, oracle.phase_weights(w3))


@pytest.mark.parametrize("shape,Cout,bias", [
    ((1, 1, 6, 10, 64), 64, False),
    ((1, 3, 9, 13, 128), 96, True),     # ragged tiles, odd sizes
    ((2, 2, 5, 7, 64), 320, True),
    ((1, 2, 19, 40, 64), 256, True),    # CTA-pair path: ragged 8 x 16 tiles, 3 tiles wide
    ((1, 1, 9, 17, 128), 512, False),   # CTA-pair path: two N blocks
    ((1, 2, 1, 1, 64), 256, True),      # a 1 x 1 input: a 2 x 2 output, each phase one tap inside
    ((1, 1, 1, 7, 64), 256, False),     # a one-row input
])
def test_upsample_small(wan, shape, Cout, bias):
    Cin = shape[-1]
    x = synth.normal_bf16(shape, 0, f"up/{shape}/x")
    w3 = synth.normal_bf16((Cout, 3, 3, Cin), 0, f"up/{shape}/w3", 0.0, float(np.sqrt(1.0 / (9 * Cin))))
    b = synth.normal_bf16((Cout,), 0, f"up/{shape}/b", 0.0, 0.01) if bias else None
    wp = wan.wan_upsample_phase_weights(to_dev(w3))
    y = wan.wan_upsample_phase_conv(to_dev(x), wp, None if b is None else to_dev(b))
    torch.cuda.synchronize()
    got = bits(y)
    bf = None if b is None else oracle.bf16_to_f64(b)
    ref = oracle.upsample_nearest_conv_f64(oracle.bf16_to_f64(x), oracle.bf16_to_f64(w3), bf)
    conv_close(got, ref, "upsample (definition)")
    # against the same bf16 phase weights (isolates the kernel from the transform's rounding)
    ref_p = oracle.phase_conv_f64(oracle.bf16_to_f64(x), oracle.bf16_to_f64(bits(wp)), bf)
    conv_close(got, ref_p, "upsample (phase form)")
    assert wan.wan_device_status() == 0


def test_upsample_full_size(wan):
    # [1, 4, 44, 78, 512] -> [1, 4, 88, 156, 512], weights N(0, 1/(9*512)), against the definition.
    x = synth.normal_bf16((1, 4, 44, 78, 512), 0, "up/cfg3/x")
    w3 = synth.normal_bf16((512, 3, 3, 512), 0, "up/cfg3/w3", 0.0, float(np.sqrt(1.0 / (9 * 512))))
    wp = wan.wan_upsample_phase_weights(to_dev(w3))
    y = wan.wan_upsample_phase_conv(to_dev(x), wp)
    torch.cuda.synchronize()
    ref = oracle.upsample_nearest_conv_f64(oracle.bf16_to_f64(x), oracle.bf16_to_f64(w3))
    conv_close(bits(y), ref, "upsample cfg3")
