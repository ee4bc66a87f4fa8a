"""Pins of the oracle's fp64 -> bf16 rounding (one rounding, nearest, ties to even)."""
import numpy as np
import pytest
import torch

from oracle import round_to_bf16, bf16_to_f64, ulp_distance_bf16


def bits(x):
    return int(round_to_bf16(np.array([x], dtype=np.float64))[0])


@pytest.mark.parametrize("value,expected", [
    (1.0, 0x3F80),
    (-2.0, 0xC000),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (1.0 + 2.0 ** -8, 0x3F80),                    # tie between 1 and 1+2^-7: to even (1)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),                # tie between 0x3F81 and 0x3F82: to even
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),       # just above the tie: up. Through fp32 the
                                                  # 2^-30 is lost first and the tie goes down.
    (1.0 + 2.0 ** -8 - 2.0 ** -30, 0x3F80),
    (3.0 * 2.0 ** 127, 0x7F80),                   # beyond the largest finite bf16 -> inf
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),       # largest finite bf16
    ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),       # tie with 2^128 rounds to even = overflow
    (2.0 ** -133, 0x0001),                        # smallest subnormal
    (2.0 ** -134, 0x0000),                        # half of it: tie, to even (zero)
    (1.5 * 2.0 ** -134, 0x0001),
    (3 * 2.0 ** -134, 0x0002),                    # tie between 1 and 2 subnormal steps: even
    (2.0 ** -126, 0x0080),                        # smallest normal
    (float("inf"), 0x7F80),
    (-float("inf"), 0xFF80),
])
def test_hand_cases(value, expected):
    assert bits(value) == expected


def test_nan():
    assert bits(float("nan")) == 0x7FC0


def test_agrees_with_torch_on_fp32_inputs():
    # For a value that is exactly an fp32, one rounding from fp64 equals torch's fp32 -> bf16
    # conversion (a library routine with round-to-nearest-even).
    rng = np.random.default_rng(1)
    raw = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f32 = raw.view(np.float32)
    f32 = f32[np.isfinite(f32)]
    ours = round_to_bf16(f32.astype(np.float64))
    theirs = torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_roundtrip_exact_values():
    all_bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bf16_to_f64(all_bits)
    finite = np.isfinite(vals)
    back = round_to_bf16(vals[finite])
    assert np.array_equal(back, all_bits[finite])


def test_ulp_distance():
    one = np.array([0x3F80], np.uint16)
    assert ulp_distance_bf16(one, np.array([0x3F81], np.uint16))[0] == 1
    assert ulp_distance_bf16(np.array([0x0000], np.uint16), np.array([0x8000], np.uint16))[0] == 0
    # smallest positive and smallest negative subnormal are two steps apart (through zero)
    assert ulp_distance_bf16(np.array([0x0001], np.uint16), np.array([0x8001], np.uint16))[0] == 2
