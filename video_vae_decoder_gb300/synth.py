"""Seeded synthetic inputs, shared by the CUDA path's tests and benchmark and by the oracle's tests.

This module holds no arithmetic of the method itself (no normalisation, no convolution, no
rounding rule of the decoder): it only draws numbers and stores them as fp32 or bf16 bits.

Generator (counter-based, so any element can be drawn on its own):
  * SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
    OOPSLA 2014): state_i = key + (i + 1) * 0x9E3779B97F4A7C15 (mod 2^64), output mix64(state_i)
    with the published finaliser (xor-shift 30, multiply 0xBF58476D1CE4E5B9, xor-shift 27,
    multiply 0x94D049BB133111EB, xor-shift 31).
  * key = mix64(seed xor FNV-1a-64(name)), one stream per named tensor.
  * uniform u_i = ((out_i >> 11) + 1) * 2^-53, in (0, 1].
  * Box-Muller (1958): normal element i takes the pair j = i // 2,
    r = sqrt(-2 ln u_{2j}), theta = 2 pi u_{2j+1}; even i -> r cos(theta), odd i -> r sin(theta).
  * value = mean + std * normal, in fp64, then rounded to fp32 (IEEE round to nearest even);
    a bf16 tensor is the fp32 value rounded to nearest even on its upper 16 bits.

`normal_torch` is the same generator written with torch int64 arithmetic so that tensors too
large for numpy can be drawn on the device; `test_synth.py` checks it against the numpy form.
"""
from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1


def fnv1a64(name: str) -> int:
    """FNV-1a 64-bit hash (Fowler, Noll, Vo) of the UTF-8 bytes of `name`."""
    h = 0xCBF29CE484222325
    for byte in name.encode("utf-8"):
        h ^= byte
        h = (h * 0x100000001B3) & MASK64
    return h


def _mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, name: str) -> int:
    return _mix64_int((seed & MASK64) ^ fnv1a64(name))


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= np.uint64(MIX1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(MIX2)
    z ^= z >> np.uint64(31)
    return z


def splitmix64_np(key: int, index: np.ndarray) -> np.ndarray:
    """Raw SplitMix64 outputs (uint64) at the given counter indices of the stream `key`."""
    state = np.uint64(key) + (np.asarray(index).astype(np.uint64) + np.uint64(1)) * np.uint64(GAMMA)
    return _mix64_np(state)


def uniform_np(key: int, index: np.ndarray) -> np.ndarray:
    """Uniforms in (0, 1] at the given counter indices (uint64 array)."""
    out = splitmix64_np(key, index)
    return ((out >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def standard_normal_at(seed: int, name: str, index: np.ndarray) -> np.ndarray:
    """Standard normals (fp64) at arbitrary flat element indices of the named stream."""
    index = np.asarray(index, dtype=np.uint64)
    key = stream_key(seed, name)
    pair = index >> np.uint64(1)
    u1 = uniform_np(key, pair * np.uint64(2))
    u2 = uniform_np(key, pair * np.uint64(2) + np.uint64(1))
    r = np.sqrt(-2.0 * np.log(u1))
    theta = 2.0 * np.pi * u2
    odd = (index & np.uint64(1)).astype(bool)
    return np.where(odd, r * np.sin(theta), r * np.cos(theta))


def normal_f32(shape, seed: int, name: str, mean: float = 0.0, std: float = 1.0,
               chunk: int = 1 << 22) -> np.ndarray:
    """fp32 array of `shape`, element i = fp32(mean + std * normal_i)."""
    count = int(np.prod(shape))
    out = np.empty(count, dtype=np.float32)
    for start in range(0, count, chunk):
        stop = min(count, start + chunk)
        idx = np.arange(start, stop, dtype=np.uint64)
        out[start:stop] = (mean + std * standard_normal_at(seed, name, idx)).astype(np.float32)
    return out.reshape(shape)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return the 16-bit patterns as uint16."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (bits + np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    rounded = np.where(nan, np.uint64(0x7FC0), rounded)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(shape, seed: int, name: str, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of `shape` drawn as fp32(mean + std * normal), rounded to bf16."""
    return f32_to_bf16_bits(normal_f32(shape, seed, name, mean, std))


# ----------------------------------------------------------------------------------------------
# torch form of the same generator (device-side drawing of large tensors)
# ----------------------------------------------------------------------------------------------

def _signed(c: int) -> int:
    return c - (1 << 64) if c >= (1 << 63) else c


def _lsr(t, k: int):
    """Logical right shift of an int64 tensor holding uint64 bit patterns."""
    return (t >> k) & ((1 << (64 - k)) - 1)


def _mix64_torch(z):
    z = z ^ _lsr(z, 30)
    z = z * _signed(MIX1)
    z = z ^ _lsr(z, 27)
    z = z * _signed(MIX2)
    return z ^ _lsr(z, 31)


def normal_torch(shape, seed: int, name: str, mean: float = 0.0, std: float = 1.0,
                 device="cpu", dtype=None, chunk: int = 1 << 26):
    """The generator above in torch int64 arithmetic; returns fp32 (or `dtype`, converted from the
    fp32 values with torch's round-to-nearest-even) on `device`."""
    import torch
    count = 1
    for s in shape:
        count *= int(s)
    out = torch.empty(count, dtype=dtype or torch.float32, device=device)
    key = _signed(stream_key(seed, name))
    for start in range(0, count, chunk):
        stop = min(count, start + chunk)
        idx = torch.arange(start, stop, dtype=torch.int64, device=device)
        pair = idx >> 1

        def uni(counter):
            state = key + (counter + 1) * _signed(GAMMA)
            o = _mix64_torch(state)
            return (_lsr(o, 11).to(torch.float64) + 1.0) * (2.0 ** -53)

        u1 = uni(pair * 2)
        u2 = uni(pair * 2 + 1)
        r = torch.sqrt(-2.0 * torch.log(u1))
        theta = 2.0 * np.pi * u2
        n = torch.where((idx & 1).bool(), r * torch.sin(theta), r * torch.cos(theta))
        out[start:stop] = (mean + std * n).to(torch.float32).to(out.dtype)
        del idx, pair, u1, u2, r, theta, n
    return out.reshape(tuple(int(s) for s in shape))


# ----------------------------------------------------------------------------------------------
# Named workloads (distributions and shapes of the decoder problems this library targets)
# ----------------------------------------------------------------------------------------------

def resblock_params(C: int, seed: int, prefix: str) -> dict:
    """Parameters of one causal ResBlock at C channels, drawn as:
    gamma = 1 + 0.1 N(0,1) and beta = 0.1 N(0,1) (fp32, per channel);
    conv weights [C, 3, 3, 3, C] ~ N(0, 1/(27 C)) (variance 1/(27 C)), bias 0.01 N(0,1) (bf16)."""
    wstd = float(np.sqrt(1.0 / (27.0 * C)))
    p = {}
    for k in (1, 2):
        p[f"gamma{k}"] = normal_f32((C,), seed, f"{prefix}/gamma{k}", 1.0, 0.1)
        p[f"beta{k}"] = normal_f32((C,), seed, f"{prefix}/beta{k}", 0.0, 0.1)
        p[f"w{k}"] = normal_bf16((C, 3, 3, 3, C), seed, f"{prefix}/w{k}", 0.0, wstd)
        p[f"b{k}"] = normal_bf16((C,), seed, f"{prefix}/b{k}", 0.0, 0.01)
    return p
