"""Helpers shared by the tests: bf16 bit moves between numpy and torch, tolerance checks."""
import numpy as np

import oracle

REL_L2_MAX = 4e-3          # conv / upsample / ResBlock acceptance: relative L2 error
MAX_ABS_FRAC = 2.0 ** -7   # and max |err| <= 2^-7 * max |ref|


def to_dev(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).to(device)


def f32_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def bits(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def conv_close(got_bits, ref, what=""):
    """ref: fp64 array (or bf16 bits). Asserts the conv acceptance criterion; returns (rel, maxabs)."""
    got = oracle.bf16_to_f64(got_bits)
    ref = oracle.bf16_to_f64(ref) if ref.dtype == np.uint16 else np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = got - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.max(np.abs(diff))) if diff.size else 0.0
    bound = MAX_ABS_FRAC * float(np.max(np.abs(ref))) if ref.size else 0.0
    assert rel <= REL_L2_MAX, f"{what}: relative L2 {rel:.3e} > {REL_L2_MAX}"
    assert mx <= bound, f"{what}: max abs err {mx:.3e} > {bound:.3e}"
    return rel, mx


def padded(a_bits, cache_bits=None):
    """fp64 padded input P = [cache or zeros; a], zero-padded by 1 in H and W: [N, T+2, H+2, W+2, C]."""
    a = oracle.bf16_to_f64(a_bits)
    N, T, H, W, C = a.shape
    c = np.zeros((N, 2, H, W, C)) if cache_bits is None else oracle.bf16_to_f64(cache_bits)
    return np.pad(np.concatenate([c, a], 1), ((0, 0), (0, 0), (1, 1), (1, 1), (0, 0)))


def sample_points(rng, N, T, H, W, count):
    """Output points (n, t, h, w): the frame corners and edges plus uniform random ones."""
    pts = set()
    for n in {0, N - 1}:
        for t in {0, T - 1}:
            for h in {0, H - 1}:
                for w in {0, W - 1}:
                    pts.add((n, t, h, w))
    while len(pts) < count:
        pts.add((int(rng.integers(N)), int(rng.integers(T)), int(rng.integers(H)), int(rng.integers(W))))
    return sorted(pts)
