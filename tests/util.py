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


def cache2_close(got_bits, ref, what=""):
    """The second conv's cache of a ResBlock holds silu(gn(h)) of the first conv's output h: h's
    conv error (up to one bf16 step at its largest magnitude), carried through the normalisation,
    then the norm's own rounding: relative L2 <= 4e-3 and max |err| <= 2 * 2^-7 max |ref|."""
    got = oracle.bf16_to_f64(got_bits)
    ref = oracle.bf16_to_f64(ref) if ref.dtype == np.uint16 else np.asarray(ref, np.float64)
    diff = got - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.max(np.abs(diff))) if diff.size else 0.0
    assert rel <= REL_L2_MAX, f"{what}: relative L2 {rel:.3e} > {REL_L2_MAX}"
    assert mx <= 2 * MAX_ABS_FRAC * float(np.max(np.abs(ref))), f"{what}: max abs err {mx:.3e}"
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


class ConvErr:
    """The conv acceptance criterion over an output compared piece by piece (for outputs whose
    oracle is computed in bands): relative L2 over the whole output and max |err| against
    2^-7 * max |ref| over the whole output."""

    def __init__(self, what="", max_abs_frac=MAX_ABS_FRAC):
        self.what = what
        self.max_abs_frac = max_abs_frac
        self.err2 = 0.0
        self.ref2 = 0.0
        self.maxerr = 0.0
        self.maxref = 0.0
        self.count = 0

    def add(self, got_bits, ref):
        got = oracle.bf16_to_f64(got_bits)
        ref = oracle.bf16_to_f64(ref) if ref.dtype == np.uint16 else np.asarray(ref, np.float64)
        assert got.shape == ref.shape, f"{self.what}: shapes {got.shape} vs {ref.shape}"
        assert np.all(np.isfinite(got)), f"{self.what}: non-finite output"
        diff = got - ref
        self.err2 += float(np.sum(diff * diff))
        self.ref2 += float(np.sum(ref * ref))
        if diff.size:
            self.maxerr = max(self.maxerr, float(np.max(np.abs(diff))))
            self.maxref = max(self.maxref, float(np.max(np.abs(ref))))
        self.count += got.size

    def rel_and_max(self):
        return float(np.sqrt(self.err2) / max(np.sqrt(self.ref2), 1e-300)), self.maxerr

    def check(self):
        rel = float(np.sqrt(self.err2) / max(np.sqrt(self.ref2), 1e-300))
        bound = self.max_abs_frac * self.maxref
        assert rel <= REL_L2_MAX, f"{self.what}: relative L2 {rel:.3e} > {REL_L2_MAX}"
        assert self.maxerr <= bound, f"{self.what}: max abs err {self.maxerr:.3e} > {bound:.3e}"
        return rel, self.maxerr


def ulp_report(got_bits, ref_bits):
    """Counts of elements by bf16 ulp distance (0, 1, 2, 3, more) and where the largest is."""
    d = oracle.ulp_distance_bf16(got_bits, ref_bits)
    counts = {k: int(np.count_nonzero(d == k)) for k in range(4)}
    counts[">3"] = int(np.count_nonzero(d > 3))
    i = int(np.argmax(d))
    return {"counts": counts, "max_ulp": int(d.flat[i]), "at": tuple(int(v) for v in np.unravel_index(i, d.shape)),
            "got": float(oracle.bf16_to_f64(np.asarray(got_bits).flat[i])),
            "ref": float(oracle.bf16_to_f64(np.asarray(ref_bits).flat[i]))}
