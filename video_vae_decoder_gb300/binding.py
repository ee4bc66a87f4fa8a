"""Python binding of the C ABI in include/wan.h (ctypes; argument marshalling only).

Every function here has the name of the C entry point it calls. Device memory comes from torch
(tensors must be CUDA, contiguous, bf16 where the ABI says bf16, fp32 for GroupNorm's gamma and
beta); work is enqueued on torch's current CUDA stream. The shared library is the in-tree build
`lib/libwan.so`; if it is missing, loading raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libwan.so")

WAN_OP_GN_SILU = 0
WAN_OP_CAUSAL_CONV3D = 1
WAN_OP_RESBLOCK = 2
WAN_OP_UPSAMPLE_PHASE_CONV = 3
WAN_OP_GN_STATS = 4
WAN_OP_GN_SILU_CONV3D = 5
WAN_OP_RESBLOCK_SHORTCUT = 6
WAN_OP_WINOGRAD_CONV3D = 7
WAN_OP_RESBLOCK_WINOGRAD = 8
WAN_OP_GN_STATS_WINOGRAD = 9

STATUS = {0: "WAN_OK", 1: "WAN_ERR_INVALID_ARG", 2: "WAN_ERR_UNSUPPORTED_SHAPE", 3: "WAN_ERR_MISALIGNED",
          4: "WAN_ERR_WORKSPACE", 5: "WAN_ERR_CUDA", 6: "WAN_ERR_TIMEOUT"}

EXPORTS = ("wan_status_string", "wan_workspace_size", "wan_gn_silu", "wan_gn_silu_clip", "wan_gn_silu_noalloc",
           "wan_causal_conv3d",
           "wan_causal_conv3d_gn_stats", "wan_gn_silu_from_stats", "wan_gn_silu_causal_conv3d", "wan_gn_silu_coefficients",
           "wan_causal_conv3d_gn_input", "wan_gn_silu_cache_update", "wan_cache_update",
           "wan_causal_conv3d_gn_input_stats", "wan_gn_silu_coefficients_from_stats",
           "wan_time_upsample", "wan_conv1x1", "wan_fold_bias", "wan_resblock_shortcut",
           "wan_upsample_phase_weights", "wan_upsample_phase_conv", "wan_resblock", "wan_winograd_weights",
           "wan_causal_conv3d_winograd", "wan_causal_conv3d_winograd_stats", "wan_resblock_winograd",
           "wan_selftest_wait_timeout",
           "wan_device_status")


class WanError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class ResblockParams(ctypes.Structure):
    _fields_ = [("gamma1", ctypes.c_void_p), ("beta1", ctypes.c_void_p), ("w1", ctypes.c_void_p),
                ("b1", ctypes.c_void_p), ("gamma2", ctypes.c_void_p), ("beta2", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("b2", ctypes.c_void_p), ("groups", ctypes.c_int),
                ("eps", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library with argument types declared. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(there is no fallback implementation)")
    L = ctypes.CDLL(LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.wan_status_string.restype = ctypes.c_char_p
    L.wan_status_string.argtypes = [I]
    L.wan_workspace_size.restype = S
    L.wan_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
    L.wan_gn_silu.restype = I
    L.wan_gn_silu.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, S, P]
    L.wan_gn_silu_clip.restype = I
    L.wan_gn_silu_clip.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, S, P]
    L.wan_gn_silu_noalloc.restype = I
    L.wan_gn_silu_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P]
    L.wan_causal_conv3d.restype = I
    L.wan_causal_conv3d.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P, S, P]
    L.wan_causal_conv3d_gn_stats.restype = I
    L.wan_causal_conv3d_gn_stats.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, S, P]
    L.wan_gn_silu_from_stats.restype = I
    L.wan_gn_silu_from_stats.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, S, P, S, P]
    L.wan_gn_silu_causal_conv3d.restype = I
    L.wan_gn_silu_causal_conv3d.argtypes = [P, P, P, I, F, P, P, P, P, P, P, I, I, I, I, I, I, P, S, P]
    L.wan_gn_silu_coefficients.restype = I
    L.wan_gn_silu_coefficients.argtypes = [P, P, P, I, I, I, I, I, I, F, P, P, S, P]
    L.wan_causal_conv3d_gn_input.restype = I
    L.wan_causal_conv3d_gn_input.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, P]
    L.wan_gn_silu_cache_update.restype = I
    L.wan_gn_silu_cache_update.argtypes = [P, P, P, P, I, I, I, I, I, P]
    L.wan_causal_conv3d_gn_input_stats.restype = I
    L.wan_causal_conv3d_gn_input_stats.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, S, P]
    L.wan_gn_silu_coefficients_from_stats.restype = I
    L.wan_gn_silu_coefficients_from_stats.argtypes = [P, S, P, P, I, I, I, I, I, I, F, P, P]
    L.wan_time_upsample.restype = I
    L.wan_time_upsample.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P]
    L.wan_conv1x1.restype = I
    L.wan_conv1x1.argtypes = [P, P, P, I, I, I, I, I, I, P]
    L.wan_fold_bias.restype = I
    L.wan_fold_bias.argtypes = [P, P, P, I, P]
    L.wan_resblock_shortcut.restype = I
    L.wan_resblock_shortcut.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, P, S, P]
    L.wan_cache_update.restype = I
    L.wan_cache_update.argtypes = [P, P, P, I, I, I, I, I, P]
    L.wan_upsample_phase_weights.restype = I
    L.wan_upsample_phase_weights.argtypes = [P, P, I, I, P]
    L.wan_upsample_phase_conv.restype = I
    L.wan_upsample_phase_conv.argtypes = [P, P, P, P, I, I, I, I, I, I, P]
    L.wan_resblock.restype = I
    L.wan_resblock.argtypes = [P, P, ctypes.POINTER(ResblockParams), P, P, I, I, I, I, I, I, P, S, P]
    L.wan_winograd_weights.restype = I
    L.wan_winograd_weights.argtypes = [P, P, I, I, P]
    L.wan_causal_conv3d_winograd.restype = I
    L.wan_causal_conv3d_winograd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, S, P]
    L.wan_causal_conv3d_winograd_stats.restype = I
    L.wan_causal_conv3d_winograd_stats.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, S, P, S, P]
    L.wan_resblock_winograd.restype = I
    L.wan_resblock_winograd.argtypes = [P, P, ctypes.POINTER(ResblockParams), P, P, P, P, I, I, I, I, I, I, P, S, P]
    L.wan_selftest_wait_timeout.restype = I
    L.wan_selftest_wait_timeout.argtypes = [I, ctypes.c_longlong, P, P, P, P, I, I, I, I, I, I, F, P, S, P]
    L.wan_device_status.restype = I
    L.wan_device_status.argtypes = [P]
    _lib = L
    return L


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check(status: int, where: str):
    if status != 0:
        raise WanError(status, where)


def _need(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor, got "
                         f"{t.device} {t.dtype} contiguous={t.is_contiguous()}")


def wan_status_string(status: int) -> str:
    return lib().wan_status_string(status).decode()


def wan_workspace_size(op: int, N: int, T: int, H: int, W: int, Cin: int, Cout: int = 0, groups: int = 0) -> int:
    return int(lib().wan_workspace_size(op, N, T, H, W, Cin, Cout, groups))


def _workspace(nbytes: int, device, ws=None):
    if nbytes == 0:
        return None
    if ws is not None and ws.numel() * ws.element_size() >= nbytes:
        return ws
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def wan_gn_silu(x, gamma, beta, groups: int, eps: float, y=None, ws=None, stream=None, whole_clip: bool = False):
    """y = silu(group_norm(x)) per (n, t, group), or per (n, group) over all frames with
    whole_clip; x [N, T, H, W, C] bf16."""
    _need(x, torch.bfloat16, "x")
    _need(gamma, torch.float32, "gamma")
    _need(beta, torch.float32, "beta")
    N, T, H, W, C = x.shape
    y = torch.empty_like(x) if y is None else y
    _need(y, torch.bfloat16, "y")
    need = wan_workspace_size(WAN_OP_GN_SILU, N, T, H, W, C, 0, groups)
    ws = _workspace(need, x.device, ws)
    fn = lib().wan_gn_silu_clip if whole_clip else lib().wan_gn_silu
    _check(fn(_ptr(x), _ptr(y), _ptr(gamma), _ptr(beta), N, T, H, W, C, groups, eps,
              _ptr(ws), need if ws is not None else 0, _stream(stream)),
           "wan_gn_silu_clip" if whole_clip else "wan_gn_silu")
    return y


def wan_gn_silu_noalloc(x, gamma, beta, groups: int, eps: float, y=None, stream=None):
    """wan_gn_silu without a workspace: the library's fixed device scratch is used instead (for
    callers that cannot allocate). Calls that overlap on the GPU race on that scratch."""
    _need(x, torch.bfloat16, "x")
    _need(gamma, torch.float32, "gamma")
    _need(beta, torch.float32, "beta")
    N, T, H, W, C = x.shape
    y = torch.empty_like(x) if y is None else y
    _need(y, torch.bfloat16, "y")
    _check(lib().wan_gn_silu_noalloc(_ptr(x), _ptr(y), _ptr(gamma), _ptr(beta), N, T, H, W, C, groups, eps,
                                     _stream(stream)), "wan_gn_silu_noalloc")
    return y


def wan_causal_conv3d(a, w, bias=None, residual=None, cache_in=None, cache_out=None, y=None, stream=None):
    """Causal 3x3x3 conv of a [N, T, H, W, Cin] with weights [Cout, 3, 3, 3, Cin] (bf16)."""
    for t, n in ((a, "a"), (w, "w"), (bias, "bias"), (residual, "residual"), (cache_in, "cache_in"),
                 (cache_out, "cache_out")):
        _need(t, torch.bfloat16, n)
    N, T, H, W, Cin = a.shape
    Cout = w.shape[0]
    y = torch.empty((N, T, H, W, Cout), dtype=torch.bfloat16, device=a.device) if y is None else y
    _need(y, torch.bfloat16, "y")
    _check(lib().wan_causal_conv3d(_ptr(a), _ptr(cache_in), _ptr(cache_out), _ptr(w), _ptr(bias), _ptr(residual),
                                   _ptr(y), N, T, H, W, Cin, Cout, None, 0, _stream(stream)), "wan_causal_conv3d")
    return y


def wan_causal_conv3d_gn_stats(a, w, groups: int, bias=None, residual=None, cache_in=None, cache_out=None, y=None,
                               stats=None, stream=None):
    """wan_causal_conv3d that also emits the GroupNorm statistics of y for wan_gn_silu_from_stats.
    Returns (y, stats); stats is a uint8 device buffer private to the library."""
    for t, n in ((a, "a"), (w, "w"), (bias, "bias"), (residual, "residual"), (cache_in, "cache_in"),
                 (cache_out, "cache_out")):
        _need(t, torch.bfloat16, n)
    N, T, H, W, Cin = a.shape
    Cout = w.shape[0]
    y = torch.empty((N, T, H, W, Cout), dtype=torch.bfloat16, device=a.device) if y is None else y
    _need(y, torch.bfloat16, "y")
    need = wan_workspace_size(WAN_OP_GN_STATS, N, T, H, W, Cin, Cout, groups)
    if need == 0:
        raise WanError(2, "wan_causal_conv3d_gn_stats")
    stats = _workspace(need, a.device, stats)
    _check(lib().wan_causal_conv3d_gn_stats(_ptr(a), _ptr(cache_in), _ptr(cache_out), _ptr(w), _ptr(bias),
                                            _ptr(residual), _ptr(y), N, T, H, W, Cin, Cout, groups, _ptr(stats),
                                            stats.numel() * stats.element_size(), _stream(stream)), "wan_causal_conv3d_gn_stats")
    return y, stats


def wan_gn_silu_from_stats(x, gamma, beta, groups: int, eps: float, stats, y=None, ws=None, stream=None):
    """silu(group_norm(x)) using the statistics wan_causal_conv3d_gn_stats emitted with x."""
    _need(x, torch.bfloat16, "x")
    _need(gamma, torch.float32, "gamma")
    _need(beta, torch.float32, "beta")
    N, T, H, W, C = x.shape
    y = torch.empty_like(x) if y is None else y
    _need(y, torch.bfloat16, "y")
    need = wan_workspace_size(WAN_OP_GN_SILU, N, T, H, W, C, 0, groups)
    ws = _workspace(need, x.device, ws)
    _check(lib().wan_gn_silu_from_stats(_ptr(x), _ptr(y), _ptr(gamma), _ptr(beta), N, T, H, W, C, groups, eps,
                                        _ptr(stats), stats.numel() * stats.element_size(), _ptr(ws), need if ws is not None else 0,
                                        _stream(stream)), "wan_gn_silu_from_stats")
    return y


def wan_gn_silu_causal_conv3d(x, gamma, beta, groups: int, eps: float, w, bias=None, residual=None, cache_in=None,
                              cache_out=None, y=None, ws=None, stream=None):
    """y = causal_conv3d(silu(group_norm(x)); cache_in) + bias + residual, and cache_out = the last two
    frames of [cache_in (or zeros); silu(group_norm(x))]; x [N, T, H, W, Cin], w [Cout, 3, 3, 3, Cin]."""
    for t, n in ((x, "x"), (w, "w"), (bias, "bias"), (residual, "residual"), (cache_in, "cache_in"),
                 (cache_out, "cache_out")):
        _need(t, torch.bfloat16, n)
    _need(gamma, torch.float32, "gamma")
    _need(beta, torch.float32, "beta")
    N, T, H, W, Cin = x.shape
    Cout = w.shape[0]
    y = torch.empty((N, T, H, W, Cout), dtype=torch.bfloat16, device=x.device) if y is None else y
    _need(y, torch.bfloat16, "y")
    need = wan_workspace_size(WAN_OP_GN_SILU_CONV3D, N, T, H, W, Cin, Cout, groups)
    ws = _workspace(need, x.device, ws)
    _check(lib().wan_gn_silu_causal_conv3d(_ptr(x), _ptr(gamma), _ptr(beta), groups, eps, _ptr(cache_in),
                                           _ptr(cache_out), _ptr(w), _ptr(bias), _ptr(residual), _ptr(y), N, T, H, W,
                                           Cin, Cout, _ptr(ws), need if ws is not None else 0, _stream(stream)),
           "wan_gn_silu_causal_conv3d")
    return y


def wan_gn_silu_coefficients(x, gamma, beta, groups: int, eps: float, coef=None, ws=None, stream=None):
    """Per-(frame, channel) GroupNorm + SiLU coefficients of x [N, T, H, W, C]: a uint8 device buffer of
    N*T*C*16 bytes, private layout, for wan_causal_conv3d_gn_input and wan_gn_silu_cache_update."""
    _need(x, torch.bfloat16, "x")
    _need(gamma, torch.float32, "gamma")
    _need(beta, torch.float32, "beta")
    N, T, H, W, C = x.shape
    coef = torch.empty(N * T * C * 16, dtype=torch.uint8, device=x.device) if coef is None else coef
    need = wan_workspace_size(WAN_OP_GN_SILU, N, T, H, W, C, 0, groups)
    ws = _workspace(need, x.device, ws)
    _check(lib().wan_gn_silu_coefficients(_ptr(x), _ptr(gamma), _ptr(beta), N, T, H, W, C, groups, eps, _ptr(coef),
                                          _ptr(ws), need if ws is not None else 0, _stream(stream)),
           "wan_gn_silu_coefficients")
    return coef


def wan_causal_conv3d_gn_input(x, coef, w, bias=None, residual=None, cache_in=None, y=None, stream=None,
                               cache_out=None):
    """y = causal_conv3d(silu(x S + B); cache_in) + bias + residual with coefficients from
    wan_gn_silu_coefficients(x, ...); Cout >= 256. cache_out (optional) receives the new history
    (written by the conv itself when it is not cache_in)."""
    for t, n in ((x, "x"), (w, "w"), (bias, "bias"), (residual, "residual"), (cache_in, "cache_in"),
                 (cache_out, "cache_out")):
        _need(t, torch.bfloat16, n)
    N, T, H, W, Cin = x.shape
    Cout = w.shape[0]
    y = torch.empty((N, T, H, W, Cout), dtype=torch.bfloat16, device=x.device) if y is None else y
    _need(y, torch.bfloat16, "y")
    _check(lib().wan_causal_conv3d_gn_input(_ptr(x), _ptr(coef), _ptr(cache_in), _ptr(cache_out), _ptr(w), _ptr(bias),
                                            _ptr(residual), _ptr(y), N, T, H, W, Cin, Cout, _stream(stream)),
           "wan_causal_conv3d_gn_input")
    return y


def wan_causal_conv3d_gn_input_stats(x, coef, w, groups: int, bias=None, residual=None, cache_in=None, y=None,
                                     stats=None, stream=None, cache_out=None):
    """wan_causal_conv3d_gn_input that also emits the GroupNorm statistics of y (for `groups` groups)
    for wan_gn_silu_coefficients_from_stats / wan_gn_silu_from_stats. Returns (y, stats)."""
    for t, n in ((x, "x"), (w, "w"), (bias, "bias"), (residual, "residual"), (cache_in, "cache_in"),
                 (cache_out, "cache_out")):
        _need(t, torch.bfloat16, n)
    N, T, H, W, Cin = x.shape
    Cout = w.shape[0]
    y = torch.empty((N, T, H, W, Cout), dtype=torch.bfloat16, device=x.device) if y is None else y
    _need(y, torch.bfloat16, "y")
    need = wan_workspace_size(WAN_OP_GN_STATS, N, T, H, W, Cin, Cout, groups)
    if need == 0:
        raise WanError(2, "wan_causal_conv3d_gn_input_stats")
    stats = _workspace(need, x.device, stats)
    _check(lib().wan_causal_conv3d_gn_input_stats(_ptr(x), _ptr(coef), _ptr(cache_in), _ptr(cache_out), _ptr(w),
                                                  _ptr(bias), _ptr(residual), _ptr(y), N, T, H, W, Cin, Cout, groups,
                                                  _ptr(stats), stats.numel() * stats.element_size(), _stream(stream)),
           "wan_causal_conv3d_gn_input_stats")
    return y, stats


def wan_gn_silu_coefficients_from_stats(stats, gamma, beta, shape, groups: int, eps: float, coef=None, stream=None):
    """The GroupNorm + SiLU coefficients of x (shape [N, T, H, W, C]) from the statistics the conv
    that wrote x emitted: a uint8 device buffer of N*T*C*16 bytes, as wan_gn_silu_coefficients'."""
    _need(gamma, torch.float32, "gamma")
    _need(beta, torch.float32, "beta")
    N, T, H, W, C = shape
    coef = torch.empty(N * T * C * 16, dtype=torch.uint8, device=stats.device) if coef is None else coef
    _check(lib().wan_gn_silu_coefficients_from_stats(_ptr(stats), stats.numel() * stats.element_size(), _ptr(gamma),
                                                     _ptr(beta), N, T, H, W, C, groups, eps, _ptr(coef),
                                                     _stream(stream)),
           "wan_gn_silu_coefficients_from_stats")
    return coef


def wan_gn_silu_cache_update(x, coef, cache_out, cache_in=None, stream=None):
    """cache_out = last two frames of [cache_in (or zeros); silu(x S + B)]; cache_out may be cache_in."""
    for t, n in ((x, "x"), (cache_in, "cache_in"), (cache_out, "cache_out")):
        _need(t, torch.bfloat16, n)
    N, T, H, W, C = x.shape
    _check(lib().wan_gn_silu_cache_update(_ptr(x), _ptr(coef), _ptr(cache_in), _ptr(cache_out), N, T, H, W, C,
                                          _stream(stream)), "wan_gn_silu_cache_update")
    return cache_out


def wan_cache_update(a, cache_out, cache_in=None, stream=None):
    """cache_out = last two frames of [cache_in (or zeros); a]; cache_out may be cache_in."""
    _need(a, torch.bfloat16, "a")
    _need(cache_out, torch.bfloat16, "cache_out")
    _need(cache_in, torch.bfloat16, "cache_in")
    N, T, H, W, C = a.shape
    _check(lib().wan_cache_update(_ptr(a), _ptr(cache_in), _ptr(cache_out), N, T, H, W, C, _stream(stream)),
           "wan_cache_update")
    return cache_out


def wan_upsample_phase_weights(w3, wp=None, stream=None):
    """[Cout, 3, 3, Cin] bf16 -> [4, Cout, 2, 2, Cin] bf16 phase weights."""
    _need(w3, torch.bfloat16, "w3")
    Cout, _, _, Cin = w3.shape
    wp = torch.empty((4, Cout, 2, 2, Cin), dtype=torch.bfloat16, device=w3.device) if wp is None else wp
    _need(wp, torch.bfloat16, "wp")
    _check(lib().wan_upsample_phase_weights(_ptr(w3), _ptr(wp), Cin, Cout, _stream(stream)),
           "wan_upsample_phase_weights")
    return wp


def wan_upsample_phase_conv(x, wp, bias=None, y=None, stream=None):
    """Nearest-x2 + 3x3 conv as four phase convs: x [N, T, H, W, Cin] -> [N, T, 2H, 2W, Cout]."""
    _need(x, torch.bfloat16, "x")
    _need(wp, torch.bfloat16, "wp")
    _need(bias, torch.bfloat16, "bias")
    N, T, H, W, Cin = x.shape
    Cout = wp.shape[1]
    y = torch.empty((N, T, 2 * H, 2 * W, Cout), dtype=torch.bfloat16, device=x.device) if y is None else y
    _need(y, torch.bfloat16, "y")
    _check(lib().wan_upsample_phase_conv(_ptr(x), _ptr(wp), _ptr(bias), _ptr(y), N, T, H, W, Cin, Cout,
                                         _stream(stream)), "wan_upsample_phase_conv")
    return y


def wan_resblock(x, params: dict, cache1, cache2, cache_valid: bool, groups: int, eps: float, out=None, ws=None,
                 stream=None):
    """One causal ResBlock on a chunk; params holds gamma1, beta1, w1, b1, gamma2, beta2, w2, b2."""
    _need(x, torch.bfloat16, "x")
    _need(cache1, torch.bfloat16, "cache1")
    _need(cache2, torch.bfloat16, "cache2")
    for k in ("gamma1", "beta1", "gamma2", "beta2"):
        _need(params[k], torch.float32, k)
    for k in ("w1", "b1", "w2", "b2"):
        _need(params.get(k), torch.bfloat16, k)
    N, T, H, W, C = x.shape
    out = torch.empty_like(x) if out is None else out
    _need(out, torch.bfloat16, "out")
    need = wan_workspace_size(WAN_OP_RESBLOCK, N, T, H, W, C, C, groups)
    ws = _workspace(need, x.device, ws)
    p = ResblockParams(_ptr(params["gamma1"]), _ptr(params["beta1"]), _ptr(params["w1"]), _ptr(params.get("b1")),
                       _ptr(params["gamma2"]), _ptr(params["beta2"]), _ptr(params["w2"]), _ptr(params.get("b2")),
                       groups, eps)
    _check(lib().wan_resblock(_ptr(x), _ptr(out), ctypes.byref(p), _ptr(cache1), _ptr(cache2), int(bool(cache_valid)),
                              N, T, H, W, C, _ptr(ws), need, _stream(stream)), "wan_resblock")
    return out


def wan_time_upsample(x, w, bias=None, first: bool = False, cache_in=None, cache_out=None, y=None, stream=None):
    """Causal 3x1x1 time conv to 2C channels, written as twice the frames (frame-interleaved); x
    [N, T, H, W, C], w [2C, 3, C]; with `first` the first frame passes through. Returns y
    [N, start + 2 (T - start), H, W, C]."""
    for t, n in ((x, "x"), (w, "w"), (bias, "bias"), (cache_in, "cache_in"), (cache_out, "cache_out")):
        _need(t, torch.bfloat16, n)
    N, T, H, W, C = x.shape
    start = 1 if first else 0
    y = torch.empty((N, start + 2 * (T - start), H, W, C), dtype=torch.bfloat16, device=x.device) if y is None else y
    _need(y, torch.bfloat16, "y")
    _check(lib().wan_time_upsample(_ptr(x), _ptr(cache_in), _ptr(cache_out), _ptr(w), _ptr(bias), _ptr(y), N, T, H, W,
                                   C, int(bool(first)), _stream(stream)), "wan_time_upsample")
    return y


def wan_conv1x1(x, w, y=None, stream=None):
    """y = x . w^T per pixel (w [Cout, Cin]), no bias."""
    _need(x, torch.bfloat16, "x")
    _need(w, torch.bfloat16, "w")
    N, T, H, W, Cin = x.shape
    Cout = w.shape[0]
    y = torch.empty((N, T, H, W, Cout), dtype=torch.bfloat16, device=x.device) if y is None else y
    _need(y, torch.bfloat16, "y")
    _check(lib().wan_conv1x1(_ptr(x), _ptr(w), _ptr(y), N, T, H, W, Cin, Cout, _stream(stream)), "wan_conv1x1")
    return y


def wan_fold_bias(b2, b_shortcut, out=None, stream=None):
    """bf16(b2 + b_shortcut): the shortcut bias folded into the second conv's."""
    _need(b2, torch.bfloat16, "b2")
    _need(b_shortcut, torch.bfloat16, "b_shortcut")
    out = torch.empty_like(b2) if out is None else out
    _check(lib().wan_fold_bias(_ptr(b2), _ptr(b_shortcut), _ptr(out), b2.numel(), _stream(stream)), "wan_fold_bias")
    return out


def wan_resblock_shortcut(x, params: dict, w_sc, cache1, cache2, cache_valid: bool, groups: int, eps: float, out=None,
                          ws=None, stream=None):
    """The channel-changing ResBlock: params as wan_resblock's with w1 [Cout, 3, 3, 3, Cin] and b2 the folded
    bias (wan_fold_bias); w_sc [Cout, Cin] the 1x1x1 shortcut."""
    _need(x, torch.bfloat16, "x")
    _need(w_sc, torch.bfloat16, "w_sc")
    _need(cache1, torch.bfloat16, "cache1")
    _need(cache2, torch.bfloat16, "cache2")
    for k in ("gamma1", "beta1", "gamma2", "beta2"):
        _need(params[k], torch.float32, k)
    for k in ("w1", "b1", "w2", "b2"):
        _need(params.get(k), torch.bfloat16, k)
    N, T, H, W, Cin = x.shape
    Cout = w_sc.shape[0]
    out = torch.empty((N, T, H, W, Cout), dtype=torch.bfloat16, device=x.device) if out is None else out
    _need(out, torch.bfloat16, "out")
    need = wan_workspace_size(WAN_OP_RESBLOCK_SHORTCUT, N, T, H, W, Cin, Cout, groups)
    ws = _workspace(need, x.device, ws)
    p = ResblockParams(_ptr(params["gamma1"]), _ptr(params["beta1"]), _ptr(params["w1"]), _ptr(params.get("b1")),
                       _ptr(params["gamma2"]), _ptr(params["beta2"]), _ptr(params["w2"]), _ptr(params.get("b2")),
                       groups, eps)
    _check(lib().wan_resblock_shortcut(_ptr(x), _ptr(out), ctypes.byref(p), _ptr(w_sc), _ptr(cache1), _ptr(cache2),
                                       int(bool(cache_valid)), N, T, H, W, Cin, Cout, _ptr(ws), need, _stream(stream)),
           "wan_resblock_shortcut")
    return out


def wan_winograd_weights(w, u=None, stream=None):
    """u [16, Cout, 3, Cin] fp16 (as torch.float16) = G g G^T per temporal tap of w [Cout, 3, 3, 3, Cin]."""
    _need(w, torch.bfloat16, "w")
    Cout, Cin = w.shape[0], w.shape[-1]
    u = torch.empty((16, Cout, 3, Cin), dtype=torch.float16, device=w.device) if u is None else u
    _need(u, torch.float16, "u")
    _check(lib().wan_winograd_weights(_ptr(w), _ptr(u), Cin, Cout, _stream(stream)), "wan_winograd_weights")
    return u


def wan_causal_conv3d_winograd(a, u, coef=None, bias=None, residual=None, cache_in=None, cache_out=None, y=None,
                               ws=None, stream=None):
    """The causal conv of a (or of silu(a S + B) with GroupNorm coefficients `coef`) through
    Winograd F(2x2, 3x3) with weights u from wan_winograd_weights."""
    for t, n in ((a, "a"), (bias, "bias"), (residual, "residual"), (cache_in, "cache_in"), (cache_out, "cache_out")):
        _need(t, torch.bfloat16, n)
    _need(u, torch.float16, "u")
    N, T, H, W, Cin = a.shape
    Cout = u.shape[1]
    y = torch.empty((N, T, H, W, Cout), dtype=torch.bfloat16, device=a.device) if y is None else y
    _need(y, torch.bfloat16, "y")
    need = wan_workspace_size(WAN_OP_WINOGRAD_CONV3D, N, T, H, W, Cin, Cout, 0)
    ws = _workspace(need, a.device, ws)
    _check(lib().wan_causal_conv3d_winograd(_ptr(a), _ptr(coef), _ptr(cache_in), _ptr(cache_out), _ptr(u), _ptr(bias),
                                            _ptr(residual), _ptr(y), N, T, H, W, Cin, Cout, _ptr(ws), need,
                                            _stream(stream)), "wan_causal_conv3d_winograd")
    return y


def wan_causal_conv3d_winograd_stats(a, u, groups: int, coef=None, bias=None, residual=None, cache_in=None,
                                     cache_out=None, y=None, stats=None, ws=None, stream=None):
    """wan_causal_conv3d_winograd that also emits the GroupNorm statistics of y (for `groups` groups)
    for wan_gn_silu_coefficients_from_stats / wan_gn_silu_from_stats. Returns (y, stats)."""
    for t, n in ((a, "a"), (bias, "bias"), (residual, "residual"), (cache_in, "cache_in"), (cache_out, "cache_out")):
        _need(t, torch.bfloat16, n)
    _need(u, torch.float16, "u")
    N, T, H, W, Cin = a.shape
    Cout = u.shape[1]
    y = torch.empty((N, T, H, W, Cout), dtype=torch.bfloat16, device=a.device) if y is None else y
    _need(y, torch.bfloat16, "y")
    need = wan_workspace_size(WAN_OP_WINOGRAD_CONV3D, N, T, H, W, Cin, Cout, 0)
    ws = _workspace(need, a.device, ws)
    st_need = wan_workspace_size(WAN_OP_GN_STATS_WINOGRAD, N, T, H, W, Cin, Cout, groups)
    if st_need == 0:
        raise WanError(2, "wan_causal_conv3d_winograd_stats")
    stats = _workspace(st_need, a.device, stats)
    _check(lib().wan_causal_conv3d_winograd_stats(_ptr(a), _ptr(coef), _ptr(cache_in), _ptr(cache_out), _ptr(u),
                                                  _ptr(bias), _ptr(residual), _ptr(y), N, T, H, W, Cin, Cout, groups,
                                                  _ptr(stats), stats.numel() * stats.element_size(), _ptr(ws), need,
                                                  _stream(stream)), "wan_causal_conv3d_winograd_stats")
    return y, stats


def wan_resblock_winograd(x, params, u1, u2, cache1, cache2, cache_valid, groups: int, eps: float, out=None, ws=None,
                          stream=None):
    """wan_resblock with both convs through Winograd F(2x2, 3x3) (u1, u2 from wan_winograd_weights)."""
    _need(x, torch.bfloat16, "x")
    _need(u1, torch.float16, "u1")
    _need(u2, torch.float16, "u2")
    N, T, H, W, C = x.shape
    out = torch.empty_like(x) if out is None else out
    need = wan_workspace_size(WAN_OP_RESBLOCK_WINOGRAD, N, T, H, W, C, C, groups)
    ws = _workspace(need, x.device, ws)
    p = ResblockParams(_ptr(params["gamma1"]), _ptr(params["beta1"]), None, _ptr(params.get("b1")),
                       _ptr(params["gamma2"]), _ptr(params["beta2"]), None, _ptr(params.get("b2")), groups, eps)
    _check(lib().wan_resblock_winograd(_ptr(x), _ptr(out), ctypes.byref(p), _ptr(u1), _ptr(u2), _ptr(cache1),
                                       _ptr(cache2), int(bool(cache_valid)), N, T, H, W, C, _ptr(ws), need,
                                       _stream(stream)), "wan_resblock_winograd")
    return out


def wan_selftest_wait_timeout(which: int, wait_cycles: int, x=None, gamma=None, beta=None, groups: int = 0,
                              eps: float = 1e-6, y=None, ws=None, stream=None) -> int:
    """Makes one bounded device wait run out on purpose (which 0: the GroupNorm kernel's grid
    barrier on x; which 1: an mbarrier wait); returns the call's status (the timeout itself is
    reported by wan_device_status)."""
    if which == 0:
        _need(x, torch.bfloat16, "x")
        _need(gamma, torch.float32, "gamma")
        _need(beta, torch.float32, "beta")
        N, T, H, W, C = x.shape
        y = torch.empty_like(x) if y is None else y
        need = wan_workspace_size(WAN_OP_GN_SILU, N, T, H, W, C, 0, groups)
        ws = _workspace(need, x.device, ws)
        return int(lib().wan_selftest_wait_timeout(0, wait_cycles, _ptr(x), _ptr(y), _ptr(gamma), _ptr(beta),
                                                   N, T, H, W, C, groups, eps, _ptr(ws), need, _stream(stream)))
    return int(lib().wan_selftest_wait_timeout(which, wait_cycles, None, None, None, None, 0, 0, 0, 0, 0, 0, eps,
                                               None, 0, _stream(stream)))


def wan_device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the library's device error status."""
    return int(lib().wan_device_status(_stream(stream)))
