"""Host-side checks of the C ABI that need no GPU: the library loads, exports every entry point
include/wan.h declares, and rejects invalid arguments before touching the device."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "wan.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wan_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from video_vae_decoder_gb300 import build, binding
    build.build()
    return binding.lib()


def test_exports_every_declared_symbol(L):
    syms = declared_symbols()
    assert "wan_resblock" in syms and "wan_gn_silu" in syms
    for s in syms:
        assert hasattr(L, s), f"{s} declared in wan.h but not exported"
    from video_vae_decoder_gb300 import binding
    assert set(binding.EXPORTS) == set(syms)


def test_status_strings(L):
    from video_vae_decoder_gb300 import binding
    for code, name in binding.STATUS.items():
        assert binding.wan_status_string(code).startswith(name)
    assert binding.wan_status_string(99) == "WAN_ERR_UNKNOWN"


def test_workspace_sizes(L):
    from video_vae_decoder_gb300 import binding as b
    assert b.wan_workspace_size(b.WAN_OP_CAUSAL_CONV3D, 1, 4, 8, 8, 64, 64) == 0
    gn = b.wan_workspace_size(b.WAN_OP_GN_SILU, 1, 4, 88, 156, 512, 0, 32)
    assert gn >= 4 * 512 * 16  # per-frame per-channel coefficients at least
    rb = b.wan_workspace_size(b.WAN_OP_RESBLOCK, 1, 4, 16, 16, 64, 64, 32)
    assert rb >= 2 * 4 * 16 * 16 * 64 * 2
    assert b.wan_workspace_size(b.WAN_OP_GN_SILU, 1, 4, 8, 8, 60, 0, 32) == 0   # groups do not divide C
    # statistics of a conv output: a 256-byte header, then a float4 + float2 per (frame, group, tile,
    # epilogue warp) for the tiling with more tiles (8 x 16: 22 x 20 at 176 x 312; 16 x 8: 11 x 39)
    st = b.wan_workspace_size(b.WAN_OP_GN_STATS, 1, 4, 176, 312, 256, 256, 32)
    assert st == 256 + 4 * 32 * (22 * 20 * 4) * 24
    st = b.wan_workspace_size(b.WAN_OP_GN_STATS, 1, 4, 88, 156, 256, 256, 32)
    assert st == 256 + 4 * 32 * (6 * 20 * 4) * 24  # 16 x 8 tiles need more here (120 against 110)
    assert b.wan_workspace_size(b.WAN_OP_GN_STATS, 1, 4, 16, 16, 64, 320, 32) == 0   # Cout % 256 != 0
    assert b.wan_workspace_size(b.WAN_OP_GN_STATS, 1, 4, 16, 16, 64, 256, 128) == 0  # 2 channels per group
    assert b.wan_workspace_size(b.WAN_OP_GN_STATS, 1, 4, 16, 16, 64, 768, 64) == 0   # 12 channels per group
    assert b.wan_workspace_size(b.WAN_OP_GN_STATS, 1, 4, 16, 16, 64, 512, 4) == 0    # 128 channels per group
    # GroupNorm + SiLU into a causal conv: Cout >= 256 never stores the activation (only the norm's
    # workspace); smaller convs read it from the workspace.
    def a256(n):
        return (n + 255) // 256 * 256
    gnws = b.wan_workspace_size(b.WAN_OP_GN_SILU, 1, 4, 16, 16, 256, 0, 32)
    assert b.wan_workspace_size(b.WAN_OP_GN_SILU_CONV3D, 1, 4, 16, 16, 256, 256, 32) == a256(gnws)
    gn1 = b.wan_workspace_size(b.WAN_OP_GN_SILU, 1, 1, 16, 16, 256, 0, 32)
    assert b.wan_workspace_size(b.WAN_OP_GN_SILU_CONV3D, 1, 1, 16, 16, 256, 256, 32) == a256(gn1)
    gn64 = b.wan_workspace_size(b.WAN_OP_GN_SILU, 1, 4, 16, 16, 64, 0, 32)
    assert b.wan_workspace_size(b.WAN_OP_GN_SILU_CONV3D, 1, 4, 16, 16, 64, 64, 32) == a256(gn64) + 4 * 16 * 16 * 64 * 2
    assert b.wan_workspace_size(b.WAN_OP_GN_SILU_CONV3D, 1, 4, 16, 16, 60, 64, 32) == 0  # groups do not divide Cin
    # statistics from the Winograd output transform: a 256-byte header, then a float4 + float2 per
    # (frame, group, 2x2 output tile); the Winograd ResBlock holds one such buffer for h
    assert b.wan_workspace_size(b.WAN_OP_GN_STATS_WINOGRAD, 1, 4, 44, 78, 1024, 1024, 32) == 256 + 4 * 32 * (22 * 39) * 24
    assert b.wan_workspace_size(b.WAN_OP_GN_STATS_WINOGRAD, 1, 2, 1, 1, 64, 256, 32) == 256 + 2 * 32 * 1 * 24
    assert b.wan_workspace_size(b.WAN_OP_GN_STATS_WINOGRAD, 1, 4, 16, 16, 64, 320, 32) == 0    # Cout % 256 != 0
    assert b.wan_workspace_size(b.WAN_OP_GN_STATS_WINOGRAD, 1, 4, 16, 16, 64, 256, 128) == 0   # 2 channels per group
    assert b.wan_workspace_size(b.WAN_OP_GN_STATS_WINOGRAD, 1, 4, 16, 16, 64, 512, 4) == 0     # 128 channels per group
    rbw = b.wan_workspace_size(b.WAN_OP_RESBLOCK_WINOGRAD, 1, 4, 44, 78, 1024, 1024, 32)
    parts = (a256(4 * 44 * 78 * 1024 * 2) + a256(4 * 1024 * 16) +
             a256(b.wan_workspace_size(b.WAN_OP_GN_STATS_WINOGRAD, 1, 4, 44, 78, 1024, 1024, 32)) +
             a256(b.wan_workspace_size(b.WAN_OP_GN_SILU, 1, 4, 44, 78, 1024, 0, 32)) +
             b.wan_workspace_size(b.WAN_OP_WINOGRAD_CONV3D, 1, 4, 44, 78, 1024, 1024, 0))
    assert rbw == parts
    # 2 channels per group: no statistics buffer (its second norm takes a pass over h)
    rbw2 = b.wan_workspace_size(b.WAN_OP_RESBLOCK_WINOGRAD, 1, 4, 44, 78, 256, 256, 128)
    assert rbw2 == (a256(4 * 44 * 78 * 256 * 2) + a256(4 * 256 * 16) +
                    a256(b.wan_workspace_size(b.WAN_OP_GN_SILU, 1, 4, 44, 78, 256, 0, 128)) +
                    b.wan_workspace_size(b.WAN_OP_WINOGRAD_CONV3D, 1, 4, 44, 78, 256, 256, 0))
    # the ResBlock: h, then the norm-into-conv workspace shared by its two convs
    assert b.wan_workspace_size(b.WAN_OP_RESBLOCK, 1, 4, 16, 16, 256, 256, 32) == \
        4 * 16 * 16 * 256 * 2 + b.wan_workspace_size(b.WAN_OP_GN_SILU_CONV3D, 1, 4, 16, 16, 256, 256, 32)


# Fake, never-dereferenced device addresses: every call below must be rejected on the host.
A = 1 << 20          # 16-byte aligned
MIS = (1 << 20) + 2  # misaligned


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_gn_rejects_invalid(L):
    f = L.wan_gn_silu
    args = dict(x=A, y=A * 3, g=A * 5, b=A * 7, N=1, T=2, H=4, W=4, C=64, G=32, eps=1e-6)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["x"], a["y"], a["g"], a["b"], a["N"], a["T"], a["H"], a["W"], a["C"], a["G"],
                 ctypes.c_float(a["eps"]), A * 9, 1 << 30, None)
    assert call(x=None) == 1
    assert call(T=0) == 1
    assert call(G=24) == 1            # does not divide 64
    assert call(C=60, G=4) == 2       # C % 8 != 0
    assert call(C=2112, G=32) == 2    # wider than the 2048 channels the kernel supports
    assert call(eps=0.0) == 1
    assert call(x=MIS) == 3
    assert call(y=A) == 1             # y overlaps x
    assert f(A, A * 3, A * 5, A * 7, 1, 2, 4, 4, 64, 32, ctypes.c_float(1e-6), A * 9, 8, None) == 4


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_gn_clip_rejects_invalid(L):
    f = L.wan_gn_silu_clip

    def call(x=A, y=A * 3, N=1, T=2, H=4, W=4, C=64, G=32, eps=1e-6, ws=A * 9, wsb=1 << 30):
        return f(x, y, A * 5, A * 7, N, T, H, W, C, G, ctypes.c_float(eps), ws, wsb, None)
    assert call(x=None) == 1
    assert call(T=0) == 1
    assert call(G=24) == 1                     # does not divide 64
    assert call(y=A) == 1                      # y overlaps x
    assert call(x=MIS) == 3
    assert call(wsb=8) == 4                    # workspace too small
    assert call(y=1 << 40, H=4096, W=4096, C=64, G=2) == 2  # a frame count of 2^29 is not exact in fp32


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_conv_rejects_invalid(L):
    f = L.wan_causal_conv3d
    ok = (A, None, None, A * 5, None, None, A * 9)
    assert f(*ok, 1, 2, 4, 4, 48, 64, None, 0, None) == 2      # Cin % 64 != 0
    assert f(*ok, 1, 2, 4, 4, 64, 63, None, 0, None) == 2      # odd Cout
    assert f(*ok, 1, 0, 4, 4, 64, 64, None, 0, None) == 1      # T = 0
    assert f(None, None, None, A * 5, None, None, A * 9, 1, 2, 4, 4, 64, 64, None, 0, None) == 1
    assert f(MIS, None, None, A * 5, None, None, A * 9, 1, 2, 4, 4, 64, 64, None, 0, None) == 3
    # y overlapping a
    assert f(A, None, None, A * 5, None, None, A + 64, 1, 2, 4, 4, 64, 64, None, 0, None) == 1
    # cache_out overlapping a
    assert f(A, None, A + 128, A * 5, None, None, A * 9, 1, 2, 4, 4, 64, 64, None, 0, None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_fused_gn_statistics_calls_reject_invalid(L):
    f = L.wan_causal_conv3d_gn_stats
    ok = (A, None, None, A * 5, None, None, A * 9)
    big = 1 << 30
    assert f(*ok, 1, 2, 16, 16, 64, 320, 32, A * 13, big, None) == 2    # Cout % 256 != 0
    assert f(*ok, 1, 2, 16, 16, 64, 256, 128, A * 13, big, None) == 2   # 2 channels per group
    assert f(*ok, 1, 2, 16, 16, 64, 256, 32, None, big, None) == 1      # no statistics buffer
    assert f(*ok, 1, 2, 16, 16, 64, 256, 32, MIS, big, None) == 3       # misaligned statistics buffer
    assert f(*ok, 1, 2, 16, 16, 64, 256, 32, A * 13, 64, None) == 1     # buffer too small
    g = L.wan_gn_silu_from_stats
    gn = (A, A * 3, A * 5, A * 7)
    assert g(*gn, 1, 2, 16, 16, 256, 32, 1e-6, None, big, A * 11, big, None) == 1      # no statistics
    assert g(*gn, 1, 2, 16, 16, 64, 32, 1e-6, A * 13, big, A * 11, big, None) == 2     # C % 256 != 0
    assert g(*gn, 1, 2, 16, 16, 256, 32, 1e-6, A * 13, 64, A * 11, big, None) == 1     # buffer too small
    assert g(*gn, 1, 2, 16, 16, 256, 32, 1e-6, A * 13, big, None, 0, None) == 4        # no workspace


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_winograd_statistics_call_rejects_invalid(L):
    f = L.wan_causal_conv3d_winograd_stats
    # a, coef, cache_in, cache_out, u, bias, residual, y; then sizes, groups, stats, its bytes, ws, its bytes
    ok = (A, None, None, None, A * 3, None, None, A * 5)
    sz = (1, 2, 16, 16, 64, 256)
    big = 1 << 30
    st, ws = A * 64, A * 32
    assert f(*ok, *sz, 32, st, big, ws, big, None) == 5       # every argument accepted: no device to run on
    assert f(*ok, 1, 2, 16, 16, 64, 320, 32, st, big, ws, big, None) == 2   # Cout % 256 != 0
    assert f(*ok, *sz, 128, st, big, ws, big, None) == 2      # 2 channels per group
    assert f(*ok, *sz, 0, st, big, ws, big, None) == 1        # no groups
    assert f(*ok, *sz, 32, None, big, ws, big, None) == 1     # no statistics buffer
    assert f(*ok, *sz, 32, MIS, big, ws, big, None) == 3      # misaligned statistics buffer
    assert f(*ok, *sz, 32, st, 64, ws, big, None) == 1        # statistics buffer too small
    assert f(*ok, *sz, 32, A * 5, big, ws, big, None) == 1    # statistics overlapping y
    assert f(*ok, *sz, 32, st, big, None, 0, None) == 4       # no workspace
    g = L.wan_gn_silu_coefficients_from_stats
    # 1 x 1 frames: the Winograd statistics (one record per frame and group) are the smallest
    assert g(st, 256 + 2 * 32 * 24 - 1, A * 3, A * 5, 1, 2, 1, 1, 256, 32, 1e-6, A * 7, None) == 1
    assert g(st, 256 + 2 * 32 * 24, A * 3, A * 5, 1, 2, 1, 1, 256, 32, 1e-6, A * 7, None) == 5


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_gn_silu_causal_conv3d_rejects_invalid(L):
    f = L.wan_gn_silu_causal_conv3d
    big = 1 << 30

    def call(x=A, groups=32, eps=1e-6, cache_in=None, cache_out=A * 20, y=A * 9, Cin=256, ws=A * 30, ws_bytes=big):
        return f(x, A * 2, A * 3, groups, eps, cache_in, cache_out, A * 5, None, None, y, 1, 2, 16, 16, Cin, 256,
                 ws, ws_bytes, None)
    assert call(x=None) == 1                        # no input
    assert call(groups=48) == 1                     # groups do not divide Cin
    assert call(eps=0.0) == 1                       # eps must be positive
    assert call(Cin=96) == 2                        # the conv wants Cin % 64 == 0
    assert call(y=A) == 1                           # y overlaps x
    assert call(cache_out=A + 4096) == 1            # the cache overlaps x
    assert call(cache_in=MIS) == 3                  # misaligned history
    assert call(ws=None) == 4                       # no workspace
    assert call(ws_bytes=64) == 4                   # workspace too small


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_gn_silu_steps_reject_invalid(L):
    big = 1 << 30
    co = L.wan_gn_silu_coefficients
    assert co(A, A * 2, A * 3, 1, 2, 16, 16, 96, 32, 1e-6, A * 4, A * 5, big, None) == 2   # C % 64 != 0
    assert co(A, A * 2, A * 3, 1, 2, 16, 16, 256, 32, 1e-6, None, A * 5, big, None) == 1  # no coefficient buffer
    assert co(A, A * 2, A * 3, 1, 2, 16, 16, 256, 32, 1e-6, A * 4, None, 0, None) == 4    # no workspace
    cv = L.wan_causal_conv3d_gn_input
    assert cv(A, None, None, None, A * 5, None, None, A * 9, 1, 2, 16, 16, 256, 256, None) == 1  # no coefficients
    assert cv(A, A * 4, None, None, A * 5, None, None, A * 9, 1, 2, 16, 16, 256, 128, None) == 2  # Cout < 256
    assert cv(A, MIS, None, None, A * 5, None, None, A * 9, 1, 2, 16, 16, 256, 256, None) == 3    # misaligned coefficients
    assert cv(A, A * 4, None, None, A * 5, None, None, A, 1, 2, 16, 16, 256, 256, None) == 1      # y overlaps x
    assert cv(A, A * 4, None, A + 4096, A * 5, None, None, A * 9, 1, 2, 16, 16, 256, 256, None) == 1  # cache_out on x
    assert cv(A, A * 4, A * 20, A * 20 + 64, A * 5, None, None, A * 9, 1, 2, 16, 16, 256, 256, None) == 1  # caches overlap
    cu = L.wan_gn_silu_cache_update
    assert cu(A, A * 4, None, None, 1, 2, 16, 16, 256, None) == 1        # no cache_out
    assert cu(A, A * 4, None, A * 20, 1, 2, 16, 16, 96, None) == 2       # C % 64 != 0
    assert cu(A, A * 4, MIS, A * 20, 1, 2, 16, 16, 256, None) == 3       # misaligned history
    assert cu(A, A * 4, None, A + 4096, 1, 2, 16, 16, 256, None) == 1    # cache overlaps x


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_adjacent_steps_reject_invalid(L):
    tu = L.wan_time_upsample
    assert tu(None, None, None, A * 5, None, A * 9, 1, 2, 8, 16, 256, 1, None) == 1     # no input
    assert tu(A, None, None, A * 5, None, A * 9, 1, 2, 8, 16, 128, 1, None) == 2       # C % 256 != 0
    assert tu(A, None, None, MIS, None, A * 9, 1, 2, 8, 16, 256, 1, None) == 3         # misaligned weights
    assert tu(A, None, None, A * 5, None, A + 4096, 1, 2, 8, 16, 256, 1, None) == 1    # y overlaps x
    c1 = L.wan_conv1x1
    assert c1(A, A * 5, A * 9, 1, 2, 8, 16, 96, 256, None) == 2    # Cin % 64 != 0
    assert c1(A, A * 5, A * 9, 1, 2, 8, 16, 128, 128, None) == 2   # Cout < 256
    assert c1(A, A * 5, A, 1, 2, 8, 16, 128, 256, None) == 1       # y overlaps x
    assert L.wan_fold_bias(None, A, A * 2, 256, None) == 1
    assert L.wan_fold_bias(A, A * 2, A * 3, 0, None) == 1
    from video_vae_decoder_gb300.binding import ResblockParams
    p = ResblockParams(A * 2, A * 3, A * 4, None, A * 5, A * 6, A * 7, None, 32, 1e-6)
    rs = L.wan_resblock_shortcut
    assert rs(A, A * 40, ctypes.byref(p), None, A * 50, A * 60, 0, 1, 2, 4, 4, 128, 256, A * 70, 1 << 30, None) == 1
    assert rs(A, A * 40, ctypes.byref(p), A * 45, A * 50, A * 60, 0, 1, 2, 4, 4, 128, 128, A * 70, 1 << 30, None) == 2
    assert rs(A, A * 40, ctypes.byref(p), A * 45, A * 50, A * 60, 0, 1, 2, 4, 4, 128, 256, A * 70, 16, None) == 4


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_resblock_and_upsample_reject_invalid(L):
    from video_vae_decoder_gb300.binding import ResblockParams
    p = ResblockParams(A * 2, A * 3, A * 4, None, A * 5, A * 6, A * 7, None, 32, 1e-6)
    f = L.wan_resblock
    assert f(A, A * 40, None, A * 50, A * 60, 0, 1, 2, 4, 4, 64, A * 70, 1 << 30, None) == 1   # no params
    assert f(A, A * 40, ctypes.byref(p), A * 50, A * 50, 0, 1, 2, 4, 4, 64, A * 70, 1 << 30, None) == 1  # caches alias
    assert f(A, A * 40, ctypes.byref(p), A * 50, A * 60, 0, 1, 2, 4, 4, 64, A * 70, 16, None) == 4      # workspace
    p.groups = 48
    assert f(A, A * 40, ctypes.byref(p), A * 50, A * 60, 0, 1, 2, 4, 4, 64, A * 70, 1 << 30, None) == 1
    assert L.wan_upsample_phase_weights(None, A, 64, 64, None) == 1
    assert L.wan_upsample_phase_weights(MIS, A * 8, 64, 64, None) == 3
    assert L.wan_upsample_phase_conv(A, A * 3, None, A * 9, 1, 1, 4, 4, 32, 64, None) == 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_gn_noalloc_refuses_sizes_beyond_its_static_scratch(L):
    # [1, 64, 176, 312, 256] with 32 groups needs more scratch than the fixed 4 MiB: refused on
    # the host with WAN_ERR_WORKSPACE, before any device work.
    from video_vae_decoder_gb300 import binding as b
    assert b.wan_workspace_size(b.WAN_OP_GN_SILU, 1, 64, 176, 312, 256, 0, 32) > 4 << 20
    f = L.wan_gn_silu_noalloc
    x, y = A, A << 12
    assert f(x, y, A * 5, A * 7, 1, 64, 176, 312, 256, 32, ctypes.c_float(1e-6), None) == 4
    assert f(None, y, A * 5, A * 7, 1, 4, 8, 8, 256, 32, ctypes.c_float(1e-6), None) == 1
    assert f(MIS, y, A * 5, A * 7, 1, 4, 8, 8, 256, 32, ctypes.c_float(1e-6), None) == 3


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers are only passed where no GPU exists")
def test_selftest_wait_timeout_rejects_invalid(L):
    f = L.wan_selftest_wait_timeout
    eps = ctypes.c_float(1e-6)
    assert f(2, 100000, None, None, None, None, 0, 0, 0, 0, 0, 0, eps, None, 0, None) == 1        # no such wait
    assert f(1, 10, None, None, None, None, 0, 0, 0, 0, 0, 0, eps, None, 0, None) == 1            # bound too short
    assert f(1, 10 ** 9, None, None, None, None, 0, 0, 0, 0, 0, 0, eps, None, 0, None) == 1       # too long
    # which = 0 checks its tensors as wan_gn_silu does, before anything is enqueued
    assert f(0, 100000, None, A * 3, A * 5, A * 7, 1, 2, 4, 4, 64, 32, eps, A * 9, 1 << 30, None) == 1
    assert f(0, 100000, MIS, A * 3, A * 5, A * 7, 1, 2, 4, 4, 64, 32, eps, A * 9, 1 << 30, None) == 3
    assert f(0, 100000, A, A * 3, A * 5, A * 7, 1, 2, 4, 4, 64, 32, eps, A * 9, 8, None) == 4
