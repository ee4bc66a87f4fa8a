#!/usr/bin/env python
"""Benchmark of the causal video-VAE decoder hot path on GB300 (one JSON line on stdout).

A step is one steady-state pass of every op of the path over one batch of synthetic input,
each op at the decoder shape it is quoted on:
  gn      GroupNorm+SiLU standalone, x [1, 4, 88, 156, 512] ~ N(0.5, var 2), 32 groups
  c256    three causal ResBlocks at C=256 on a 4-frame chunk [1, 4, 176, 312, 256] with the
          two-frame caches carried from the previous chunk (per block: the norm's coefficients, the
          causal conv normalising its input and writing the new history, the same for conv 2 with
          the residual; each conv's history alternates between two buffers)
  up      phase-weight transform [512, 3, 3, 512] and the nearest-x2 + 3x3 upsample as four phase
          convs, [1, 4, 44, 78, 512] -> [1, 4, 88, 156, 512]
  c1024   two causal ResBlocks at C=1024 on [1, 4, 44, 78, 1024] with carried caches, their convs
          through Winograd F(2x2, 3x3) with fp16 operands (weights transformed once, as the
          pages' prepare() does; FLOPs counted as the direct conv's)
  head    causal 3x3x3 conv 256 -> 12 channels on [1, 16, 704, 1248, 256] (zero history)
value = useful convolution FLOPs of the step / step time (TFLOP/s); the per-op times, GN GB/s,
ResBlock ms and the dominant kernel's roofline fraction are reported beside it. The step's
working set (about 8 GB) is far larger than L2, so no flush is inserted between steps.

--impl reference times the fp64 CPU oracle on the host cores (a bounded sample of the C=256
ResBlock workload per step), in the same unit.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal conv3d TFLOP/s (% bf16 peak); GN+SiLU GB/s (% HBM); ResBlock ms"
EPS = 1e-6
GROUPS = 32


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def conv_flops(N, T, H, W, Cin, Cout):
    return 2.0 * N * T * H * W * Cout * 27 * Cin


def wino_flops(N, T, H, W, Cin, Cout):
    """Tensor work of the Winograd F(2x2, 3x3) causal conv: per 2x2 output tile, 16 component
    products over 3 temporal taps x Cin input channels for each output channel."""
    return 2.0 * N * T * ((H + 1) // 2) * ((W + 1) // 2) * 16 * Cout * 3 * Cin


def phase_flops(N, T, H, W, Cin, Cout):
    return 2.0 * N * T * H * W * 4 * Cout * 4 * Cin


# ------------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and parts[0] != self.uuid:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        load = [s for s in sm]
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------------------------------------
# the GPU workload
# ------------------------------------------------------------------------------------------------
CASES = ("all", "gn", "c256", "up", "c1024", "head")


class Workload:
    def __init__(self, dev, case="all", seed=0, head_frames=16):
        import numpy as np
        import torch
        from video_vae_decoder_gb300 import synth
        self.dev = dev
        bf = torch.bfloat16

        def n(shape, name, mean=0.0, std=1.0, dtype=bf):
            return synth.normal_torch(shape, seed, name, mean, std, device=dev, dtype=dtype)

        def block(C, prefix):
            wstd = float(np.sqrt(1.0 / (27 * C)))
            p = {}
            for k in (1, 2):
                p[f"gamma{k}"] = n((C,), f"{prefix}/gamma{k}", 1.0, 0.1, torch.float32)
                p[f"beta{k}"] = n((C,), f"{prefix}/beta{k}", 0.0, 0.1, torch.float32)
                p[f"w{k}"] = n((C, 3, 3, 3, C), f"{prefix}/w{k}", 0.0, wstd)
                p[f"b{k}"] = n((C,), f"{prefix}/b{k}", 0.0, 0.01)
            return p

        self.case = case
        want = (lambda part: case in ("all", part))
        # gn: standalone GroupNorm+SiLU at decode-mid scale (its gamma/beta also serve the e2e leg)
        self.gn_x = n((1, 4, 88, 156, 512), "bench/gn/x", 0.5, float(np.sqrt(2.0)))
        self.gn_g = n((512,), "bench/gn/gamma", 1.0, 0.1, torch.float32)
        self.gn_b = n((512,), "bench/gn/beta", 0.0, 0.1, torch.float32)
        self.gn_y = torch.empty_like(self.gn_x)
        # c256: decoder stage
        small = (1, 1, 8, 8)
        self.x4 = n((1, 4, 176, 312, 256) if want("c256") else small + (256,), "bench/c256/x")
        self.blocks4 = [block(256, f"bench/c256/block{i}") for i in range(3 if want("c256") else 0)]
        # up: spatial upsample
        self.x3 = n((1, 4, 44, 78, 512) if want("up") else small + (512,), "bench/up/x")
        self.w3 = n((512, 3, 3, 512), "bench/up/w3", 0.0, float(np.sqrt(1.0 / (9 * 512))))
        self.wp = torch.empty((4, 512, 2, 2, 512), dtype=bf, device=dev)
        self.y3 = torch.empty((1, 4, 88, 156, 512), dtype=bf, device=dev)
        # c1024: widest stage
        self.x5 = n((1, 4, 44, 78, 1024) if want("c1024") else small + (1024,), "bench/c1024/x")
        self.blocks5 = [block(1024, f"bench/c1024/block{i}") for i in range(2 if want("c1024") else 0)]
        # head
        hshape = (1, head_frames, 704, 1248, 256) if want("head") else (1, 1, 8, 8, 256)
        self.xh = n(hshape, "bench/head/x")
        self.wh = n((12, 3, 3, 3, 256), "bench/head/w", 0.0, float(np.sqrt(1.0 / (27 * 256))))
        self.yh = torch.empty(hshape[:-1] + (12,), dtype=bf, device=dev)

        def stage_bufs(x, nblk):
            N, T, H, W, C = x.shape
            caches = [(torch.zeros((N, 2, H, W, C), dtype=bf, device=dev),
                       torch.zeros((N, 2, H, W, C), dtype=bf, device=dev)) for _ in range(nblk)]
            # the second buffer of each conv's history: the step's convs read one and write the other
            self.alt.extend(torch.zeros((N, 2, H, W, C), dtype=bf, device=dev) for _ in range(2 * nblk))
            outs = [torch.empty_like(x) for _ in range(nblk)]
            coef = torch.empty(N * T * C * 16, dtype=torch.uint8, device=dev)  # GroupNorm coefficients
            return caches, outs, coef, torch.empty_like(x)
        self.alt = []
        self.c4, self.o4, self.k4, self.h4 = stage_bufs(self.x4, 3)
        self.alt4, self.alt = self.alt, []
        self.c5, self.o5, self.k5, self.h5 = stage_bufs(self.x5, 2)
        self.alt5, self.alt = self.alt, []
        from video_vae_decoder_gb300 import binding as wan
        # the C=1024 convs' Winograd weights, transformed once per weight set (prepare)
        self.u5 = [(wan.wan_winograd_weights(p["w1"]), wan.wan_winograd_weights(p["w2"])) for p in self.blocks5]
        self.wino_ws = torch.empty(wan.wan_workspace_size(wan.WAN_OP_WINOGRAD_CONV3D, *self.x5.shape, self.x5.shape[-1],
                                                          0), dtype=torch.uint8, device=dev)
        self.rbw_ws = torch.empty(wan.wan_workspace_size(wan.WAN_OP_RESBLOCK_WINOGRAD, *self.x5.shape, self.x5.shape[-1],
                                                         GROUPS), dtype=torch.uint8, device=dev)
        # GroupNorm statistics written by the C=1024 stage's Winograd convs with their outputs (h,
        # then the block's output) for the norm that reads them next
        st_bytes = wan.wan_workspace_size(wan.WAN_OP_GN_STATS_WINOGRAD, *self.x5.shape, self.x5.shape[-1], GROUPS)
        self.st5 = [torch.empty(st_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        need = max(wan.wan_workspace_size(wan.WAN_OP_GN_SILU, *t.shape, 0, GROUPS)
                   for t in (self.gn_x, self.x4, self.x5))
        self.gn_ws = torch.empty(need, dtype=torch.uint8, device=dev)
        need_rb = max(wan.wan_workspace_size(wan.WAN_OP_RESBLOCK, *t.shape, t.shape[-1], GROUPS)
                      for t in (self.x4, self.x5))
        self.rb_ws = torch.empty(need_rb, dtype=torch.uint8, device=dev)

        # useful FLOPs / bytes of the parts in the step
        self.flops = {}
        if want("c256"):
            self.flops["c256"] = 6 * conv_flops(1, 4, 176, 312, 256, 256)
        if want("c1024"):
            self.flops["c1024"] = 4 * conv_flops(1, 4, 44, 78, 1024, 1024)
        if want("up"):
            self.flops["up"] = phase_flops(1, 4, 44, 78, 512, 512)
        if want("head"):
            self.flops["head"] = conv_flops(1, head_frames, 704, 1248, 256, 12)
        self.gn_bytes = 4.0 * self.gn_x.numel()

    # ---- one step as the sequence of C-ABI calls, each bracketed by events -----------------
    def step_calls(self):
        """[(tag, kernels launched, callable)] for one step."""
        from video_vae_decoder_gb300 import binding as wan
        want = (lambda part: self.case in ("all", part))
        calls = []
        if want("gn"):
            calls.append(("gn", 1, lambda: wan.wan_gn_silu(self.gn_x, self.gn_g, self.gn_b, GROUPS, EPS, self.gn_y,
                                                           self.gn_ws)))

        def stage(tag, x, blocks, caches, outs, coef, h, alt, us=None):
            # Each ResBlock as the calls wan_resblock (wan_resblock_winograd with `us`) makes, twice
            # (GroupNorm + SiLU into each conv): the norm's coefficients (one pass over its input),
            # then the conv normalising its operand tiles as they arrive (or its input as it is
            # transformed), which also writes the conv's new history: each conv has two history
            # buffers, reads one and writes the other, and they swap every step. On the Winograd
            # stage every norm after the first takes its coefficients from the statistics that the
            # conv which wrote its input emitted (the stage's first norm reads x with a pass).
            cur = x
            st = self.st5 if us is not None else None
            for i, (p, (c1, c2), out) in enumerate(zip(blocks, caches, outs)):
                h1 = [c1, alt[2 * i]]      # conv 1's history: [read, write]
                h2 = [c2, alt[2 * i + 1]]  # conv 2's
                chained_in = st is not None and i > 0          # cur's statistics from the previous block
                emit_out = st is not None and i + 1 < len(blocks)  # out's, for the next block

                def n1(cur=cur, p=p, chained_in=chained_in):
                    if chained_in:
                        wan.wan_gn_silu_coefficients_from_stats(st[1], p["gamma1"], p["beta1"], cur.shape, GROUPS, EPS,
                                                                coef)
                    else:
                        wan.wan_gn_silu_coefficients(cur, p["gamma1"], p["beta1"], GROUPS, EPS, coef, self.gn_ws)

                def k1(cur=cur, p=p, hb=h1, i=i):
                    if st is not None:
                        wan.wan_causal_conv3d_winograd_stats(cur, us[i][0], GROUPS, coef, p["b1"], None, hb[0], hb[1], h,
                                                             st[0], self.wino_ws)
                    elif us is not None:
                        wan.wan_causal_conv3d_winograd(cur, us[i][0], coef, p["b1"], None, hb[0], hb[1], h, self.wino_ws)
                    else:
                        wan.wan_causal_conv3d_gn_input(cur, coef, p["w1"], p["b1"], None, hb[0], h, cache_out=hb[1])
                    hb.reverse()

                def n2(p=p):
                    if st is not None:
                        wan.wan_gn_silu_coefficients_from_stats(st[0], p["gamma2"], p["beta2"], h.shape, GROUPS, EPS,
                                                                coef)
                    else:
                        wan.wan_gn_silu_coefficients(h, p["gamma2"], p["beta2"], GROUPS, EPS, coef, self.gn_ws)

                def k2(cur=cur, p=p, hb=h2, out=out, i=i, emit_out=emit_out):
                    if emit_out:
                        wan.wan_causal_conv3d_winograd_stats(h, us[i][1], GROUPS, coef, p["b2"], cur, hb[0], hb[1], out,
                                                             st[1], self.wino_ws)
                    elif us is not None:
                        wan.wan_causal_conv3d_winograd(h, us[i][1], coef, p["b2"], cur, hb[0], hb[1], out, self.wino_ws)
                    else:
                        wan.wan_causal_conv3d_gn_input(h, coef, p["w2"], p["b2"], cur, hb[0], out, cache_out=hb[1])
                    hb.reverse()
                kc = 3 if us is not None else 1  # Winograd: input transform, component GEMMs, output transform
                calls.extend([(f"{tag}.coefst" if chained_in else f"{tag}.coef", 1, n1), (f"{tag}.conv", kc, k1),
                              (f"{tag}.coefst" if st is not None else f"{tag}.coef", 1, n2), (f"{tag}.conv", kc, k2)])
                cur = out

        if want("c256"):
            stage("c256", self.x4, self.blocks4, self.c4, self.o4, self.k4, self.h4, self.alt4)
        if want("up"):
            calls.append(("up.weights", 1, lambda: wan.wan_upsample_phase_weights(self.w3, self.wp)))
            calls.append(("up.conv", 1, lambda: wan.wan_upsample_phase_conv(self.x3, self.wp, None, self.y3)))
        if want("c1024"):
            stage("c1024", self.x5, self.blocks5, self.c5, self.o5, self.k5, self.h5, self.alt5, self.u5)
        if want("head"):
            calls.append(("head.conv", 1, lambda: wan.wan_causal_conv3d(self.xh, self.wh, None, None, None, None,
                                                                        self.yh)))
        return calls

    # ---- the same step through the public calls a user makes (wan_resblock etc.) ------------
    def public_step(self, x2, x4, x3, x5, xh, wait=None):
        """The step as a user runs it. `wait(i)`, if given, is called before the first use of
        input i (x2, x4, x3, x5, xh in that order), e.g. to wait for its copy to arrive."""
        from video_vae_decoder_gb300 import binding as wan
        wait = wait or (lambda i: None)
        wait(0)
        wan.wan_gn_silu(x2, self.gn_g, self.gn_b, GROUPS, EPS, self.gn_y, self.gn_ws)
        wait(1)
        cur = x4
        for p, (c1, c2), out in zip(self.blocks4, self.c4, self.o4):
            wan.wan_resblock(cur, p, c1, c2, True, GROUPS, EPS, out, self.rb_ws)
            cur = out
        wan.wan_upsample_phase_weights(self.w3, self.wp)
        wait(2)
        wan.wan_upsample_phase_conv(x3, self.wp, None, self.y3)
        wait(3)
        cur = x5
        for p, (u1, u2), (c1, c2), out in zip(self.blocks5, self.u5, self.c5, self.o5):
            wan.wan_resblock_winograd(cur, p, u1, u2, c1, c2, True, GROUPS, EPS, out, self.rbw_ws)
            cur = out
        wait(4)
        wan.wan_causal_conv3d(xh, self.wh, None, None, None, None, self.yh)
        return (self.gn_y, self.o4[-1], self.y3, self.o5[-1], self.yh)


def max_over_ranks(x, world, device):
    """The largest of the ranks' values of x: the job takes as long as its slowest rank."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step, world, ms_per_step):
    """Whole-job throughput of `world` replicas that each run one step of the given FLOPs in
    ms_per_step (the slowest rank's time): every rank's work counts."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def time_adjacent(dev, reps=10):
    """The decoder steps next to the ResBlock, timed on their own (outside the step): the causal
    3x1x1 time upsample of the widest stage [1,4,44,78,1024] -> [1,8,44,78,1024] with history,
    a channel-changing ResBlock 512 -> 256 at [1,4,176,312,512] (1x1x1 shortcut, folded bias), and
    GroupNorm + SiLU applied on its own at the C=256 chunk size [1,4,176,312,256] (225 MB moved).
    CUDA events around each call, an L2 flush (256 MB written) before each, 3 warm-up calls."""
    import numpy as np
    import torch
    from video_vae_decoder_gb300 import binding as wan, synth
    bf = torch.bfloat16

    def n(shape, name, mean=0.0, std=1.0, dtype=bf):
        return synth.normal_torch(shape, 0, name, mean, std, device=dev, dtype=dtype)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return statistics.mean(ms)
    out = {}
    C = 1024
    x = n((1, 4, 44, 78, C), "bench/tup/x")
    w = n((2 * C, 3, C), "bench/tup/w", 0.0, float(np.sqrt(1.0 / (3 * C))))
    b = n((2 * C,), "bench/tup/b", 0.0, 0.01)
    cache = n((1, 2, 44, 78, C), "bench/tup/c")
    y = torch.empty((1, 8, 44, 78, C), dtype=bf, device=dev)
    ms = timed(lambda: wan.wan_time_upsample(x, w, b, False, cache, None, y))
    fl = 2.0 * 4 * 44 * 78 * 3 * C * 2 * C
    out["time_upsample_c1024"] = {"ms": ms, "tflops": fl / ms / 1e9, "shape": "[1,4,44,78,1024] -> [1,8,44,78,1024]"}
    del x, w, b, cache, y
    Cin, Cout = 512, 256
    x = n((1, 4, 176, 312, Cin), "bench/rbsc/x")
    p = {"gamma1": n((Cin,), "bench/rbsc/g1", 1.0, 0.1, torch.float32),
         "beta1": n((Cin,), "bench/rbsc/be1", 0.0, 0.1, torch.float32),
         "w1": n((Cout, 3, 3, 3, Cin), "bench/rbsc/w1", 0.0, float(np.sqrt(1.0 / (27 * Cin)))),
         "b1": n((Cout,), "bench/rbsc/b1", 0.0, 0.01),
         "gamma2": n((Cout,), "bench/rbsc/g2", 1.0, 0.1, torch.float32),
         "beta2": n((Cout,), "bench/rbsc/be2", 0.0, 0.1, torch.float32),
         "w2": n((Cout, 3, 3, 3, Cout), "bench/rbsc/w2", 0.0, float(np.sqrt(1.0 / (27 * Cout))))}
    p["b2"] = wan.wan_fold_bias(n((Cout,), "bench/rbsc/b2", 0.0, 0.01), n((Cout,), "bench/rbsc/bsc", 0.0, 0.01))
    w_sc = n((Cout, Cin), "bench/rbsc/wsc", 0.0, float(np.sqrt(1.0 / Cin)))
    c1 = torch.zeros((1, 2, 176, 312, Cin), dtype=bf, device=dev)
    c2 = torch.zeros((1, 2, 176, 312, Cout), dtype=bf, device=dev)
    o = torch.empty((1, 4, 176, 312, Cout), dtype=bf, device=dev)
    ws = torch.empty(wan.wan_workspace_size(wan.WAN_OP_RESBLOCK_SHORTCUT, 1, 4, 176, 312, Cin, Cout, GROUPS),
                     dtype=torch.uint8, device=dev)
    ms = timed(lambda: wan.wan_resblock_shortcut(x, p, w_sc, c1, c2, True, GROUPS, EPS, o, ws))
    px = 4 * 176 * 312
    fl = 2.0 * px * (27 * Cin * Cout + 27 * Cout * Cout + Cin * Cout)
    out["resblock_shortcut_512_to_256"] = {"ms": ms, "tflops": fl / ms / 1e9, "shape": "[1,4,176,312,512] -> 256"}
    del x, p, w_sc, c1, c2, o, ws
    C = 256
    x = n((1, 4, 176, 312, C), "bench/gn256/x", 0.5, float(np.sqrt(2.0)))
    g = n((C,), "bench/gn256/gamma", 1.0, 0.1, torch.float32)
    be = n((C,), "bench/gn256/beta", 0.0, 0.1, torch.float32)
    y = torch.empty_like(x)
    ws = torch.empty(wan.wan_workspace_size(wan.WAN_OP_GN_SILU, *x.shape, 0, GROUPS), dtype=torch.uint8, device=dev)
    ms = timed(lambda: wan.wan_gn_silu(x, g, be, GROUPS, EPS, y, ws))
    gbs = 4.0 * x.numel() / ms / 1e6
    out["gn_silu_c256_chunk"] = {"ms": ms, "gbs": gbs, "frac": gbs / peaks()["hbm_gbs"],
                                 "shape": "[1,4,176,312,256], 4 B per element (x read, y written)"}
    assert wan.wan_device_status() == 0
    return out


def timed_graph_steps(calls, steps, stream):
    """Capture two consecutive steps as two CUDA graphs and time `steps` steps replaying them in
    turn (CUDA events on the stream around the whole timed region)."""
    import torch
    try:
        graphs = []
        side = torch.cuda.Stream()  # capture runs on a stream of its own; replays go on `stream`
        side.wait_stream(stream)
        for _ in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _, _, fn in calls:
                    fn()
            graphs.append(g)
        stream.wait_stream(side)
        for k in range(4):  # warm-up replays
            graphs[k % 2].replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(steps):
            graphs[k % 2].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return {"ms_per_step": e0.elapsed_time(e1) / steps, "graphs": 2}
    except Exception as exc:  # capture refused: the eager timing stands
        torch.cuda.synchronize()
        return {"unavailable": str(exc).splitlines()[0][:200]}


def run_ours(args, rank, world, dev):
    import torch
    from video_vae_decoder_gb300 import binding as wan
    torch.cuda.set_device(dev)
    wl = Workload(dev, args.case, head_frames=args.head_frames)
    calls = wl.step_calls()
    stream = torch.cuda.current_stream()
    # warm-up (also fills the caches: the timed steps are steady-state chunks with history)
    for _ in range(max(args.warmup, 0)):
        for _, _, fn in calls:
            fn()
    torch.cuda.synchronize()
    assert wan.wan_device_status() == 0

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(args.steps):
        ev[s][0].record(stream)
        for i, (_, _, fn) in enumerate(calls):
            fn()
            ev[s][i + 1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    assert wan.wan_device_status() == 0
    # Optionally the same step replayed from CUDA graphs (one per direction of the histories' two
    # buffers, replayed alternately, so every timed step reads the history the step before wrote),
    # reported beside the eager step time.
    graph = timed_graph_steps(calls, args.steps, stream) if args.graph else None
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    assert wan.wan_device_status() == 0

    per_tag = {}
    step_ms = []
    for s in range(args.steps):
        step_ms.append(ev[s][0].elapsed_time(ev[s][-1]))
        for i, (tag, _, _) in enumerate(calls):
            per_tag.setdefault(tag, []).append(ev[s][i].elapsed_time(ev[s][i + 1]))
    ms_eager = statistics.mean(step_ms)
    ms = max_over_ranks(ms_eager, world, dev)
    flops = sum(wl.flops.values())
    pk = peaks()

    def tot(prefix):  # mean total ms per step of the calls with this tag
        return sum(statistics.mean(v) * (len(v) // args.steps) for k, v in per_tag.items() if k == prefix)

    def per_launch(prefix):
        v = per_tag.get(prefix, [])
        return statistics.mean(v) if v else 0.0

    # Every kernel here runs for well under a millisecond to a few milliseconds, and the timed region
    # lasts a fraction of a second: the burst bf16 figure (best of ten 8192^3 GEMMs) is the tensor
    # peak they are measured against; the fraction of the seconds-long sustained figure is given
    # beside it.
    pk_tf = pk["bf16_tflops"]
    kernels = {}
    shares = {}

    def tensor_kernel(name, ms_launch, flops_launch, total):
        tf = flops_launch / ms_launch / 1e9
        kernels[name] = {"ms": ms_launch, "tflops": tf, "total_ms": total, "bound": "tensor",
                         "frac": tf / pk_tf, "frac_of_sustained": tf / pk["bf16_tflops_sustained"]}
        shares[name] = total

    def hbm_kernel(name, ms_launch, bytes_launch, total):
        gbs = bytes_launch / ms_launch / 1e6
        kernels[name] = {"ms": ms_launch, "gbs": gbs, "total_ms": total, "bound": "hbm", "frac": gbs / pk["hbm_gbs"]}
        shares[name] = total

    if "c256.conv" in per_tag:
        tensor_kernel("conv_c256", per_launch("c256.conv"), conv_flops(1, 4, 176, 312, 256, 256), tot("c256.conv"))
        # the norm's coefficients: one read of its input (2 bytes per element); the cache frames:
        # 2 of the 4 frames read and written
        hbm_kernel("gn_coef_c256", per_launch("c256.coef"), 2.0 * wl.x4.numel(), tot("c256.coef"))
        kernels["resblock_c256_ms"] = (tot("c256.coef") + tot("c256.conv")) / 3.0
    if "c1024.conv" in per_tag:
        # Winograd F(2x2, 3x3): 16 component products of 3 temporal taps x Cin per 2x2 outputs, the
        # algorithm's tensor work (its three kernels timed together as one call); the direct
        # conv's count per call gives the equivalent rate.
        cm = per_launch("c1024.conv")
        tensor_kernel("conv_c1024_winograd", cm, wino_flops(1, 4, 44, 78, 1024, 1024), tot("c1024.conv"))
        kernels["conv_c1024_winograd"]["direct_equivalent_tflops"] = conv_flops(1, 4, 44, 78, 1024, 1024) / cm / 1e9
        hbm_kernel("gn_coef_c1024", per_launch("c1024.coef"), 2.0 * wl.x5.numel(), tot("c1024.coef"))
        # the later norms' coefficients from the statistics the Winograd convs emitted: one CTA per
        # (frame, group) reading its records (24 B each, one per 2x2 tile), bound by latency rather
        # than by a roofline, so it stays out of `rooflines`
        sm = per_launch("c1024.coefst")
        st_bytes = 24.0 * wl.x5.shape[0] * wl.x5.shape[1] * GROUPS * ((wl.x5.shape[2] + 1) // 2) * \
            ((wl.x5.shape[3] + 1) // 2)
        kernels["gn_coef_from_stats_c1024"] = {"ms": sm, "gbs": st_bytes / sm / 1e6 if sm else 0.0,
                                               "total_ms": tot("c1024.coefst"), "bound": "latency"}
        kernels["resblock_c1024_ms"] = (tot("c1024.coef") + tot("c1024.coefst") + tot("c1024.conv")) / 2.0
    if "head.conv" in per_tag:
        # Bound by whichever takes longer at the measured peaks: its useful MMAs or its HBM bytes.
        hm = per_launch("head.conv")
        hbytes = (wl.xh.numel() + wl.yh.numel()) * 2
        t_tensor = wl.flops["head"] / (pk_tf * 1e12)
        t_hbm = hbytes / (pk["hbm_gbs"] * 1e9)
        kernels["head_256_to_12"] = {
            "ms": hm, "tflops": wl.flops["head"] / hm / 1e9, "hbm_gbs_in_out": hbytes / hm / 1e6,
            "total_ms": hm, "bound": "tensor" if t_tensor >= t_hbm else "hbm",
            "frac": max(t_tensor, t_hbm) * 1e3 / hm, "frac_tensor": t_tensor * 1e3 / hm, "frac_hbm": t_hbm * 1e3 / hm}
        shares["head_256_to_12"] = hm
    if "up.conv" in per_tag:
        tensor_kernel("upsample_phase_conv", per_launch("up.conv"), wl.flops["up"], tot("up.conv"))
    if "gn" in per_tag:
        hbm_kernel("gn_silu_decode_mid", per_launch("gn"), wl.gn_bytes, tot("gn"))
    # DRAM bytes (read + write) per launch from `ncu --set full` captures of the current build of
    # each kernel (profiles/); the head's from a single-pass capture of the 16-frame launch; the
    # Winograd conv's is its three kernels' sum, averaged over the stage's four calls (three of
    # them writing statistics, two with the residual).
    traffic = {"conv_c256": 172.575744e6 + 125.743872e6, "gn_coef_c256": 112.540416e6 + 3.522304e6,
               "gn_coef_c1024": 28.202496e6, "conv_c1024_winograd": 161.323e6 + 447.922e6 + 243.859e6,
               "upsample_phase_conv": 22.554112e6 + 4.61184e6, "gn_silu_decode_mid": 68.827392e6 + 11.028992e6,
               "head_256_to_12": 9.9e9 + 0.343e9}
    rooflines = []
    for name, k in kernels.items():
        if not isinstance(k, dict) or "frac" not in k:
            continue
        tensor = k["bound"] == "tensor"
        achieved = k["tflops"] if tensor else (k["gbs"] if "gbs" in k else k["hbm_gbs_in_out"])
        peak = pk_tf if tensor else pk["hbm_gbs"]
        if name == "head_256_to_12":  # its fraction is ideal time / time, against its own bound
            achieved = peak * k["frac"]
        rooflines.append({"kernel": name, "bound": k["bound"], "achieved": achieved, "peak": peak,
                          "unit": "TFLOP/s" if tensor else "GB/s", "frac": k["frac"],
                          "traffic": traffic.get(name), "share_of_step": k["total_ms"] / ms_eager,
                          "peak_source": (f"{pk['source']} burst bf16 GEMM" if tensor else f"{pk['source']} HBM copy")})
    dom = max(shares, key=shares.get)
    roof = dict(next(r for r in rooflines if r["kernel"] == dom))
    if roof["bound"] == "tensor":
        roof["frac_of_sustained"] = roof["achieved"] / pk["bf16_tflops_sustained"]
    launches = sum(k for _, k, _ in calls) * args.steps

    out = {
        "metric": METRIC, "value": job_tflops(flops, world, ms), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded counter-based normals; random-init weights of the decoder shapes)",
        "config": {"workload": "decoder hot path, one steady-state 4-frame chunk: GN+SiLU [1,4,88,156,512]; "
                               "3 causal ResBlocks C=256 [1,4,176,312,256]; nearest-x2+3x3 upsample as 4 phase convs "
                               "[1,4,44,78,512]->[1,4,88,156,512]; 2 causal ResBlocks C=1024 [1,4,44,78,1024] (convs through "
                               "Winograd F(2x2,3x3), fp16 operands); head conv 256->12 [1,16,704,1248,256]",
                   "useful_tflop_per_step": flops / 1e12,
                   "flop_count": "direct-convolution FLOPs (2 M N K) for every conv, the Winograd ones included", "l2": "no flush: the step's working set (~8 GB) exceeds L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "kernels": kernels, "wall_s_timed": wall, "clocks": clocks, "gpu_launches": launches, "roofline": roof,
        "ms_per_step_eager": ms_eager, "cuda_graph": graph,
        "rooflines": rooflines,
    }
    if args.case == "all" and not args.no_adjacent:
        out["adjacent_steps"] = time_adjacent(dev)
    if not args.no_e2e and args.case == "all":
        out["e2e"] = run_e2e(args, wl, dev, flops)
    return out


def run_e2e(args, wl, dev, flops):
    """The same step through the public calls with HOST buffers, as a stream of chunks: every step
    copies its inputs in from pinned memory and its results out, all inside the timed region. The
    copies run on their own streams (inputs in the order the step needs them, device inputs
    double-buffered), so one step's compute overlaps the next step's input copies; the compute of
    a call waits for its input's copy event."""
    import torch
    ins = [wl.gn_x, wl.x4, wl.x3, wl.x5, wl.xh]
    host_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ins]
    for h, d in zip(host_in, ins):
        h.copy_(d)
    dev_in = [[torch.empty_like(t) for t in ins] for _ in range(2)]
    outs = wl.public_step(*dev_in[0])
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in ins] for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]  # compute of the step that used buffer b is done
    ev_out = torch.cuda.Event()                        # the previous step's results are on the host

    def step(k):
        b = k % 2
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_done[b])
            for i, (h, d) in enumerate(zip(host_in, dev_in[b])):
                d.copy_(h, non_blocking=True)
                ev_in[b][i].record(s_in)
        if k >= 1:
            main.wait_event(ev_out)  # results of step k-1 copied out before they are overwritten
        o = wl.public_step(*dev_in[b], wait=lambda i: main.wait_event(ev_in[b][i]))
        ev_done[b].record(main)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            for h, d in zip(host_out, o):
                h.copy_(d, non_blocking=True)
            ev_out.record(s_out)

    for k in range(max(1, args.warmup)):
        step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    steps = max(1, min(args.steps, 10))
    e0.record(s_in)
    for k in range(steps):
        step(k)
    e1.record(s_out)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "wan_gn_silu, wan_resblock x3, wan_resblock_winograd x2, wan_upsample_phase_weights, "
                   "wan_upsample_phase_conv, "
                   "wan_causal_conv3d from pinned host buffers; copies on their own streams, double-buffered "
                   "device inputs (host link measured at ~211 GB/s in, ~193 GB/s out)"}


# ------------------------------------------------------------------------------------------------
# the oracle on the host cores
# ------------------------------------------------------------------------------------------------
SAMPLE_SHAPE = (1, 4, 32, 312, 256)


def oracle_sample():
    import numpy as np
    import oracle
    from video_vae_decoder_gb300 import synth
    x = synth.normal_bf16(SAMPLE_SHAPE, 0, "bench/c256/x")
    p = synth.resblock_params(256, 0, "bench/cpu/block")
    flops = 2 * conv_flops(*SAMPLE_SHAPE, 256)

    def run():
        t = time.perf_counter()
        oracle.resblock(x, p, GROUPS, float(np.float32(EPS)))
        return time.perf_counter() - t
    return run, flops


def cpu_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(k)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count() or 1


ONE_THREAD_SHAPE = (1, 1, 8, 312, 256)  # one frame of 8 rows: the smallest unit of the sample


def one_thread_sample():
    """The oracle ResBlock on ONE_THREAD_SHAPE in this process (started with one BLAS thread)."""
    import numpy as np
    import oracle
    from video_vae_decoder_gb300 import synth
    x = synth.normal_bf16(ONE_THREAD_SHAPE, 0, "bench/c256/x1")
    p = synth.resblock_params(256, 0, "bench/cpu/block")
    flops = 2 * conv_flops(*ONE_THREAD_SHAPE, 256)
    t = time.perf_counter()
    oracle.resblock(x, p, GROUPS, float(np.float32(EPS)))
    s = time.perf_counter() - t
    return {"value": flops / s / 1e12, "unit": "TFLOP/s", "cores": 1,
            "sample": f"ResBlock on {list(ONE_THREAD_SHAPE)}, {flops / 1e9:.1f} GFLOP of conv work, {s:.2f} s"}


def one_thread_baseline():
    """one_thread_sample() in a fresh interpreter whose BLAS and OpenMP pools have one thread."""
    import subprocess
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--one-thread-sample"], env=env,
                       capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"unavailable": (r.stderr.strip().splitlines() or ["failed"])[-1][:200]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(reps=1):
    run, flops = oracle_sample()
    secs = [run() for _ in range(reps)]
    s = min(secs)
    return {"value": flops / s / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": f"fp64 numpy oracle ResBlock (GN+SiLU, 2 causal convs C=256) on {list(SAMPLE_SHAPE)}, "
                      f"{flops / 1e9:.0f} GFLOP of conv work, {s:.2f} s",
            "one_thread": one_thread_baseline()}


def run_reference(args):
    run, flops = oracle_sample()
    for _ in range(max(args.warmup, 0)):
        run()
    secs = [run() for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(secs)
    v = flops / (ms * 1e-3) / 1e12
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"fp64 CPU oracle: causal ResBlock C=256 on {list(SAMPLE_SHAPE)} "
                                   "(a bounded slice of the [1,4,176,312,256] chunk)"},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": f"ResBlock on {list(SAMPLE_SHAPE)} per step"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-adjacent", action="store_true", help="skip timing the steps next to the ResBlock")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step replayed from CUDA graphs (measured no faster: launches are not the limit)")
    ap.add_argument("--head-frames", type=int, default=16,
                    help="frames of the head's input (smaller values make a case small enough for ncu --set full)")
    ap.add_argument("--case", default="all", choices=CASES,
                    help="time one part of the step only (profiling captures); the default is the whole step")
    ap.add_argument("--adjacent-only", action="store_true",
                    help="time only the steps next to the ResBlock (profiling captures of those kernels); prints "
                         "their figures, not the step's line")
    ap.add_argument("--one-thread-sample", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.one_thread_sample:
        print(json.dumps(one_thread_sample()))
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)  # before the process group, so every rank's NCCL work uses its own GPU
    if world > 1:
        torch.distributed.init_process_group("nccl")
    from video_vae_decoder_gb300 import binding
    binding.lib()
    if args.adjacent_only:
        if rank == 0:
            torch.cuda.set_device(dev)
            print(json.dumps({"adjacent_steps": time_adjacent(dev)}), flush=True)
        return
    out = run_ours(args, rank, world, dev)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            out["cpu_baseline"] = cpu_baseline()
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
