"""Resuming a chunked decode in a fresh process: the temporal caches are the only state carried
between chunks, so chunk k+1 run in a new process from caches saved after chunk k gives the same
bits as running both chunks in one process.

Two child processes run a C=256 causal ResBlock (the norm applied in the CTA-pair conv's operand
prologue): the first runs chunk 0 from zero caches and saves the caches to files; the second,
started afresh, loads them and runs chunk 1 with cache_valid set. The test process runs both
chunks itself and compares outputs and caches bit for bit."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from util import to_dev, f32_dev, bits
from video_vae_decoder_gb300 import synth

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EPS = float(np.float32(1e-6))
SHAPE = (1, 4, 16, 32, 256)

CHILD = r"""
import sys
import numpy as np
import torch
root, stage, d = sys.argv[1], sys.argv[2], sys.argv[3]
sys.path.insert(0, root)
from video_vae_decoder_gb300 import binding as wan, synth
eps = float(np.float32(1e-6))

def to_dev(b):
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).cuda()

def save(name, t):
    np.save(f"{d}/{name}.npy", t.view(torch.int16).cpu().numpy().view(np.uint16))

x = synth.normal_bf16((1, 4, 16, 32, 256), 0, "resume/x")
p = synth.resblock_params(256, 0, "resume/block")
prm = {k: (torch.from_numpy(v).cuda() if v.dtype == np.float32 else to_dev(v)) for k, v in p.items()}
if stage == "first":
    c1 = torch.zeros((1, 2, 16, 32, 256), dtype=torch.bfloat16, device="cuda")
    c2 = torch.zeros_like(c1)
    out = wan.wan_resblock(to_dev(np.ascontiguousarray(x[:, :2])), prm, c1, c2, False, 32, eps)
else:
    c1 = to_dev(np.load(f"{d}/first_c1.npy"))
    c2 = to_dev(np.load(f"{d}/first_c2.npy"))
    out = wan.wan_resblock(to_dev(np.ascontiguousarray(x[:, 2:])), prm, c1, c2, True, 32, eps)
torch.cuda.synchronize()
assert wan.wan_device_status() == 0
save(stage + "_out", out)
save(stage + "_c1", c1)
save(stage + "_c2", c2)
"""


def _child(stage, d):
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, stage, str(d)], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, f"{stage} chunk process failed:\n{r.stderr[-3000:]}"


def test_resblock_chunk_resumed_in_a_fresh_process_is_bit_identical(wan, tmp_path):
    _child("first", tmp_path)
    _child("second", tmp_path)

    x = synth.normal_bf16(SHAPE, 0, "resume/x")
    p = synth.resblock_params(256, 0, "resume/block")
    prm = {k: (f32_dev(v) if v.dtype == np.float32 else to_dev(v)) for k, v in p.items()}
    c1 = torch.zeros((1, 2, 16, 32, 256), dtype=torch.bfloat16, device="cuda")
    c2 = torch.zeros_like(c1)
    outs, caches = [], []
    for i, s in enumerate((0, 2)):
        outs.append(wan.wan_resblock(to_dev(np.ascontiguousarray(x[:, s:s + 2])), prm, c1, c2, i > 0, 32, EPS))
        torch.cuda.synchronize()
        caches.append((bits(c1).copy(), bits(c2).copy()))
    assert wan.wan_device_status() == 0

    for i, stage in enumerate(("first", "second")):
        got = np.load(tmp_path / f"{stage}_out.npy")
        assert np.array_equal(got, bits(outs[i])), f"{stage} chunk output differs"
        assert np.array_equal(np.load(tmp_path / f"{stage}_c1.npy"), caches[i][0]), f"{stage} cache 1 differs"
        assert np.array_equal(np.load(tmp_path / f"{stage}_c2.npy"), caches[i][1]), f"{stage} cache 2 differs"
    # The resumed chunk saw history: its output is not the one zero caches give.
    fresh = wan.wan_resblock(to_dev(np.ascontiguousarray(x[:, 2:])), prm, torch.zeros_like(c1), torch.zeros_like(c2),
                             False, 32, EPS)
    torch.cuda.synchronize()
    assert not np.array_equal(bits(fresh), bits(outs[1]))
