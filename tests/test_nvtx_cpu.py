"""Every entry point that enqueues work opens an NVTX range named after itself for the whole call.

A child process loads libwan.so with an NVTX injection library (tests/nvtx_recorder.c, built here
with the host compiler) that records each range push and pop, then calls every entry point with
NULL pointers and zero sizes: each one validates its arguments, returns an error status and
launches nothing, so no GPU is needed, and its range must still open and close once."""
import os
import shutil
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HOST_QUERIES = {"wan_status_string", "wan_workspace_size"}  # no launches, no range


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        inc = os.path.join(d, "include")
        if d and os.path.exists(os.path.join(inc, "nvtx3", "nvToolsExt.h")):
            return inc
    return None


def test_every_entry_point_opens_one_range_named_after_it(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    inc = _cuda_include()
    if not cc or not inc:
        pytest.skip("needs a C compiler and the NVTX headers")
    from video_vae_decoder_gb300 import binding, build
    build.build()
    so = tmp_path / "librecorder.so"
    subprocess.run([cc, "-shared", "-fPIC", "-O1", "-I", inc, os.path.join(ROOT, "tests", "nvtx_recorder.c"),
                    "-o", str(so)], check=True, capture_output=True, text=True)
    log = tmp_path / "ranges.log"
    script = textwrap.dedent("""
        import ctypes, json, sys
        sys.path.insert(0, sys.argv[1])
        from video_vae_decoder_gb300 import binding
        L = binding.lib()
        out = {}
        for name in binding.EXPORTS:
            if name in ("wan_status_string", "wan_workspace_size"):
                continue
            f = getattr(L, name)
            args = []
            for t in f.argtypes:  # numbers as zero, every pointer (data, stream, params) NULL
                scalar = issubclass(t, ctypes._SimpleCData) and t not in (ctypes.c_void_p, ctypes.c_char_p)
                args.append(t(0) if scalar else None)
            out[name] = int(f(*args))
        print(json.dumps(out))
    """)
    env = dict(os.environ, NVTX_INJECTION64_PATH=str(so), WAN_NVTX_LOG=str(log))
    r = subprocess.run([sys.executable, "-c", script, ROOT], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    status = json.loads(r.stdout.strip().splitlines()[-1])
    called = [n for n in binding.EXPORTS if n not in HOST_QUERIES]
    assert set(status) == set(called)
    assert all(s != 0 for s in status.values()), status  # every call refused its NULL arguments
    events = log.read_text().splitlines()
    # The log holds, per call in order, "push <its name>" ... "pop", with nothing left open.
    depth = 0
    outer = []
    for e in events:
        if e.startswith("push "):
            if depth == 0:
                outer.append(e[5:])
            depth += 1
        else:
            assert e == "pop" and depth > 0, events
            depth -= 1
    assert depth == 0
    assert outer == called
