"""Launch planning on the host (no GPU): compiles tests/host/launch_plans.cu
against the built library and runs it.  It checks the decode kernel's
shared-memory plan and phase-B work split over model shapes and SM counts,
the packed W_kvb layout and its bank swizzle, and the W8A8 workspace carve
(see that file's header for the list)."""
import os
import shutil
import subprocess

import pytest

from mla_attention_kv_gb300 import build as BLD

HERE = os.path.dirname(os.path.abspath(__file__))


def test_launch_plans(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    lib = BLD.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "launch_plans")
    cmd = [nvcc, "-std=c++17", "-O1", "-o", exe, os.path.join(HERE, "host", "launch_plans.cu"),
           "-L" + libdir, "-lmla_prolog", "-Xlinker", "-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert r.stdout.strip().endswith("0 failed checks")
