"""The host-side tile schedule, checked without a GPU: a small C++ program includes the
library's host source and verifies the schedule's invariants (coverage of every tile's K
range exactly once and in order, split-tile bookkeeping, balance across CTAs)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "block_scaled_fp4_persistent_gb300", "csrc")


def test_schedule_invariants(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "schedule_check")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                    os.path.join(HERE, "cpp", "schedule_check.cu"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
