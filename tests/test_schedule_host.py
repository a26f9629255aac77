"""Host logic of the attention work schedules (no GPU): a small C++ program
compiled from tests/native/schedule_check.cu against the kernels' own
work.cuh checks stream-K ranges, units, partial slots and the combine's cut
table, and split-KV shares, over many shapes (see the program's header)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    return None


def test_work_schedules(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = tmp_path / "schedule_check"
    src = os.path.join(ROOT, "tests", "native", "schedule_check.cu")
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-I" + os.path.join(ROOT, "include"), src, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == "OK", out.stdout + out.stderr
