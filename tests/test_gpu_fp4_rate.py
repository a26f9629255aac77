"""GPU: the rate of the block-scaled FP4 MMA (tests/native/fp4_mma_rate.cu):
M128 N128 K64 (the attention kernel's S-MMA shape) and M128 N256 K64 (the
widest single-CTA shape), operands resident in shared memory, no TMA -- the
dense NVFP4 peak the bench's FP4 roofline takes (FLOP per clock per SM times
the SM count and the maximum SM clock).  Checks that the probe runs,
completes its waits, and reports a plausible rate; prints the figures (run
with -s to see them)."""

import os
import re
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fp4_mma_rate(tmp_path):
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = tmp_path / "fp4_mma_rate"
    src = os.path.join(ROOT, "tests", "native", "fp4_mma_rate.cu")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", src, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    print(out.stdout)
    assert out.returncode == 0 and out.stdout.strip().endswith("ok"), out.stdout + out.stderr
    rates = [float(m) for m in re.findall(r"([0-9.]+) TFLOP/s", out.stdout)]
    errs = [int(m) for m in re.findall(r"err (\d+)", out.stdout)]
    assert rates and all(e == 0 for e in errs)
    assert max(rates) > 2000.0, rates          # far below any working tensor pipe
    per_clk = [float(m) for m in re.findall(r"([0-9]+) FLOP/clk/SM", out.stdout)]
    assert max(per_clk) <= 1.05 * 32768, per_clk   # the figure the bench's FP4 roofline is built on
