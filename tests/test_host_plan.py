"""Host logic of sa_attn_fwd_host's chunking (no GPU): a small C++ program
compiled from tests/native/host_plan_check.cc against the library's own
host_plan.h checks the chunk plans over many shapes, SM counts and chunk
requests (see the program's header)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_host_pipeline_chunk_plans(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "host_plan_check"
    src = os.path.join(ROOT, "tests", "native", "host_plan_check.cc")
    r = subprocess.run([cxx, "-std=c++17", "-O1", src, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == "OK", out.stdout + out.stderr
