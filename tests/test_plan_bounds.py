"""Host-only check of the decode kernels' index arithmetic (no GPU).

tests/plan_check/plan_check.cu compiles the library's planning unit into a
host program that replays, for every launch plan over a grid of shapes, token
counts, formats and call forms, the kernel's row ranges, bulk-copy sizes and
destinations, consumed units, activation offsets and staging writes, checking
each against the buffer it addresses (and that calls too large for shared
memory split into token subsets that fit).  Every new launch shape was checked
this way before it first ran on a GPU.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _nvcc():
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


def test_every_launch_plan_stays_in_bounds(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "plan_check")
    src = os.path.join(HERE, "plan_check")
    r = subprocess.run([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a", "-o", exe,
                        os.path.join(src, "plan_check.cu"), os.path.join(src, "stubs.cu")],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:]
    assert " 0 failures" in r.stdout and "checked" in r.stdout, r.stdout
