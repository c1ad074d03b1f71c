"""Host-side checks of the prefill work-unit plan and the key-split plans.

tests/unit_plan_check.cu includes the kernel sources and checks, on the CPU,
that the work units of a launch cover every (batch, head, 128-row block) tile
exactly once in both unit orders, that a causal unit's K/V tile count is the
brute-force count up to its diagonal, and that the tail-split and decode split
plans are sound.  It is compiled with nvcc (no GPU needed) and run here.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_unit_plan(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    exe = os.path.join(str(tmp_path), "unit_plan_check")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O1", "-std=c++17", "--expt-relaxed-constexpr",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "exact_attention_forward_06_gb300", "csrc"),
           os.path.join(ROOT, "tests", "unit_plan_check.cu"), "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-2000:]
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout[-2000:]
    assert "all checks passed" in run.stdout
