"""The library used from plain C: tests/c_abi_check.c includes only
include/attn.h and the CUDA runtime header, links libattn.so, and checks a
causal GQA prefill and a paged decode step, each against a double-precision
host reference of its own written from the definition.  On CPU the program
must compile and link; on a GPU it must run and exit 0."""
import os
import shutil
import subprocess

import pytest

from exact_attention_forward_06_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "tests", "c_abi_check.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    if not os.path.exists(_binding.LIBRARY_PATH):
        import __graft_entry__
        __graft_entry__.build()
    lib_dir = os.path.dirname(_binding.LIBRARY_PATH)
    exe = os.path.join(str(out_dir), "c_abi_check")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", SOURCE, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), "-L", lib_dir, "-lattn", "-L", os.path.join(CUDA, "lib64"),
           "-lcudart", "-lm", f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.access(_compile(tmp_path), os.X_OK)


@pytest.mark.gpu
def test_c_program_runs_prefill_and_decode(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    res = subprocess.run([_compile(tmp_path)], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "prefill: 0 of" in res.stdout and "decode: 0 of" in res.stdout, res.stdout
