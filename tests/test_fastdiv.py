"""The kernels divide by launch constants (query tiles per head, heads, the grid,
shard rows and heads of the output layout) with a multiply-high and a shift
(FastDiv in csrc/kernels.h).  This compiles a host program against that header
and checks the result against the division operator for divisors 1 .. 1200, the
workloads' sizes and values near 2^20, 2^30 and 2^31, on edge and pseudo-random
dividends below 2^31 (the kernels' dividends are ints)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "dit_attention_ulysses_gb300", "csrc")


def _cuda_include():
    nvcc = shutil.which("nvcc")
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc))) if nvcc else "/usr/local/cuda"
    return os.path.join(root, "include")


def test_fastdiv_matches_division(tmp_path):
    cxx = shutil.which("g++")
    inc = _cuda_include()
    if cxx is None or not os.path.exists(os.path.join(inc, "cuda_runtime.h")):
        pytest.skip("needs g++ and the CUDA headers")
    exe = str(tmp_path / "fastdiv_check")
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, "-I", inc, os.path.join(HERE, "fastdiv_check.cpp"),
                    "-o", exe], check=True, capture_output=True, text=True)
    r = subprocess.run([exe, "152", "148", "132", "960", "23680"], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0" in r.stdout
