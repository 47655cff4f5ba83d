"""Host build and run of tests/cpp/varlen_check.cpp: the packed-response index math the
kernels share (varlen_build, varlen_find) on random response lengths and tile sizes."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_varlen_index_math(tmp_path):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = tmp_path / "varlen_check"
    r = subprocess.run([nvcc, "-x", "c++", "-std=c++17", "-O1", os.path.join(HERE, "cpp", "varlen_check.cpp"),
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == "OK", out.stdout + out.stderr
