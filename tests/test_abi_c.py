"""The header compiles as C (C99, gcc) and a C program links against the library and calls
it: the boundary is usable without C++ or Python."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c_program_links_and_calls_the_library(tmp_path):
    from long_context_grpo_gb300 import build
    lib = build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "abi_c_check"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic",
                        os.path.join(HERE, "cpp", "abi_c_check.c"), "-o", str(exe),
                        lib, "-Wl,-rpath," + os.path.dirname(lib)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.startswith("OK"), (out.returncode, out.stdout, out.stderr)
