"""The C ABI from a plain C program (gcc, include/ts.h, libts.so): no Python
or torch types cross the boundary.  Host-only calls, so it runs without a GPU."""
import os
import subprocess

import pytest

from long_context_attention_tree_b300 import build as ts_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_uses_the_abi(tmp_path):
    lib = ts_build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "c_abi_check")
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c_abi_check.c"), "-L", libdir, "-l:libts.so",
                           "-Wl,-rpath," + libdir, "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "FAIL" not in r.stdout and r.stdout.count("ok ") >= 9
