"""The library's C ABI from a plain C program: tests/c_abi/check_abi.c includes include/moe.h,
is compiled with gcc and linked against the built library, and checks sizes, status strings
and host-side argument errors (no GPU needed)."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

from sparse_moe_ffn_router_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_caller(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    binding.load_library()  # builds the library when it is missing
    lib = binding.library_path()
    exe = tmp_path / "check_abi"
    subprocess.run(["gcc", "-std=c11", "-O1", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "check_abi.c"), lib,
                    f"-Wl,-rpath,{os.path.dirname(lib)}", "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C ABI checks passed" in r.stdout
