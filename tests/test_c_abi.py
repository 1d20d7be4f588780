"""The C ABI used from a plain C program (gcc, -std=c11, no C++ and no torch).

Needs no GPU: every call in the program is answered on the host.
"""
import os
import subprocess

import pytest

import mixture_experts_layer_06_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_boundary_from_plain_c(tmp_path):
    lib = moe.library_path()
    if not os.path.exists(lib):
        pytest.skip("the CUDA library has not been built")
    exe = tmp_path / "abi_from_c"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "abi_from_c.c"), "-o", str(exe),
                    "-L", os.path.dirname(lib), "-lmoe_gb300", "-Wl,-rpath," + os.path.dirname(lib)],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"
