"""libred.so from plain C: tests/c/red_c_client.c includes only red.h and
the CUDA runtime API, owns its buffers and stream, and checks closed-form
results (no Python, no torch on that path)."""
import os
import subprocess

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu

CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
PKG = os.path.join(ROOT, "int_tensor_reductions_gb300")


def test_c_client(tmp_path):
    from int_tensor_reductions_gb300 import _build
    _build.build_lib()
    exe = tmp_path / "red_c_client"
    subprocess.run(["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-I" + os.path.join(ROOT, "include"),
                    "-I" + os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c", "red_c_client.c"),
                    "-o", str(exe), "-L" + PKG, "-lred", "-Wl,-rpath," + PKG,
                    "-L" + os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA, "lib64")],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
