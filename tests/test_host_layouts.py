"""Workspace layouts of the library checked on the host over the supported
shapes (tests/host_layout_check.cc, built with the host C++ compiler against
the library's own headers; no GPU and no CUDA library needed at run time)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "int4_grouped_gemm_gb300", "csrc")


def _cuda_include():
    for base in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if base and os.path.exists(os.path.join(base, "include", "cuda_bf16.h")):
            return os.path.join(base, "include")
    nvcc = shutil.which("nvcc")
    if nvcc:
        inc = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include")
        if os.path.exists(os.path.join(inc, "cuda_bf16.h")):
            return inc
    return None


def test_workspace_layouts(tmp_path):
    inc = _cuda_include()
    cxx = shutil.which("g++") or shutil.which("c++")
    if inc is None or cxx is None:
        pytest.skip("no host C++ compiler or CUDA headers")
    exe = tmp_path / "layout_check"
    subprocess.check_call([cxx, "-std=c++17", "-O1", "-I" + CSRC, "-I" + inc,
                           os.path.join(ROOT, "tests", "host_layout_check.cc"), "-o", str(exe)])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
