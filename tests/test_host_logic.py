"""The scheduling logic the host and the kernels share (lin_internal.h: the
clustered kernels' banded tile order, the split plan of a persistent launch),
compiled for the CPU with the host C++ compiler and checked there
(tests/host_logic_check.cpp). No GPU."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_include():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda.h")):
            return os.path.join(cand, "include")
    return None


def test_tile_order_and_split_plan(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    inc = _cuda_include()
    if not cxx or not inc:
        pytest.skip("needs a host C++ compiler and the CUDA headers")
    exe = tmp_path / "host_logic_check"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "transformer_linear_layer_tcgen05_gb300", "csrc"),
                    "-I", inc, os.path.join(ROOT, "tests", "host_logic_check.cpp"),
                    "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], stdout=subprocess.PIPE, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout
