"""The C-ABI library builds, loads and exports every symbol of include/lin.h
(CPU only: no compute call is made).

The host-side validation of the library rejects bad dims, shapes, alignment
and aliasing before it touches CUDA, so those paths are exercised here too
with fake, never-dereferenced addresses.
"""

import os
import re

import pytest

from transformer_linear_layer_tcgen05_gb300 import build, lin

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "lin.h")


@pytest.fixture(scope="module")
def L():
    build.build_library()
    return lin.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lin_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_family():
    names = declared_functions()
    for form in ("matmul", "matmul_residual", "matmul_residual_swiglu_a"):
        assert f"lin_{form}" in names and f"lin_{form}_w16" in names
    assert {"lin_status_string", "lin_get_device_status", "lin_last_cuda_error",
            "lin_selftest_wait_timeout", "lin_version", "lin_last_launch_info"} <= set(names)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_checked_build_exports_the_same_symbols():
    # the checked build (device checks on) is the same ABI in another file
    import ctypes
    path = build.build_library(checked=True)
    assert path.endswith("liblin_checked.so") and path != build.LIB_PATH
    C = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(C, name), name
    C.lin_status_string.restype = ctypes.c_char_p
    assert C.lin_status_string(8) == b"LIN_ERROR_DEVICE_CHECK"


def test_binding_covers_every_compute_entry_point():
    for name in declared_functions():
        if name.startswith("lin_matmul"):
            assert name in lin.SIGNATURES
            assert hasattr(lin, name)
            if name.endswith("_host"):   # a forward form on host operands
                assert name[len("lin_"):-len("_host")] in lin.HOST_FORM_FUNCS
                continue
            # a _noalloc variant is its base form with a fixed workspace
            assert name[len("lin_"):].removesuffix("_noalloc") in lin.FORM_FUNCS
        if name.startswith(("lin_lm_head", "lin_gate_up")):
            assert name in lin.SIGNATURES and name[len("lin_"):] in lin.OTHER_FUNCS


def test_noalloc_validates_before_touching_cuda(L):
    # rejected like the base entry point, without any CUDA call
    fake = 1 << 40
    f = L.lin_matmul_residual_swiglu_a_w16_noalloc
    assert f(fake, fake, fake, fake, fake, -1, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE
    assert f(fake, fake, fake, fake, fake, 8, 12, 8, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE
    assert f(fake, fake, fake, fake, fake, 0, 8, 8, None) == lin.LIN_SUCCESS
    assert lin.lin_last_launch_info() == (0, 0)


def test_launch_info_after_rejected_and_empty_calls(L):
    # a call rejected by validation, or one with nothing to do, launches
    # nothing and takes no workspace
    fake = 1 << 40
    assert L.lin_matmul_w16(fake, fake, fake, -1, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE
    assert lin.lin_last_launch_info() == (0, 0)
    assert L.lin_matmul_w16(fake, fake, fake, 0, 8, 8, None) == lin.LIN_SUCCESS
    assert lin.lin_last_launch_info() == (0, 0)


def test_status_strings(L):
    for code, name in lin.STATUS.items():
        assert lin.status_string(code) == name
    assert lin.status_string(99) == "LIN_ERROR_UNKNOWN"
    assert L.lin_version() >= 100


# Fake device addresses: validation rejects these calls before any CUDA call.
X, W, R, Y, G, U = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000, 0x60000000


def test_negative_dims_and_null_pointers(L):
    assert L.lin_matmul(X, W, Y, -1, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul(X, W, Y, 8, 8, -4, None) == lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul(X, W, None, 8, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul(None, W, Y, 8, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul_residual(X, W, None, Y, 8, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul_residual_swiglu_a(G, None, W, R, Y, 8, 8, 8, None) == \
        lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul_residual_swiglu_a_w16(None, U, W, R, Y, 8, 8, 8, None) == \
        lin.LIN_ERROR_INVALID_VALUE


def test_empty_problems_are_noops(L):
    assert L.lin_matmul(None, None, None, 0, 8, 8, None) == lin.LIN_SUCCESS
    assert L.lin_matmul_residual_w16(None, None, None, None, 8, 0, 8, None) == lin.LIN_SUCCESS


def test_shape_rules(L):
    assert L.lin_matmul(X, W, Y, 8, 8, 6, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE   # K % 4
    assert L.lin_matmul(X, W, Y, 8, 6, 8, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE   # N % 4
    assert L.lin_matmul_w16(X, W, Y, 8, 12, 8, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE  # N % 8
    assert L.lin_matmul(X, W, Y, 2**31, 8, 8, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE


def test_alignment_rule(L):
    assert L.lin_matmul(X + 4, W, Y, 8, 8, 8, None) == lin.LIN_ERROR_MISALIGNED
    assert L.lin_matmul_residual(X, W, R + 8, Y, 8, 8, 8, None) == lin.LIN_ERROR_MISALIGNED
    assert L.lin_matmul_w16(X, W + 2, Y, 8, 8, 8, None) == lin.LIN_ERROR_MISALIGNED


def test_aliasing_rule(L):
    # in-place residual
    assert L.lin_matmul_residual(X, W, Y, Y, 8, 8, 8, None) == lin.LIN_ERROR_ALIASING
    # Y overlapping the tail of X: X is 8x8 f32 = 256 bytes
    assert L.lin_matmul(X, W, X + 240, 8, 8, 8, None) == lin.LIN_ERROR_ALIASING
    assert L.lin_matmul_residual_swiglu_a(G, U, W, R, U + 16, 8, 8, 8, None) == \
        lin.LIN_ERROR_ALIASING
    # adjacent but disjoint is not aliasing (it fails later, at the device check)
    assert L.lin_matmul(X, W, X + 256, 8, 8, 8, None) != lin.LIN_ERROR_ALIASING


def test_host_forms_validate_before_touching_cuda(L):
    # the device forms' dims, pointer, shape and aliasing rules, checked
    # before the operands' memory type is looked up (no CUDA call)
    assert L.lin_matmul_host(X, W, Y, -1, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul_host(X, W, None, 8, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul_residual_host(X, W, None, Y, 8, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul_residual_swiglu_a_w16_host(G, None, W, R, Y, 8, 8, 8, None) == \
        lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul_host(X, W, Y, 8, 8, 6, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE
    assert L.lin_matmul_w16_host(X, W, Y, 8, 12, 8, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE
    assert L.lin_matmul_residual_host(X, W, Y, Y, 8, 8, 8, None) == lin.LIN_ERROR_ALIASING
    assert L.lin_matmul_host(X, W, X + 240, 8, 8, 8, None) == lin.LIN_ERROR_ALIASING
    assert L.lin_matmul_residual_swiglu_a_host(G, U, W, R, U + 16, 8, 8, 8, None) == \
        lin.LIN_ERROR_ALIASING
    assert L.lin_matmul_host(None, None, None, 0, 8, 8, None) == lin.LIN_SUCCESS
    assert lin.lin_last_launch_info() == (0, 0)
    assert L.lin_set_host_block_bytes(100) == lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_set_host_block_bytes(0) == lin.LIN_SUCCESS


def test_transposed_forms_validate_before_touching_cuda(L):
    # dX[M,K] = dY[M,N] @ W[K,N]^T: N is the contraction, K the output width
    fake = 1 << 40
    assert L.lin_matmul_t(fake, fake, fake, -1, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE
    assert L.lin_matmul_t(fake, fake, fake, 8, 8, 6, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE
    assert L.lin_matmul_t(fake, fake, fake, 8, 6, 8, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE
    # binary16 W [K,N]: its rows (N elements) must be whole 16-byte units
    assert L.lin_matmul_t_w16(fake, fake, fake, 8, 12, 8, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE
    assert L.lin_matmul_t_w16(fake, fake, fake, 0, 16, 8, None) == lin.LIN_SUCCESS
    assert lin.lin_last_launch_info() == (0, 0)
    # dX may not overlap dY or W ...
    assert L.lin_matmul_t(X, W, X, 8, 8, 8, None) == lin.LIN_ERROR_ALIASING
    assert L.lin_matmul_t_acc(X, W, W, 8, 8, 8, None) == lin.LIN_ERROR_ALIASING
    # ... but the accumulating forms read and write dX itself (rejected here
    # only later, because the fake addresses are not device memory)
    assert L.lin_matmul_t_acc(X, W, Y, 8, 8, 8, None) != lin.LIN_ERROR_ALIASING
    assert L.lin_matmul_t_acc(None, W, Y, 8, 8, 8, None) == lin.LIN_ERROR_INVALID_VALUE


def test_lm_head_cross_entropy_validates_before_touching_cuda(L):
    import ctypes
    fake = 1 << 40
    f = L.lin_lm_head_cross_entropy_w16
    a, b, c = ctypes.c_float(0.0), ctypes.c_float(0.0), ctypes.c_float(1.0)
    assert f(fake, fake, fake, fake, fake, None, 8, 8, 8, a, b, c, None) == lin.LIN_ERROR_INVALID_VALUE
    assert f(fake, fake, fake, fake, fake, fake, -1, 8, 8, a, b, c, None) == lin.LIN_ERROR_INVALID_VALUE
    assert f(fake, fake, fake, fake, fake, fake, 8, 12, 8, a, b, c, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE
    assert f(fake, fake, fake, fake, fake, fake, 8, 16, 6, a, b, c, None) == lin.LIN_ERROR_UNSUPPORTED_SHAPE
    assert f(fake + 2, fake, fake, fake, fake, fake, 8, 16, 8, a, b, c, None) == lin.LIN_ERROR_MISALIGNED
    # dLogits over X
    assert f(fake, fake + (1 << 30), fake + (2 << 30), fake, fake + (3 << 30), fake + (4 << 30),
             8, 16, 8, a, b, c, None) == lin.LIN_ERROR_ALIASING


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    # no fallback: with liblin.so missing every call raises before any work,
    # and the package never imports the oracle
    import subprocess
    import sys
    monkeypatch.setattr(lin, "LIB_PATH", str(tmp_path / "liblin.so"))
    monkeypatch.setattr(lin, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        lin.lib()
    with pytest.raises(RuntimeError, match="not built"):
        lin.lin_last_launch_info()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import sys; import transformer_linear_layer_tcgen05_gb300.lin, "
            "transformer_linear_layer_tcgen05_gb300.build, "
            "transformer_linear_layer_tcgen05_gb300.workloads; "
            "sys.exit(1 if any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules) else 0)")
    assert subprocess.run([sys.executable, "-c", code], cwd=root).returncode == 0


def test_binding_checks_tensors_before_calling(L):
    # the tensor layer rejects wrong devices, dtypes and shapes itself (no
    # library call is made)
    import torch
    X = torch.zeros((8, 8))
    W = torch.zeros((8, 8))
    with pytest.raises(TypeError):
        lin.lin_matmul(X, W, X.clone())                  # CPU tensors for a device form
    with pytest.raises(ValueError):
        lin.lin_matmul_host(X, torch.zeros((4, 8)), torch.zeros((8, 8)))   # K mismatch
    with pytest.raises(TypeError):
        lin.lin_matmul_w16_host(X, W, torch.zeros((8, 8)))                 # f32 as W16
    with pytest.raises(ValueError):
        lin.lin_matmul_residual_host(X, W, torch.zeros((8, 4)), torch.zeros((8, 8)))  # R shape
    with pytest.raises(ValueError):
        lin.lin_matmul_host(X.t(), W, torch.zeros((8, 8)))                 # not contiguous
