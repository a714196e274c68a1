"""Helpers for the GPU tests: build/load the library, move the generator's
numpy inputs to the device, and compare a device result with the oracle."""

import numpy as np
import pytest

import oracle
from transformer_linear_layer_tcgen05_gb300 import build, lin
from transformer_linear_layer_tcgen05_gb300 import workloads as wl

# Spec acceptance bound on the normalised error.
TOL = 4e-3


def require_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    build.build_library()
    lin.lib()


def to_device(d: dict) -> dict:
    import torch
    out = {}
    for k, v in d.items():
        if v.dtype == np.uint16:
            out[k] = torch.from_numpy(v.view(np.int16)).cuda()
        else:
            out[k] = torch.from_numpy(v).cuda()
    return out


def run_device(form: str, d_dev: dict, M: int, N: int):
    import torch
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    lin.run_form(form, d_dev, Y)
    torch.cuda.synchronize()
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    return Y


def oracle_error(form: str, d: dict, Y: np.ndarray, rows=None) -> float:
    Yref, S = oracle.reference(form, d, rows=rows)
    R = None
    if "R" in d:
        R = d["R"] if rows is None else d["R"][rows]
    return oracle.normalised_error(Y, Yref, S, R)


def integer_inputs(form: str, M: int, N: int, K: int, seed: int) -> dict:
    """Small-integer inputs for which every product, partial sum and operand
    rounding of the GPU path is exact: |X|, |UP|, |W| <= 4 and GATE in
    [40, 60], so sigma(GATE) is 1.0 in float32 and float64 alike, every A
    value is an integer of magnitude <= 240 (exact in binary16) and every
    partial sum is an integer below K * 960 < 2**24 for K <= 16384."""
    rng = np.random.default_rng(seed)
    d = {}
    if wl.form_is_at(form):   # dW[K,N] = X[M,K]^T @ dY[M,N] (+ R [K,N])
        if wl.form_is_swiglu(form):
            d["GATE"] = rng.integers(40, 61, size=(M, K)).astype(np.float32)
            d["UP"] = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
        else:
            d["X"] = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
        d["DY"] = rng.integers(-4, 5, size=(M, N)).astype(np.float32)
        if wl.form_has_residual(form):
            d["R"] = rng.integers(-64, 65, size=(K, N)).astype(np.float32)
        return d
    if wl.form_is_t(form):   # dX[M,K] = dY[M,N] @ W[K,N]^T (+ R [M,K])
        d["DY"] = rng.integers(-4, 5, size=(M, N)).astype(np.float32)
        w = rng.integers(-4, 5, size=(K, N)).astype(np.float32)
        if wl.form_is_w16(form):
            d["W16"] = w.astype(np.float16).view(np.uint16)
        else:
            d["W"] = w
        if wl.form_has_residual(form):
            d["R"] = rng.integers(-64, 65, size=(M, K)).astype(np.float32)
        if wl.form_is_swiglu_bwd(form):   # sigma(GATE) == 1.0: every gradient an integer
            d["GATE"] = rng.integers(40, 61, size=(M, K)).astype(np.float32)
            d["UP"] = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
        return d
    if wl.form_is_swiglu(form):
        d["GATE"] = rng.integers(40, 61, size=(M, K)).astype(np.float32)
        d["UP"] = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    else:
        d["X"] = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    w = rng.integers(-4, 5, size=(K, N)).astype(np.float32)
    if wl.form_is_w16(form):
        d["W16"] = w.astype(np.float16).view(np.uint16)
    else:
        d["W"] = w
    if wl.form_has_residual(form):
        d["R"] = rng.integers(-64, 65, size=(M, N)).astype(np.float32)
    return d
