"""Seeded synthetic inputs for the forward linear-layer family.

This module draws random inputs and nothing else: it holds none of the
method's arithmetic (no product, no activation, no residual). Both the CUDA
path (through the tests and ``bench.py``) and the fp64 oracle consume what it
returns, so it is the one piece the two sides share.

The five named workloads are the transformer shapes of the
"03_linear_forward" page ("Ne Yapar?": seq_len M = 512, d_model 768, FFN
width 3072, lm_head 16384) plus one scaled-up SwiGLU down projection.
Distributions use N(mean, variance) notation: W ~ N(0, 1/768) has standard
deviation sqrt(1/768) (a Xavier-style variance), GATE ~ N(0, 4) has standard
deviation 2.

Generator: numpy ``Generator(PCG64(seed))``, seed = 1000 + workload index,
arrays drawn in the order GATE-or-X, UP, W, R; float32 draws come from
``standard_normal(dtype=float32)`` scaled by the standard deviation in
float32. Binary16 weights are the round-to-nearest-even cast of the float32
draw (numpy ``astype(float16)``), stored as their uint16 bit patterns, the way
an f32 master copy is cast to f16 for mixed precision.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

FORWARD_FORMS = (
    "matmul",
    "matmul_residual",
    "matmul_residual_swiglu_a",
    "matmul_w16",
    "matmul_residual_w16",
    "matmul_residual_swiglu_a_w16",
)
# backward input gradient dX[M,K] = dY[M,N] @ W[K,N]^T (+ dX)
T_FORMS = (
    "matmul_t",
    "matmul_t_acc",
    "matmul_t_w16",
    "matmul_t_acc_w16",
)
# backward weight gradient dW[K,N] = X[M,K]^T @ dY[M,N] (+ dW)
AT_FORMS = (
    "matmul_at",
    "matmul_at_acc",
    "matmul_at_swiglu_a",       # dW_down = (silu(GATE) * UP)^T @ dY
    "matmul_at_swiglu_a_acc",
)
# the FFN down projection's input gradient and the SwiGLU backward in one
# call: dA = dY @ W^T on chip, outputs dGATE and dUP [M,K]
SWIGLU_BWD_FORMS = (
    "matmul_t_swiglu_backward",
    "matmul_t_swiglu_backward_w16",
)
FORMS = FORWARD_FORMS + T_FORMS + AT_FORMS + SWIGLU_BWD_FORMS


def form_is_t(form: str) -> bool:
    """dX = dY @ W^T: output [M,K], contraction over N."""
    return form.startswith("matmul_t")


def form_is_swiglu_bwd(form: str) -> bool:
    return "swiglu_backward" in form


def form_is_at(form: str) -> bool:
    """dW = X^T @ dY: output [K,N], contraction over the M rows."""
    return form.startswith("matmul_at")


def form_has_residual(form: str) -> bool:
    """An R input added to the product: the forward residual [M,N], or the
    initial dX [M,K] of an accumulating transposed form."""
    return "residual" in form or "_acc" in form


def form_is_swiglu(form: str) -> bool:
    return "swiglu" in form


def form_is_w16(form: str) -> bool:
    return form.endswith("_w16")


@dataclass(frozen=True)
class Workload:
    """One named problem: form, dims (M, N, K) and input distributions."""

    index: int
    name: str
    form: str
    M: int
    N: int
    K: int
    a_var: float = 1.0          # X, or UP for the SwiGLU forms
    gate_var: float = 4.0       # GATE (SwiGLU forms only)
    w_var: float = 1.0          # W / W_down
    r_var: float = 1.0          # R (residual forms only)
    outlier_frac: float = 0.0   # GATE entries replaced by +-U(20, 100)

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def describe(self) -> str:
        return f"{self.form} M={self.M} N={self.N} K={self.K}"


WORKLOADS = (
    Workload(1, "attn_proj_f32", "matmul", 512, 768, 768, w_var=1.0 / 768),
    Workload(2, "ffn_up_residual_f32", "matmul_residual", 512, 3072, 768,
             w_var=1.0 / 768),
    Workload(3, "ffn_down_swiglu_f32", "matmul_residual_swiglu_a", 512, 768, 3072,
             w_var=1.0 / 3072, outlier_frac=0.01),
    Workload(4, "lm_head_w16", "matmul_w16", 512, 16384, 768, w_var=0.02),
    Workload(5, "ffn_down_swiglu_w16_16k", "matmul_residual_swiglu_a_w16",
             16384, 2048, 8192, w_var=1.0 / 8192),
)

# Backward input gradients of the same layers (dX = dY @ W^T; the contraction
# runs over the forward's output width N): measured beside the forward table,
# not part of the five configurations.
BACKWARD_WORKLOADS = (
    Workload(11, "attn_proj_dx_f32", "matmul_t", 512, 768, 768, w_var=1.0 / 768),
    Workload(12, "ffn_up_dx_f32", "matmul_t", 512, 3072, 768, w_var=1.0 / 768),
    Workload(13, "attn_proj_dw_f32", "matmul_at", 512, 768, 768, w_var=1.0),
    Workload(16, "ffn_up_dw_f32", "matmul_at", 512, 3072, 768, w_var=1.0),
    Workload(17, "ffn_down_dw_swiglu_f32", "matmul_at_swiglu_a", 512, 768, 3072, w_var=1.0,
             outlier_frac=0.01),
    Workload(18, "ffn_down_dgu_swiglu_f32", "matmul_t_swiglu_backward", 512, 768, 3072,
             w_var=1.0 / 3072, outlier_frac=0.01),
    Workload(14, "lm_head_dx_w16", "matmul_t_w16", 512, 16384, 768, w_var=0.02),
    Workload(15, "ffn_down_dx_w16_16k", "matmul_t_w16", 16384, 2048, 8192, w_var=1.0 / 8192),
    Workload(19, "ffn_down_dgu_w16_16k", "matmul_t_swiglu_backward_w16", 16384, 2048, 8192,
             w_var=1.0 / 8192),
)

WORKLOADS_BY_NAME = {w.name: w for w in WORKLOADS + BACKWARD_WORKLOADS}


def output_shape(form: str, M: int, N: int, K: int) -> tuple:
    """Shape of the output: Y [M,N], dX [M,K] (transposed forms) or dW [K,N]."""
    if form_is_at(form):
        return (K, N)
    return (M, K) if form_is_t(form) else (M, N)


def _normal(rng: np.random.Generator, shape, var: float) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    a *= np.float32(math.sqrt(var))
    return a


def _outliers(rng: np.random.Generator, a: np.ndarray, frac: float) -> None:
    """Replace a Bernoulli(frac) subset of entries by +-U(20, 100) in place."""
    if frac <= 0.0:
        return
    mask = rng.random(size=a.shape) < frac
    n = int(mask.sum())
    sign = np.where(rng.random(size=n) < 0.5, -1.0, 1.0)
    mag = rng.uniform(20.0, 100.0, size=n)
    a[mask] = (sign * mag).astype(np.float32)


def generate(form: str, M: int, N: int, K: int, seed: int, *, a_var: float = 1.0,
             gate_var: float = 4.0, w_var: float | None = None, r_var: float = 1.0,
             outlier_frac: float = 0.0) -> dict:
    """Draw the inputs of ``form`` at dims (M, N, K).

    Returns a dict of C-contiguous numpy arrays named as in the C ABI:
    ``X`` [M,K] float32 or ``GATE``/``UP`` [M,K] float32; ``W`` [K,N] float32
    or ``W16`` [K,N] uint16 (binary16 bits); ``R`` [M,N] float32 for the
    residual forms. ``w_var`` defaults to 1/K. The transposed forms draw
    ``DY`` [M,N] (variance ``a_var``) in place of X, then W, then ``R`` =
    the initial dX [M,K] of the accumulating ones. The weight-gradient forms
    draw ``X`` [M,K], ``DY`` [M,N] (variance ``w_var``) and ``R`` = the
    initial dW [K,N].
    """
    if form not in FORMS:
        raise ValueError(f"unknown form {form!r}")
    rng = np.random.Generator(np.random.PCG64(seed))
    if w_var is None:
        w_var = 1.0 / max(K, 1)
    out = {}
    if form_is_at(form):   # X [M,K] (or GATE, UP), dY [M,N], R = the initial dW [K,N]
        if form_is_swiglu(form):
            gate = _normal(rng, (M, K), gate_var)
            _outliers(rng, gate, outlier_frac)
            out["GATE"] = gate
            out["UP"] = _normal(rng, (M, K), a_var)
        else:
            out["X"] = _normal(rng, (M, K), a_var)
        out["DY"] = _normal(rng, (M, N), w_var)
        if form_has_residual(form):
            out["R"] = _normal(rng, (K, N), r_var)
        return out
    if form_is_t(form):
        out["DY"] = _normal(rng, (M, N), a_var)
        w = _normal(rng, (K, N), w_var)
        if form_is_w16(form):
            out["W16"] = w.astype(np.float16).view(np.uint16)
        else:
            out["W"] = w
        if form_has_residual(form):
            out["R"] = _normal(rng, (M, K), r_var)
        if form_is_swiglu_bwd(form):   # the forward's GATE and UP [M,K]
            gate = _normal(rng, (M, K), gate_var)
            _outliers(rng, gate, outlier_frac)
            out["GATE"] = gate
            out["UP"] = _normal(rng, (M, K), 1.0)
        return out
    if form_is_swiglu(form):
        gate = _normal(rng, (M, K), gate_var)
        _outliers(rng, gate, outlier_frac)
        out["GATE"] = gate
        out["UP"] = _normal(rng, (M, K), a_var)
    else:
        out["X"] = _normal(rng, (M, K), a_var)
    w = _normal(rng, (K, N), w_var)
    if form_is_w16(form):
        out["W16"] = w.astype(np.float16).view(np.uint16)
    else:
        out["W"] = w
    if form_has_residual(form):
        out["R"] = _normal(rng, (M, N), r_var)
    return out


def generate_workload(w: Workload) -> dict:
    """Inputs of a named workload (seed 1000 + its index)."""
    return generate(w.form, w.M, w.N, w.K, w.seed, a_var=w.a_var, gate_var=w.gate_var,
                    w_var=w.w_var, r_var=w.r_var, outlier_frac=w.outlier_frac)


def input_bytes(form: str, M: int, N: int, K: int) -> int:
    """Bytes of every input read once plus Y written once (the algorithmic
    traffic of one call; the SwiGLU hidden matrix is not counted because the
    fused form never stores it)."""
    w = K * N * (2 if form_is_w16(form) else 4)
    if form_is_at(form):  # X (or GATE, UP), dY in; dW [K,N] out (read too when accumulating)
        a = 2 * M * K * 4 if form_is_swiglu(form) else M * K * 4
        return a + M * N * 4 + (K * N * 4 if form_has_residual(form) else 0) + K * N * 4
    if form_is_swiglu_bwd(form):   # dY, W, GATE, UP in; dGATE, dUP out
        return M * N * 4 + w + 2 * M * K * 4 + 2 * M * K * 4
    if form_is_t(form):   # dY [M,N] in, dX [M,K] out (read too when accumulating)
        return M * N * 4 + w + (M * K * 4 if form_has_residual(form) else 0) + M * K * 4
    a = 2 * M * K * 4 if form_is_swiglu(form) else M * K * 4
    r = M * N * 4 if form_has_residual(form) else 0
    y = M * N * 4
    return a + w + r + y
