"""fp64 CPU oracle for the forward linear-layer family.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The CUDA library and
its Python binding never import it, and it imports nothing from them: the two
sides share no code. The only thing both sides consume is the seeded input
generator in ``transformer_linear_layer_tcgen05_gb300.workloads``, which holds
none of the method's arithmetic.

What is computed, and where the pages define it
-----------------------------------------------
Page "matmul ve matmul_residual -- Tiled Matrix Multiply (Forward)"
(llm.istanbul/learn/tr/03_linear_forward), section "Ne Yapar?":

* ``matmul``                    Y[M,N] = X[M,K] @ W[K,N]
* ``matmul_residual``           Y = X @ W + R, R[M,N] added in the epilogue
* ``matmul_residual_swiglu_a``  Y = (silu(GATE) * UP) @ W_down + R, the
                                element-wise SwiGLU product feeding W_down
* ``*_w16``                     the same three with W stored as IEEE binary16
                                (list of forward kernels at the top of the page;
                                "matmul_w16 -- f16 weight versiyonu")

Page "ffn_gelu_backward ve ffn_swiglu_backward"
(llm.istanbul/learn/tr/09_backward_ffn), section "SiLU'" and
"WGSL-Spesifik Notlar" note 2: silu(x) = x * sigma(x) with the stable,
sign-branched sigmoid -- for x >= 0 it is 1 / (1 + exp(-x)), otherwise
e / (1 + e) with e = exp(x), so exp() never sees a positive argument and no
clamp is applied. The same page (note 3) says the forward kernels share this
helper.

Backward input gradient (``matmul_t``; the material does not include the
pages' backward-linear page, "11_backward_linear"). Reading: the input
gradient of Y = X @ W is the adjoint of the forward map X -> X @ W under the
Frobenius inner product, dX = dY @ W^T, i.e. the unique dX with
sum(dX * X) == sum(dY * (X @ W)) for every X; ``matmul_t_acc`` adds it to
an existing dX (dX += dY @ W^T), ``_w16`` takes W as binary16 bits. dY is
[M,N], W is [K,N] as the forward stores it, dX is [M,K]. The weight
gradient (``matmul_at``) is the adjoint with respect to W: dW = X^T @ dY
[K,N], the unique dW with sum(dW * W) == sum(dY * (X @ W)) for every W;
``matmul_at_acc`` adds it to an existing dW. ``matmul_at_swiglu_a`` is the
weight gradient of the SwiGLU down projection, (silu(GATE) * UP)^T @ dY,
the left factor recomputed from GATE and UP as in the forward form.

SwiGLU backward (page "ffn_gelu_backward ve ffn_swiglu_backward",
09_backward_ffn, sections "SwiGLU backward", "SiLU'" and the
"ffn_swiglu_backward" walk-through): for the hidden gradient g,
grad_gate = g * up * silu'(gate) and grad_up = g * silu(gate), with
silu'(x) = s * (1 + x * (1 - s)), s the stable sigmoid, each passed through
nan_guard (page "00_shared", "C. NaN/Inf Guard": x if x == x and
|x| < F32_MAX, else 0). ``matmul_t_swiglu_backward`` applies it to
g = dY @ W^T, the input gradient of the SwiGLU form's down projection.

Cross-entropy (page "cross_entropy ve sum_losses -- Fused Loss + dLogits",
07_loss, sections "Ne Yapar?" and "Satir Satir -- cross_entropy"): for a logits row l over
the vocabulary V with target t, LSE = row_max + log sum_v exp(l_v -
row_max) (the sum guarded below by 1e-30), loss = LSE - (1 - alpha) l_t -
alpha mean(l) + beta LSE^2, and dLogits_v = ((p_v - target_dist_v) +
2 beta LSE p_v) * inv_norm with p = softmax(l) and target_dist =
(1 - alpha) one_hot(t) + alpha / V; a target outside [0, V) gives loss 0
and dLogits 0. ``sum_losses`` adds the per-row losses. ``lm_head_cross_entropy``
applies both to the logits X @ W16 of the lm_head projection.

Gate and up projections (``gate_up_w16``): the pages name GATE and UP as the
outputs of the FFN's gate and up projections (03_linear_forward, the
SwiGLU form's bind group) without describing their producer. Reading: the
two plain products GATE = X @ W_gate and UP = X @ W_up of one X, binary16
weights, evaluated here as two ``matmul_w16`` calls.

Everything is evaluated in float64. Inputs are widened exactly: float32 to
float64 by numpy, binary16 bit patterns by ``f16_bits_to_f64`` below (an
IEEE 754 decoder written from the format's definition). Every contraction
(the forward products, both backward products and the normaliser) is the
plain triple loop of ``gemm_f64.c`` in this directory: for each output row i,
for k in ascending order, for every column j, Y[i,j] += A[i,k] * B[k,j] and
S[i,j] += |A[i,k] * B[k,j]|, in fp64 with no fused multiply-add; it is
compiled by gcc on first use (``build_native.py``). The transposed operands
of the backward products are copied to row-major form first (a copy, no
arithmetic). Nothing is blocked, fused or reordered beyond the definitions
above.

Acceptance metric (the normalised error) is ``normalised_error``: for every
output element, |Y - Y_ref| / S with S[i,j] = sum_k |A[i,k] * W[k,j]|, A being
X or silu(GATE) * UP. Where S is 0 nothing was accumulated and the element
must equal the residual (or 0) exactly.

Every function here is pinned by ``tests/test_oracle.py`` against closed forms,
hand-computed fixtures in ``tests/golden/``, exact integer brute force,
invariants and numpy's own binary16 type.
"""

from __future__ import annotations

import ctypes
import math

import numpy as np

__all__ = [
    "sigmoid",
    "silu",
    "f16_bits_to_f64",
    "swiglu_a",
    "matmul",
    "matmul_residual",
    "matmul_residual_swiglu_a",
    "matmul_w16",
    "matmul_residual_w16",
    "matmul_residual_swiglu_a_w16",
    "matmul_t",
    "matmul_t_acc",
    "matmul_t_w16",
    "matmul_t_acc_w16",
    "matmul_at",
    "matmul_at_acc",
    "matmul_at_swiglu_a",
    "matmul_at_swiglu_a_acc",
    "silu_derivative",
    "nan_guard",
    "ffn_swiglu_backward",
    "matmul_t_swiglu_backward",
    "matmul_t_swiglu_backward_w16",
    "cross_entropy",
    "lm_head_cross_entropy_w16",
    "gate_up_w16",
    "normaliser",
    "normalised_error",
    "reference",
    "contraction_threads",
    "FORMS",
]

FORMS = (
    "matmul",
    "matmul_residual",
    "matmul_residual_swiglu_a",
    "matmul_w16",
    "matmul_residual_w16",
    "matmul_residual_swiglu_a_w16",
    "matmul_t",
    "matmul_t_acc",
    "matmul_t_w16",
    "matmul_t_acc_w16",
    "matmul_at",
    "matmul_at_acc",
    "matmul_at_swiglu_a",
    "matmul_at_swiglu_a_acc",
    "matmul_t_swiglu_backward",
    "matmul_t_swiglu_backward_w16",
)


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# The contraction: the triple loop of gemm_f64.c
# --------------------------------------------------------------------------

_LIB = None


def _gemm_lib():
    global _LIB
    if _LIB is None:
        from . import build_native

        lib = ctypes.CDLL(build_native.build())
        lib.oracle_gemm_f64.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 3
        lib.oracle_gemm_f64.restype = None
        lib.oracle_gemm_threads.argtypes = []
        lib.oracle_gemm_threads.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def contraction_threads() -> int:
    """Host threads the contraction's row loop runs on."""
    return int(_gemm_lib().oracle_gemm_threads())


def _contract(A, B, with_s: bool):
    """(Y, S) with Y[i,j] = sum_k A[i,k] B[k,j] and, if asked, S[i,j] =
    sum_k |A[i,k] B[k,j]| (else None): the triple loop, k ascending."""
    A = np.ascontiguousarray(_f64(A))
    B = np.ascontiguousarray(_f64(B))
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch: {A.shape} @ {B.shape}")
    M, K = A.shape
    N = B.shape[1]
    Y = np.zeros((M, N))
    S = np.zeros((M, N)) if with_s else None
    if M and N:
        _gemm_lib().oracle_gemm_f64(A.ctypes.data, B.ctypes.data, Y.ctypes.data,
                                    S.ctypes.data if with_s else None, M, N, K)
    return Y, S


# --------------------------------------------------------------------------
# Activation (09_backward_ffn, "SiLU'" and "WGSL-Spesifik Notlar" note 2)
# --------------------------------------------------------------------------

def sigmoid(x) -> np.ndarray:
    """Stable sigmoid, branched on the sign of x.

    x >= 0: 1 / (1 + exp(-x));  x < 0: e / (1 + e) with e = exp(x).
    exp() therefore only sees arguments <= 0: no overflow, and very negative
    x underflows gracefully towards 0 (09_backward_ffn, note 2).
    """
    x = _f64(x)
    out = np.empty_like(x)
    nonneg = x >= 0.0
    out[nonneg] = 1.0 / (1.0 + np.exp(-x[nonneg]))
    e = np.exp(x[~nonneg])
    out[~nonneg] = e / (1.0 + e)
    return out


def silu(x) -> np.ndarray:
    """silu(x) = x * sigmoid(x) (09_backward_ffn, "SiLU'": forward)."""
    x = _f64(x)
    return x * sigmoid(x)


# --------------------------------------------------------------------------
# binary16 decoding (the f16 weights of the *_w16 forms)
# --------------------------------------------------------------------------

def f16_bits_to_f64(bits) -> np.ndarray:
    """Decode IEEE 754 binary16 bit patterns (uint16) to float64, exactly.

    Layout: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
    exponent 0      -> subnormal: (-1)^s * 2^-14 * (f / 1024)
    exponent 1..30  -> normal:    (-1)^s * 2^(e-15) * (1 + f / 1024)
    exponent 31     -> +-inf (f == 0) or NaN (f != 0)
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    normal = np.ldexp(1.0 + f / 1024.0, (e - 15).astype(np.int64))
    subnormal = np.ldexp(f / 1024.0, -14)
    mag = np.where(e == 0, subnormal, normal)
    mag = np.where(e == 31, np.where(f == 0.0, np.inf, np.nan), mag)
    return sign * mag


# --------------------------------------------------------------------------
# The three definitions (03_linear_forward, "Ne Yapar?")
# --------------------------------------------------------------------------

def swiglu_a(gate, up) -> np.ndarray:
    """A[i,k] = silu(GATE[i,k]) * UP[i,k]: the SwiGLU hidden matrix that
    matmul_residual_swiglu_a feeds into W_down (03_linear_forward, "Ne Yapar?"
    and "Önemli Optimizasyonlar" 3)."""
    return silu(gate) * _f64(up)


def matmul(X, W) -> np.ndarray:
    """Y[M,N] = X[M,K] @ W[K,N], row-major, in float64."""
    X = _f64(X)
    W = _f64(W)
    if X.ndim != 2 or W.ndim != 2 or X.shape[1] != W.shape[0]:
        raise ValueError(f"shape mismatch: X{X.shape} @ W{W.shape}")
    return _contract(X, W, False)[0]


def matmul_residual(X, W, R) -> np.ndarray:
    """Y = X @ W + R (R[M,N] added in the epilogue)."""
    Y = matmul(X, W)
    R = _f64(R)
    if R.shape != Y.shape:
        raise ValueError(f"residual shape {R.shape} != output shape {Y.shape}")
    return Y + R


def matmul_residual_swiglu_a(GATE, UP, W, R) -> np.ndarray:
    """Y = (silu(GATE) * UP) @ W_down + R, GATE and UP [M,K], W_down [K,N]."""
    GATE = _f64(GATE)
    UP = _f64(UP)
    if GATE.shape != UP.shape:
        raise ValueError(f"GATE{GATE.shape} and UP{UP.shape} differ")
    return matmul_residual(swiglu_a(GATE, UP), W, R)


def matmul_w16(X, W16) -> np.ndarray:
    """matmul with W given as binary16 bit patterns (uint16 [K,N])."""
    return matmul(X, f16_bits_to_f64(W16))


def matmul_residual_w16(X, W16, R) -> np.ndarray:
    """matmul_residual with binary16 weights."""
    return matmul_residual(X, f16_bits_to_f64(W16), R)


def matmul_residual_swiglu_a_w16(GATE, UP, W16, R) -> np.ndarray:
    """matmul_residual_swiglu_a with binary16 W_down."""
    return matmul_residual_swiglu_a(GATE, UP, f16_bits_to_f64(W16), R)


def matmul_t(DY, W) -> np.ndarray:
    """dX[M,K] = dY[M,N] @ W[K,N]^T: the adjoint of X -> X @ W (input
    gradient of the forward "matmul"), in float64."""
    DY = _f64(DY)
    W = _f64(W)
    if DY.ndim != 2 or W.ndim != 2 or DY.shape[1] != W.shape[1]:
        raise ValueError(f"shape mismatch: dY{DY.shape} @ W{W.shape}^T")
    return _contract(DY, W.T, False)[0]


def matmul_t_acc(DY, W, DX0) -> np.ndarray:
    """dX0 + dY @ W^T (the accumulating form)."""
    Y = matmul_t(DY, W)
    DX0 = _f64(DX0)
    if DX0.shape != Y.shape:
        raise ValueError(f"initial dX shape {DX0.shape} != output shape {Y.shape}")
    return DX0 + Y


def matmul_t_w16(DY, W16) -> np.ndarray:
    """matmul_t with W given as binary16 bit patterns (uint16 [K,N])."""
    return matmul_t(DY, f16_bits_to_f64(W16))


def matmul_t_acc_w16(DY, W16, DX0) -> np.ndarray:
    """matmul_t_acc with binary16 weights."""
    return matmul_t_acc(DY, f16_bits_to_f64(W16), DX0)


def matmul_at(X, DY) -> np.ndarray:
    """dW[K,N] = X[M,K]^T @ dY[M,N]: the adjoint of W -> X @ W (weight
    gradient of the forward "matmul"), in float64."""
    X = _f64(X)
    DY = _f64(DY)
    if X.ndim != 2 or DY.ndim != 2 or X.shape[0] != DY.shape[0]:
        raise ValueError(f"shape mismatch: X{X.shape}^T @ dY{DY.shape}")
    return _contract(X.T, DY, False)[0]


def matmul_at_acc(X, DY, DW0) -> np.ndarray:
    """dW0 + X^T @ dY (the accumulating form)."""
    Y = matmul_at(X, DY)
    DW0 = _f64(DW0)
    if DW0.shape != Y.shape:
        raise ValueError(f"initial dW shape {DW0.shape} != output shape {Y.shape}")
    return DW0 + Y


def matmul_at_swiglu_a(GATE, UP, DY) -> np.ndarray:
    """dW[K,N] = (silu(GATE) * UP)[M,K]^T @ dY[M,N]: the weight gradient of
    W_down in matmul_residual_swiglu_a, in float64."""
    GATE = _f64(GATE)
    UP = _f64(UP)
    if GATE.shape != UP.shape:
        raise ValueError(f"GATE{GATE.shape} and UP{UP.shape} differ")
    return matmul_at(swiglu_a(GATE, UP), DY)


def matmul_at_swiglu_a_acc(GATE, UP, DY, DW0) -> np.ndarray:
    """dW0 + (silu(GATE) * UP)^T @ dY."""
    return matmul_at_acc(swiglu_a(_f64(GATE), _f64(UP)), DY, DW0)


F32_MAX = float(np.finfo(np.float32).max)


def silu_derivative(x) -> np.ndarray:
    """silu'(x) = s * (1 + x * (1 - s)), s = sigmoid(x) (09_backward_ffn, "SiLU'")."""
    x = _f64(x)
    s = sigmoid(x)
    return s * (1.0 + x * (1.0 - s))


def nan_guard(x) -> np.ndarray:
    """x where x == x and |x| < F32_MAX, else 0 (00_shared, "C. NaN/Inf Guard").
    The limit is binary32's: a float64 value beyond it is what binary32
    arithmetic would have turned into an infinity."""
    x = _f64(x)
    with np.errstate(invalid="ignore"):
        ok = (x == x) & (np.abs(x) < F32_MAX)
    return np.where(ok, x, 0.0)


def ffn_swiglu_backward(G, GATE, UP):
    """(grad_gate, grad_up) for the hidden gradient G of A = silu(GATE) * UP:
    nan_guard(G * UP * silu'(GATE)) and nan_guard(G * silu(GATE))."""
    G = _f64(G)
    GATE = _f64(GATE)
    UP = _f64(UP)
    if not (G.shape == GATE.shape == UP.shape):
        raise ValueError(f"G{G.shape}, GATE{GATE.shape} and UP{UP.shape} differ")
    with np.errstate(invalid="ignore", over="ignore"):
        dgate = nan_guard(G * UP * silu_derivative(GATE))
        dup = nan_guard(G * silu(GATE))
    return dgate, dup


def matmul_t_swiglu_backward(DY, W, GATE, UP):
    """ffn_swiglu_backward of dA = dY @ W^T (dY [M,N], W [K,N], GATE/UP [M,K])."""
    return ffn_swiglu_backward(matmul_t(DY, W), GATE, UP)


def matmul_t_swiglu_backward_w16(DY, W16, GATE, UP):
    """matmul_t_swiglu_backward with binary16 W_down bits."""
    return matmul_t_swiglu_backward(DY, f16_bits_to_f64(W16), GATE, UP)


def cross_entropy(logits, targets, alpha=0.0, beta=0.0, inv_norm=1.0):
    """(losses [M], dlogits [M,V]) of the pages' fused cross-entropy with
    label smoothing alpha and z-loss beta, in float64."""
    L = _f64(logits)
    if L.ndim != 2:
        raise ValueError("logits must be [M, V]")
    M, V = L.shape
    t = np.asarray(targets).astype(np.int64).reshape(-1)
    if t.shape != (M,):
        raise ValueError("one target per row")
    losses = np.zeros(M)
    dl = np.zeros((M, V))
    for s in range(M):
        if not (0 <= t[s] < V):
            continue                      # ignored row: loss 0, gradient 0
        row = L[s]
        mx = np.max(row)
        denom = max(float(np.sum(np.exp(row - mx))), 1e-30)
        lse = mx + math.log(denom)
        p = np.exp(row - mx) / denom
        losses[s] = lse - (1.0 - alpha) * row[t[s]] - alpha * float(np.mean(row)) \
            + beta * lse * lse
        tgt = np.full(V, alpha / V)
        tgt[t[s]] += 1.0 - alpha
        dl[s] = ((p - tgt) + 2.0 * beta * lse * p) * inv_norm
    return losses, dl


def lm_head_cross_entropy_w16(X, W16, targets, alpha=0.0, beta=0.0, inv_norm=1.0):
    """(losses, dlogits, loss_sum) for logits = X @ W16 (binary16 bits)."""
    losses, dl = cross_entropy(matmul_w16(X, W16), targets, alpha, beta, inv_norm)
    return losses, dl, float(np.sum(losses))


def gate_up_w16(X, WG16, WU16):
    """(GATE, UP) = (X @ W_gate, X @ W_up), binary16 weight bits [K,N]: the
    producer of the SwiGLU form's inputs (not on the pages; two matmul_w16
    products of one X)."""
    return matmul_w16(X, WG16), matmul_w16(X, WU16)


# --------------------------------------------------------------------------
# Acceptance metric
# --------------------------------------------------------------------------

def normaliser(A, W) -> np.ndarray:
    """S[i,j] = sum_k |A[i,k] * W[k,j]|, in float64 (the triple loop).

    A is the left operand as the definition states it (X, or
    silu(GATE) * UP), before any rounding a fast path may apply; W is the
    weight matrix as stored (binary16 values decoded exactly).
    """
    return _contract(A, W, True)[1]


def normalised_error(Y, Y_ref, S, R=None) -> float:
    """max_ij |Y - Y_ref| / S over all elements.

    Elements with S == 0 accumulated nothing: there Y must equal float32(R)
    (or 0 without a residual) exactly, else the error is reported as inf.
    Non-finite Y anywhere is an infinite error.
    """
    Y = _f64(Y)
    Y_ref = _f64(Y_ref)
    S = _f64(S)
    if not (Y.shape == Y_ref.shape == S.shape):
        raise ValueError("Y, Y_ref and S must have one shape")
    if Y.size == 0:
        return 0.0
    if not np.all(np.isfinite(Y)):
        return float("inf")
    zero = S == 0.0
    err = 0.0
    if np.any(~zero):
        err = float(np.max(np.abs(Y[~zero] - Y_ref[~zero]) / S[~zero]))
    if np.any(zero):
        expect = np.zeros_like(Y) if R is None else _f64(np.asarray(R, dtype=np.float32))
        if not np.array_equal(Y[zero], expect[zero]):
            return float("inf")
    return err


def reference(form: str, inputs: dict, rows=None):
    """Evaluate ``form`` on an input dict; return (Y_ref, S).

    ``inputs`` holds the arrays named by the C ABI: X or GATE/UP (DY for the
    transposed forms), W (float32) or W16 (uint16 bit patterns), and R for
    the residual forms (the initial dX of the accumulating ones). ``rows`` picks
    a subset of output rows: every output row depends only on the same row of
    X / GATE / UP / R, so a row subset is the definition applied to those rows.
    """
    if form not in FORMS:
        raise ValueError(f"unknown form {form!r}")
    sel = (lambda a: a) if rows is None else (lambda a: np.asarray(a)[rows])
    # Y and its normaliser S come from one pass of the triple loop; the
    # residual (or the initial value of an accumulating form) is added after
    # the sum, as in matmul_residual / matmul_t_acc / matmul_at_acc.
    if form.startswith("matmul_at"):
        # dW row k depends on column k of X (all rows of X and dY): ``rows``
        # picks output rows of dW here
        X = swiglu_a(inputs["GATE"], inputs["UP"]) if "swiglu" in form else _f64(inputs["X"])
        DY = _f64(inputs["DY"])
        Xk = X if rows is None else X[:, rows]
        if Xk.shape[0] != DY.shape[0]:
            raise ValueError(f"shape mismatch: X{Xk.shape}^T @ dY{DY.shape}")
        Y, S = _contract(Xk.T, DY, True)
        if "_acc" in form:
            Y = _plus(Y, sel(inputs["R"]))
        return Y, S
    w16 = form.endswith("_w16")
    W = f16_bits_to_f64(inputs["W16"]) if w16 else _f64(inputs["W"])
    if "swiglu_backward" in form:
        # two outputs: ((dGATE, dUP), (S_dGATE, S_dUP)). As for the product,
        # S sums the magnitudes of the terms: the product's S times those of
        # the element-wise factor, silu'(x) = s + x*s*(1-s) -> s + |x|*s*(1-s)
        # (its two terms cancel near x = -1.28, where silu' is 0) and
        # silu(x) = x*s -> |x|*s.
        DY = _f64(sel(inputs["DY"]))
        GATE = _f64(sel(inputs["GATE"]))
        UP = _f64(sel(inputs["UP"]))
        if DY.shape[1] != W.shape[1]:
            raise ValueError(f"shape mismatch: dY{DY.shape} @ W{W.shape}^T")
        dA, S = _contract(DY, W.T, True)
        dgate, dup = ffn_swiglu_backward(dA, GATE, UP)
        s = sigmoid(GATE)
        with np.errstate(invalid="ignore", over="ignore"):
            Sg = nan_guard(S * np.abs(UP) * (s + np.abs(GATE) * s * (1.0 - s)))
            Su = nan_guard(S * np.abs(GATE) * s)
        return (dgate, dup), (Sg, Su)
    if form.startswith("matmul_t"):
        # dX row i depends only on dY row i (and R row i)
        A = _f64(sel(inputs["DY"]))
        if A.shape[1] != W.shape[1]:
            raise ValueError(f"shape mismatch: dY{A.shape} @ W{W.shape}^T")
        Y, S = _contract(A, W.T, True)
        if "_acc" in form:
            Y = _plus(Y, sel(inputs["R"]))
        return Y, S
    if "swiglu" in form:
        A = swiglu_a(sel(inputs["GATE"]), sel(inputs["UP"]))
    else:
        A = _f64(sel(inputs["X"]))
    Y, S = _contract(A, W, True)
    if "residual" in form:
        Y = _plus(Y, sel(inputs["R"]))
    return Y, S


def _plus(Y, R) -> np.ndarray:
    """Y + R for an [M,N] residual (or initial value) R."""
    R = _f64(R)
    if R.shape != Y.shape:
        raise ValueError(f"residual shape {R.shape} != output shape {Y.shape}")
    return Y + R
