"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: hand-computed
fixtures in tests/golden/, closed forms of the sigmoid, exact integer brute
force, numpy's own binary16 type, and invariants the definitions imply.
Definitions: llm.istanbul 03_linear_forward ("Ne Yapar?") and
09_backward_ffn ("SiLU'", "WGSL-Spesifik Notlar" note 2).
"""

import itertools
import math

import numpy as np
import pytest

import oracle
from tests.golden_io import read_blocks, read_rows


# ---------------------------------------------------------------- fixtures

def test_golden_matmul_and_residual():
    g = read_blocks("matmul_3x2x4.txt")
    assert np.array_equal(oracle.matmul(g["X"], g["W"]), g["Y_matmul"])
    assert np.array_equal(oracle.matmul_residual(g["X"], g["W"], g["R"]), g["Y_residual"])
    assert np.array_equal(oracle.normaliser(g["X"], g["W"]), g["S"])


def test_golden_swiglu():
    g = read_blocks("swiglu_2x2x2.txt")
    A = oracle.swiglu_a(g["GATE"], g["UP"])
    np.testing.assert_allclose(A, g["A"], rtol=1e-15, atol=0)
    Y = oracle.matmul_residual_swiglu_a(g["GATE"], g["UP"], g["W"], g["R"])
    np.testing.assert_allclose(Y, g["Y"], rtol=1e-15, atol=0)
    np.testing.assert_allclose(oracle.normaliser(A, g["W"]), g["S"], rtol=1e-15, atol=0)


def test_golden_sigmoid_closed_forms():
    for x, s, y in read_rows("sigmoid_closed_forms.txt"):
        x, s, y = float(x), float(s), float(y)
        got_s = float(oracle.sigmoid(np.array([x]))[0])
        got_y = float(oracle.silu(np.array([x]))[0])
        assert math.isclose(got_s, s, rel_tol=1e-15, abs_tol=0.0), (x, got_s, s)
        assert math.isclose(got_y, y, rel_tol=1e-15, abs_tol=0.0), (x, got_y, y)


def test_golden_f16_bits():
    for hx, val in read_rows("f16_bits.txt"):
        got = float(oracle.f16_bits_to_f64(np.array([int(hx, 16)], dtype=np.uint16))[0])
        want = float(val)
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), hx


# ---------------------------------------------------------------- sigmoid / silu

def test_sigmoid_symmetry_and_range():
    x = np.linspace(-60.0, 60.0, 4801)
    s = oracle.sigmoid(x)
    np.testing.assert_allclose(s + oracle.sigmoid(-x), 1.0, rtol=0, atol=4.5e-16)  # 2 ulp of 1
    assert np.all((s >= 0.0) & (s <= 1.0))
    assert np.all(np.diff(s) >= 0.0)            # monotone non-decreasing


def test_sigmoid_no_overflow_or_nan():
    x = np.concatenate([np.linspace(-1000.0, 1000.0, 20001), [-1e300, 1e300, -745.2, 710.0]])
    with np.errstate(over="raise", invalid="raise"):
        s = oracle.sigmoid(x)
        y = oracle.silu(x)
    assert np.all(np.isfinite(s)) and np.all(np.isfinite(y[np.abs(x) <= 1e3]))


def test_silu_identities():
    x = np.linspace(-30.0, 30.0, 1201)
    # x*s(x) - (-x)*s(-x) = x*(s(x) + s(-x)) = x
    np.testing.assert_allclose(oracle.silu(x) - oracle.silu(-x), x, rtol=0, atol=1e-13)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    # derivative at 0 is sigma(0) = 1/2: central difference
    h = 1e-6
    d = (oracle.silu(np.array([h])) - oracle.silu(np.array([-h])))[0] / (2 * h)
    assert abs(d - 0.5) < 1e-9


def test_sigmoid_branch_matches_logistic_where_safe():
    # In the range where exp(-x) cannot overflow, the textbook 1/(1+e^-x) is a
    # library-independent special case of the same function.
    x = np.linspace(-30.0, 30.0, 601)
    np.testing.assert_allclose(oracle.sigmoid(x), 1.0 / (1.0 + np.exp(-x)), rtol=1e-14, atol=0)


# ---------------------------------------------------------------- binary16

def test_f16_decoder_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_bits_to_f64(bits)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


# ---------------------------------------------------------------- contraction

def _int_matrix(rng, shape, lo=-4, hi=4):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64)


def _brute(X, W):
    M, K = X.shape
    N = W.shape[1]
    out = [[0] * N for _ in range(M)]
    for i, j in itertools.product(range(M), range(N)):
        out[i][j] = sum(int(X[i, k]) * int(W[k, j]) for k in range(K))
    return np.array(out, dtype=np.float64).reshape(M, N)


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (2, 3, 4), (5, 1, 7), (8, 8, 8), (3, 7, 2), (6, 5, 1)])
def test_integer_brute_force(M, K, N):
    rng = np.random.default_rng(M * 100 + K * 10 + N)
    X, W, R = _int_matrix(rng, (M, K)), _int_matrix(rng, (K, N)), _int_matrix(rng, (M, N))
    want = _brute(X, W)
    assert np.array_equal(oracle.matmul(X, W), want)
    assert np.array_equal(oracle.matmul_residual(X, W, R), want + R)
    assert np.array_equal(oracle.normaliser(X, W), _brute(np.abs(X), np.abs(W)))


def test_identity_and_one_hot_weights():
    rng = np.random.default_rng(7)
    X = rng.standard_normal((5, 6))
    assert np.array_equal(oracle.matmul(X, np.eye(6)), X)
    for k in range(6):
        for j in (0, 3):
            W = np.zeros((6, 4))
            W[k, j] = 1.0
            Y = oracle.matmul(X, W)
            assert np.array_equal(Y[:, j], X[:, k])
            assert np.count_nonzero(Y[:, [c for c in range(4) if c != j]]) == 0


def test_residual_invariant_exact():
    rng = np.random.default_rng(11)
    X, W, R = _int_matrix(rng, (9, 13)), _int_matrix(rng, (13, 6)), _int_matrix(rng, (9, 6))
    assert np.array_equal(oracle.matmul_residual(X, W, R) - oracle.matmul(X, W), R)


def test_swiglu_reduces_to_product_for_large_gate():
    # sigma(g) == 1.0 exactly in float64 for g >= 40 (e^-40 < 2^-53), so
    # silu(g) = g and the fused form is the plain integer product (G*U)@W + R.
    rng = np.random.default_rng(3)
    G = rng.integers(40, 60, size=(4, 6)).astype(np.float64)
    U = _int_matrix(rng, (4, 6))
    W, R = _int_matrix(rng, (6, 5)), _int_matrix(rng, (4, 5))
    Y = oracle.matmul_residual_swiglu_a(G, U, W, R)
    assert np.array_equal(Y, _brute(G * U, W) + R)


def test_swiglu_zero_gate_kills_row():
    # silu(0) = 0, so a zero GATE row contributes nothing: Y row == R row.
    rng = np.random.default_rng(5)
    G = rng.standard_normal((3, 8))
    G[1] = 0.0
    U, W, R = rng.standard_normal((3, 8)), rng.standard_normal((8, 4)), rng.standard_normal((3, 4))
    Y = oracle.matmul_residual_swiglu_a(G, U, W, R)
    assert np.array_equal(Y[1], R[1])


def test_swiglu_composition_invariant():
    rng = np.random.default_rng(9)
    G, U = 2 * rng.standard_normal((7, 12)), rng.standard_normal((7, 12))
    W, R = rng.standard_normal((12, 5)), rng.standard_normal((7, 5))
    fused = oracle.matmul_residual_swiglu_a(G, U, W, R)
    staged = oracle.matmul_residual(oracle.swiglu_a(G, U), W, R)
    assert np.array_equal(fused, staged)


def test_w16_forms_match_f32_forms_on_representable_weights():
    rng = np.random.default_rng(13)
    Wf = rng.standard_normal((6, 8)).astype(np.float16)
    bits = Wf.view(np.uint16)
    W = Wf.astype(np.float64)
    X, G, U = rng.standard_normal((3, 6)), rng.standard_normal((3, 6)), rng.standard_normal((3, 6))
    R = rng.standard_normal((3, 8))
    assert np.array_equal(oracle.matmul_w16(X, bits), oracle.matmul(X, W))
    assert np.array_equal(oracle.matmul_residual_w16(X, bits, R), oracle.matmul_residual(X, W, R))
    assert np.array_equal(oracle.matmul_residual_swiglu_a_w16(G, U, bits, R),
                          oracle.matmul_residual_swiglu_a(G, U, W, R))


def test_shape_errors():
    with pytest.raises(ValueError):
        oracle.matmul(np.zeros((2, 3)), np.zeros((2, 3)))
    with pytest.raises(ValueError):
        oracle.matmul_residual(np.zeros((2, 3)), np.zeros((3, 4)), np.zeros((4, 2)))
    with pytest.raises(ValueError):
        oracle.matmul_residual_swiglu_a(np.zeros((2, 3)), np.zeros((3, 2)), np.zeros((3, 4)),
                                        np.zeros((2, 4)))


# ---------------------------------------------------------------- metric

def test_normalised_error_values():
    g = read_blocks("matmul_3x2x4.txt")
    S = g["S"]
    Y = g["Y_matmul"].copy()
    assert oracle.normalised_error(Y, g["Y_matmul"], S) == 0.0
    Y[2, 3] += 0.23                   # S[2,3] = 23 -> error 0.01
    assert math.isclose(oracle.normalised_error(Y, g["Y_matmul"], S), 0.01, rel_tol=1e-12)
    Y[0, 0] += 0.5                    # S[0,0] = 1  -> error 0.5 dominates
    assert math.isclose(oracle.normalised_error(Y, g["Y_matmul"], S), 0.5, rel_tol=1e-12)
    Y[1, 1] = np.nan
    assert oracle.normalised_error(Y, g["Y_matmul"], S) == math.inf


def test_normalised_error_zero_rows():
    S = np.array([[0.0, 0.0], [1.0, 2.0]])
    R = np.array([[0.1, -2.0], [0.0, 0.0]], dtype=np.float32)
    ref = np.array([[0.1, -2.0], [1.0, 1.0]])
    Y = np.array([[np.float32(0.1), -2.0], [1.0, 1.0]])
    assert oracle.normalised_error(Y, ref, S, R) == 0.0
    Y2 = Y.copy()
    Y2[0, 0] = 0.1 + 1e-9                # not the float32 residual
    assert oracle.normalised_error(Y2, ref, S, R) == math.inf
    assert oracle.normalised_error(np.zeros((2, 2)), np.zeros((2, 2)), np.zeros((2, 2))) == 0.0


def test_reference_row_subset_equals_full():
    from transformer_linear_layer_tcgen05_gb300.workloads import generate, output_shape
    for form in oracle.FORMS:
        inp = generate(form, 20, 16, 12, seed=42)
        Y, S = oracle.reference(form, inp)
        last = output_shape(form, 20, 16, 12)[0] - 1
        rows = np.array([0, 3, last, 7])
        if "swiglu_backward" in form:   # two outputs and two normalisers
            (Yg, Yu), (Sg, Su) = Y, S
            (Ygr, Yur), (Sgr, Sur) = oracle.reference(form, inp, rows=rows)
            for a, b in ((Ygr, Yg), (Yur, Yu), (Sgr, Sg), (Sur, Su)):
                assert np.array_equal(a, b[rows])
            assert np.all(Sg >= np.abs(Yg) - 1e-12) and np.all(Su >= np.abs(Yu) - 1e-12)
            continue
        Yr, Sr = oracle.reference(form, inp, rows=rows)
        assert np.array_equal(Yr, Y[rows]) and np.array_equal(Sr, S[rows])
        assert np.all(S >= np.abs(Y - (inp["R"] if "R" in inp else 0.0)) - 1e-12)


# ---------------------------------------------------------------- backward: dX = dY @ W^T
# The backward-linear page is not in the material; matmul_t is read as the
# adjoint of the forward product (oracle module docstring). These pins tie it
# to that definition, not to its own formula.

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 5), (4, 1, 3), (3, 6, 2)])
def test_matmul_t_integer_brute_force(M, N, K):
    rng = np.random.default_rng(100 + M * 7 + N * 3 + K)
    DY = rng.integers(-4, 5, size=(M, N)).astype(np.float32)
    W = rng.integers(-4, 5, size=(K, N)).astype(np.float32)
    want = np.zeros((M, K))
    for i, k, n in itertools.product(range(M), range(K), range(N)):
        want[i, k] += float(DY[i, n]) * float(W[k, n])
    assert np.array_equal(oracle.matmul_t(DY, W), want)


@pytest.mark.parametrize("M,N,K", [(3, 5, 7), (8, 2, 4), (1, 9, 6)])
def test_matmul_t_is_the_adjoint_of_matmul(M, N, K):
    # sum(dY * (X @ W)) == sum(dX * X) for every X: exact on integers, and
    # non-square shapes catch a transposed operand
    rng = np.random.default_rng(7 * M + N + K)
    X = rng.integers(-5, 6, size=(M, K)).astype(np.float32)
    W = rng.integers(-5, 6, size=(K, N)).astype(np.float32)
    DY = rng.integers(-5, 6, size=(M, N)).astype(np.float32)
    lhs = float(np.sum(oracle.matmul(X, W) * DY))
    rhs = float(np.sum(oracle.matmul_t(DY, W) * X))
    assert lhs == rhs
    # and it is the only such map: unit X picks out single entries
    dX = oracle.matmul_t(DY, W)
    for i, k in [(0, 0), (M - 1, K - 1), (M // 2, K // 2)]:
        E = np.zeros((M, K), dtype=np.float32)
        E[i, k] = 1.0
        assert float(np.sum(oracle.matmul(E, W) * DY)) == dX[i, k]


def test_matmul_t_acc_and_w16():
    rng = np.random.default_rng(11)
    DY = rng.integers(-4, 5, size=(4, 8)).astype(np.float32)
    Wf = rng.integers(-4, 5, size=(6, 8)).astype(np.float32)
    D0 = rng.integers(-64, 65, size=(4, 6)).astype(np.float32)
    assert np.array_equal(oracle.matmul_t_acc(DY, Wf, D0) - oracle.matmul_t(DY, Wf),
                          D0.astype(np.float64))
    # binary16 weights decoded by numpy's own float16 type
    W16 = (rng.standard_normal((6, 8)) * 0.3).astype(np.float16)
    bits = W16.view(np.uint16)
    want = np.zeros((4, 6))
    for i, k, n in itertools.product(range(4), range(6), range(8)):
        want[i, k] += float(DY[i, n]) * float(W16[k, n])
    np.testing.assert_allclose(oracle.matmul_t_w16(DY, bits), want, rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(oracle.matmul_t_acc_w16(DY, bits, D0), want + D0,
                               rtol=1e-15, atol=1e-15)
    with pytest.raises(ValueError):
        oracle.matmul_t(DY, Wf.T)
    with pytest.raises(ValueError):
        oracle.matmul_t_acc(DY, Wf, D0.T)


def test_reference_t_forms():
    rng = np.random.default_rng(5)
    d = {"DY": rng.standard_normal((5, 8)).astype(np.float32),
         "W": rng.standard_normal((3, 8)).astype(np.float32),
         "R": rng.standard_normal((5, 3)).astype(np.float32)}
    d["DY"][2] = 0.0                      # a zero row accumulates nothing
    Y, S = oracle.reference("matmul_t_acc", d)
    assert Y.shape == S.shape == (5, 3)
    assert np.all(S + 1e-12 >= np.abs(Y - d["R"]))      # |sum| <= sum of |terms|
    assert np.all(S[2] == 0.0) and np.array_equal(Y[2], d["R"][2].astype(np.float64))
    Ysub, Ssub = oracle.reference("matmul_t_acc", d, rows=[4, 1])
    assert np.array_equal(Ysub, Y[[4, 1]]) and np.array_equal(Ssub, S[[4, 1]])


# ---------------------------------------------------------------- backward: dW = X^T @ dY

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 2, 5), (5, 4, 1), (2, 6, 3)])
def test_matmul_at_integer_brute_force(M, N, K):
    rng = np.random.default_rng(200 + M * 7 + N * 3 + K)
    X = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    DY = rng.integers(-4, 5, size=(M, N)).astype(np.float32)
    want = np.zeros((K, N))
    for k, n, m in itertools.product(range(K), range(N), range(M)):
        want[k, n] += float(X[m, k]) * float(DY[m, n])
    assert np.array_equal(oracle.matmul_at(X, DY), want)


@pytest.mark.parametrize("M,N,K", [(3, 5, 7), (9, 2, 4), (6, 8, 1)])
def test_matmul_at_is_the_adjoint_in_w(M, N, K):
    # sum(dY * (X @ W)) == sum(dW * W) for every W, exactly on integers; unit
    # W pick out single entries of dW
    rng = np.random.default_rng(13 * M + N + K)
    X = rng.integers(-5, 6, size=(M, K)).astype(np.float32)
    W = rng.integers(-5, 6, size=(K, N)).astype(np.float32)
    DY = rng.integers(-5, 6, size=(M, N)).astype(np.float32)
    dW = oracle.matmul_at(X, DY)
    assert float(np.sum(oracle.matmul(X, W) * DY)) == float(np.sum(dW * W))
    for k, n in [(0, 0), (K - 1, N - 1), (K // 2, N // 2)]:
        E = np.zeros((K, N), dtype=np.float32)
        E[k, n] = 1.0
        assert float(np.sum(oracle.matmul(X, E) * DY)) == dW[k, n]


def test_matmul_at_acc_and_reference_rows():
    rng = np.random.default_rng(17)
    d = {"X": rng.integers(-4, 5, size=(6, 5)).astype(np.float32),
         "DY": rng.integers(-4, 5, size=(6, 3)).astype(np.float32),
         "R": rng.integers(-64, 65, size=(5, 3)).astype(np.float32)}
    Y, S = oracle.reference("matmul_at_acc", d)
    assert np.array_equal(Y - oracle.matmul_at(d["X"], d["DY"]), d["R"].astype(np.float64))
    assert np.all(S >= np.abs(Y - d["R"]))
    Ysub, Ssub = oracle.reference("matmul_at_acc", d, rows=[4, 0])
    assert np.array_equal(Ysub, Y[[4, 0]]) and np.array_equal(Ssub, S[[4, 0]])
    with pytest.raises(ValueError):
        oracle.matmul_at(d["X"], d["DY"][:5])


def test_matmul_at_swiglu_a_is_the_adjoint_of_the_swiglu_form():
    # GATE >= 40: sigma(GATE) == 1.0 in float64, so A = GATE * UP exactly and
    # the identity sum(dY * Y(W)) == sum(dW * W) holds exactly (R = 0)
    rng = np.random.default_rng(23)
    M, N, K = 7, 5, 6
    G = rng.integers(40, 61, size=(M, K)).astype(np.float32)
    U = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    W = rng.integers(-4, 5, size=(K, N)).astype(np.float32)
    DY = rng.integers(-4, 5, size=(M, N)).astype(np.float32)
    Y = oracle.matmul_residual_swiglu_a(G, U, W, np.zeros((M, N), dtype=np.float32))
    dW = oracle.matmul_at_swiglu_a(G, U, DY)
    assert float(np.sum(Y * DY)) == float(np.sum(dW * W))
    want = np.zeros((K, N))
    for k, n, m in itertools.product(range(K), range(N), range(M)):
        want[k, n] += float(G[m, k]) * float(U[m, k]) * float(DY[m, n])
    assert np.array_equal(dW, want)
    D0 = rng.integers(-64, 65, size=(K, N)).astype(np.float32)
    assert np.array_equal(oracle.matmul_at_swiglu_a_acc(G, U, DY, D0) - dW, D0.astype(np.float64))


# ---------------------------------------------------------------- SwiGLU backward (09_backward_ffn)

def test_silu_derivative_closed_forms_and_identities():
    # silu'(0) = 1/2; sigma(ln 3) = 3/4 gives silu'(ln 3) = 3/4 (1 + ln(3)/4)
    assert oracle.silu_derivative(np.array([0.0]))[0] == 0.5
    assert math.isclose(oracle.silu_derivative(np.array([math.log(3.0)]))[0],
                        0.75 * (1.0 + math.log(3.0) / 4.0), rel_tol=1e-15)
    # silu'(x) + silu'(-x) = 1, and a central difference of silu agrees
    x = np.linspace(-30.0, 30.0, 601)
    np.testing.assert_allclose(oracle.silu_derivative(x) + oracle.silu_derivative(-x), 1.0,
                               rtol=0, atol=1e-13)   # fp64 rounding of x*s*(1-s), |x| <= 30
    h = 1e-6
    fd = (oracle.silu(x + h) - oracle.silu(x - h)) / (2 * h)
    np.testing.assert_allclose(oracle.silu_derivative(x), fd, rtol=0, atol=1e-8)
    # far out: silu' -> 1 for large x, -> 0 (from below) for very negative x
    assert oracle.silu_derivative(np.array([100.0]))[0] == 1.0
    assert abs(oracle.silu_derivative(np.array([-100.0]))[0]) < 1e-40


def test_nan_guard_is_the_pages_finite_check():
    f32max = float(np.finfo(np.float32).max)
    x = np.array([np.nan, np.inf, -np.inf, f32max, -f32max, 3.4e38, -1e-45, 0.0, 2.5])
    assert np.array_equal(oracle.nan_guard(x), [0, 0, 0, 0, 0, 3.4e38, -1e-45, 0.0, 2.5])


def test_ffn_swiglu_backward_values():
    # large gates: sigma == 1 in float64, so silu = gate, silu' = 1 exactly
    G = np.array([[3.0, -2.0, 0.5]])
    gate = np.array([[40.0, 50.0, 60.0]])
    up = np.array([[2.0, -3.0, 4.0]])
    dg, du = oracle.ffn_swiglu_backward(G, gate, up)
    assert np.array_equal(dg, G * up) and np.array_equal(du, G * gate)
    # gate 0: silu(0) = 0, silu'(0) = 1/2
    dg, du = oracle.ffn_swiglu_backward(np.array([4.0]), np.array([0.0]), np.array([3.0]))
    assert dg[0] == 6.0 and du[0] == 0.0
    # non-finite inputs and overflowing products are guarded to 0
    dg, du = oracle.ffn_swiglu_backward(np.array([1.0, 1.0, 1e30]), np.array([np.nan, np.inf, 1e10]),
                                        np.array([1.0, 1.0, 1e10]))
    assert np.array_equal(dg, [0.0, 0.0, 0.0]) and np.array_equal(du, [0.0, 0.0, 0.0])


def test_matmul_t_swiglu_backward_composes_the_pages_steps():
    # the fused form is the pages' element-wise backward applied to dY @ W^T
    # (two steps the tests above pin separately); brute force on integers
    rng = np.random.default_rng(31)
    DY = rng.integers(-4, 5, size=(3, 5)).astype(np.float32)
    W = rng.integers(-4, 5, size=(4, 5)).astype(np.float32)
    gate = rng.integers(40, 61, size=(3, 4)).astype(np.float32)
    up = rng.integers(-4, 5, size=(3, 4)).astype(np.float32)
    dg, du = oracle.matmul_t_swiglu_backward(DY, W, gate, up)
    for i, k in itertools.product(range(3), range(4)):
        dA = sum(float(DY[i, n]) * float(W[k, n]) for n in range(5))
        assert dg[i, k] == dA * float(up[i, k]) and du[i, k] == dA * float(gate[i, k])


# ---------------------------------------------------------------- cross-entropy (07_loss)

def test_cross_entropy_closed_forms():
    V = 8
    # uniform logits: p = 1/V, loss = log V; ignored target: loss 0, gradient 0
    losses, dl = oracle.cross_entropy(np.zeros((2, V)), [3, V + 1])
    assert math.isclose(losses[0], math.log(V), rel_tol=1e-15) and losses[1] == 0.0
    np.testing.assert_allclose(dl[0], np.full(V, 1.0 / V) - np.eye(V)[3], rtol=0, atol=1e-16)
    assert np.all(dl[1] == 0.0)
    # a dominant target logit: loss -> 0; shifting every logit changes nothing
    L = np.zeros((1, V))
    L[0, 5] = 60.0
    assert oracle.cross_entropy(L, [5])[0][0] < 1e-25
    a, b = oracle.cross_entropy(L + 1000.0, [5])
    c, d = oracle.cross_entropy(L, [5])
    assert math.isclose(a[0], c[0], abs_tol=1e-12) and np.allclose(b, d, atol=1e-15)
    # label smoothing and z-loss terms, by hand: uniform logits l = 2
    l, _ = oracle.cross_entropy(np.full((1, V), 2.0), [0], alpha=0.1, beta=0.01)
    lse = 2.0 + math.log(V)
    assert math.isclose(l[0], lse - 0.9 * 2.0 - 0.1 * 2.0 + 0.01 * lse * lse, rel_tol=1e-14)


@pytest.mark.parametrize("alpha,beta", [(0.0, 0.0), (0.1, 0.0), (0.0, 1e-3), (0.2, 1e-2)])
def test_cross_entropy_gradient_is_the_loss_derivative(alpha, beta):
    # dLogits / inv_norm is d loss / d logits: central differences agree, and
    # each row's gradient sums to 2 beta LSE inv_norm
    rng = np.random.default_rng(9)
    L = rng.standard_normal((3, 7)) * 3.0
    t = [0, 4, 6]
    losses, dl = oracle.cross_entropy(L, t, alpha, beta, inv_norm=0.5)
    h = 1e-6
    for s, v in [(0, 0), (1, 3), (2, 6), (2, 2)]:
        Lp, Lm = L.copy(), L.copy()
        Lp[s, v] += h
        Lm[s, v] -= h
        fd = (oracle.cross_entropy(Lp, t, alpha, beta)[0][s] -
              oracle.cross_entropy(Lm, t, alpha, beta)[0][s]) / (2 * h)
        assert math.isclose(dl[s, v] / 0.5, fd, rel_tol=1e-6, abs_tol=1e-8)
    for s in range(3):
        mx = np.max(L[s])
        lse = mx + math.log(np.sum(np.exp(L[s] - mx)))
        assert math.isclose(float(np.sum(dl[s])), 2 * beta * lse * 0.5, abs_tol=1e-12)


def test_gate_up_brute_force():
    rng = np.random.default_rng(41)
    X = rng.integers(-4, 5, size=(3, 5)).astype(np.float32)
    wg = (rng.standard_normal((5, 4)) * 0.5).astype(np.float16)
    wu = (rng.standard_normal((5, 4)) * 0.5).astype(np.float16)
    G, U = oracle.gate_up_w16(X, wg.view(np.uint16), wu.view(np.uint16))
    for i, n in itertools.product(range(3), range(4)):
        assert G[i, n] == sum(float(X[i, k]) * float(wg[k, n]) for k in range(5))
        assert U[i, n] == sum(float(X[i, k]) * float(wu[k, n]) for k in range(5))


# ---------------------------------------------------------------- hand-worked fixtures of the
# widened rows: the SwiGLU-backward normalisers and the loss total

def test_golden_swiglu_backward_and_normalisers():
    # tests/golden/swiglu_backward_1x2x4.txt: sigma(+-ln 3), gate 0 and
    # gate 40 worked by hand, including the normalisers S_dGATE, S_dUP that
    # widen the acceptance bound of the fused SwiGLU backward
    g = read_blocks("swiglu_backward_1x2x4.txt")
    W16 = g["W"].astype(np.float16).view(np.uint16)
    for form, w in (("matmul_t_swiglu_backward", {"W": g["W"].astype(np.float32)}),
                    ("matmul_t_swiglu_backward_w16", {"W16": W16})):
        d = {"DY": g["DY"].astype(np.float32), "GATE": g["GATE"], "UP": g["UP"], **w}
        (dgate, dup), (Sg, Su) = oracle.reference(form, d)
        for got, want in ((dgate, g["DGATE"]), (dup, g["DUP"]), (Sg, g["SG"]), (Su, g["SU"])):
            np.testing.assert_allclose(got, want, rtol=4e-15, atol=0, err_msg=form)
    # the direct function gives the same gradients
    dgate, dup = oracle.matmul_t_swiglu_backward(g["DY"], g["W"], g["GATE"], g["UP"])
    np.testing.assert_allclose(dgate, g["DGATE"], rtol=4e-15, atol=0)
    np.testing.assert_allclose(dup, g["DUP"], rtol=4e-15, atol=0)


def test_golden_lm_head_cross_entropy_total():
    # tests/golden/cross_entropy_total.txt: per-row losses and their SUM
    # (page 07_loss, "sum_losses"), with and without smoothing and z-loss
    X = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]], dtype=np.float32)
    W16 = np.array([[0x0000] * 4, [0x3C00, 0, 0, 0]], dtype=np.uint16)
    targets = [1, 0, 7]
    for alpha, beta, l0, l1, l2, total in (map(float, r) for r in
                                           read_rows("cross_entropy_total.txt")):
        losses, dl, got_total = oracle.lm_head_cross_entropy_w16(X, W16, targets, alpha, beta)
        np.testing.assert_allclose(losses, [l0, l1, l2], rtol=1e-15, atol=0)
        assert math.isclose(got_total, total, rel_tol=1e-15), (alpha, beta, got_total, total)
        assert np.all(dl[2] == 0.0)            # the ignored row has no gradient
