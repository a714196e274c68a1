"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

* exact: small-integer inputs make every operand rounding and partial sum
  exact, so the GPU result must equal the oracle bit for bit;
* tolerance: random inputs of the workload generator, normalised error
  max |Y - Y_ref| / sum_k |A W| <= 4e-3 (the acceptance bound), on shapes
  that span several tiles and a ragged tail in M, N and K;
* the five named workloads at full size (the 16k-token SwiGLU one on a
  sample of rows that includes the first and last rows of several tiles).
"""

import numpy as np
import pytest

from tests.gpu_util import (TOL, integer_inputs, oracle_error, require_gpu, run_device,
                            to_device)
import oracle
from transformer_linear_layer_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F32_FORMS = ("matmul", "matmul_residual", "matmul_residual_swiglu_a")
W16_FORMS = ("matmul_w16", "matmul_residual_w16", "matmul_residual_swiglu_a_w16")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


# (M, N, K): several tiles plus ragged tails; N % 8 == 0 so the w16 forms run too.
# The last two split K across CTAs when tiles are few (per-tile kernel: 2 and
# 8 K ranges on a 152-SM GB300): for the f32 forms that read X the CTAs of
# a tile form a cluster and sum their partial tiles through distributed
# shared memory (ragged rows and columns included); the SwiGLU forms' partial
# tiles go to the workspace and the split-sum kernel.
EXACT_SHAPES = [(256, 256, 128), (129, 136, 20), (1, 8, 4), (300, 264, 68), (128, 392, 256),
                (257, 136, 1028)]


@pytest.mark.parametrize("form", wl.FORWARD_FORMS)
@pytest.mark.parametrize("shape", EXACT_SHAPES)
def test_exact_small_integers(form, shape):
    M, N, K = shape
    d = integer_inputs(form, M, N, K, seed=M + 7 * N + 13 * K)
    Y = run_device(form, to_device(d), M, N).cpu().numpy().astype(np.float64)
    Yref, _ = oracle.reference(form, d)
    assert np.array_equal(Y, Yref), f"max |diff| = {np.max(np.abs(Y - Yref))}"


# Persistent launches that split the last partial round along K (clustered
# kernels, binary16 forms): each tail tile's K ranges leave f32 partial
# tiles that the warp completing a quadrant adds up in K order. On a GB300
# with 36 resident clusters of four, the first shape splits its 6 tiles 4
# ways with no whole round before; the second runs two whole rounds, then
# splits its last 2 tiles 2 ways.
SPLIT_SHAPES = [(300, 2048, 2048), (4736, 2048, 1024)]


@pytest.mark.parametrize("form", W16_FORMS)
@pytest.mark.parametrize("shape", SPLIT_SHAPES)
def test_split_tail_exact(form, shape):
    M, N, K = shape
    d = integer_inputs(form, M, N, K, seed=M + N + K)
    Y = run_device(form, to_device(d), M, N).cpu().numpy().astype(np.float64)
    Yref, _ = oracle.reference(form, d)
    assert np.array_equal(Y, Yref), f"max |diff| = {np.max(np.abs(Y - Yref))}"


@pytest.mark.parametrize("form", W16_FORMS)
def test_split_tail_random_reproducible(form):
    import torch
    M, N, K = SPLIT_SHAPES[0]
    d = wl.generate(form, M, N, K, seed=23, outlier_frac=0.01)
    dd = to_device(d)
    Y1 = run_device(form, dd, M, N)
    Y2 = run_device(form, dd, M, N)
    assert torch.equal(Y1, Y2)
    err = oracle_error(form, d, Y1.cpu().numpy())
    assert err <= TOL, err


RANDOM_SHAPES = [(300, 392, 200), (257, 136, 1028), (64, 1024, 96), (513, 264, 516)]


@pytest.mark.parametrize("form", wl.FORWARD_FORMS)
@pytest.mark.parametrize("shape", RANDOM_SHAPES)
def test_random_within_bound(form, shape):
    M, N, K = shape
    d = wl.generate(form, M, N, K, seed=17 + M + N + K, outlier_frac=0.01)
    Y = run_device(form, to_device(d), M, N).cpu().numpy()
    err = oracle_error(form, d, Y)
    assert err <= TOL, err


@pytest.mark.parametrize("w", wl.WORKLOADS, ids=lambda w: w.name)
def test_named_workload(w):
    d = wl.generate_workload(w)
    Y = run_device(w.form, to_device(d), w.M, w.N).cpu().numpy()
    if w.M * w.N * w.K > 2 ** 34:
        # full-size SwiGLU down projection: the oracle evaluates a sample of
        # rows (each output row depends only on the same input row)
        rng = np.random.default_rng(w.seed)
        edges = [0, 1, 127, 128, 129, 255, 8191, 8192, w.M - 129, w.M - 128, w.M - 1]
        rows = np.unique(np.concatenate([edges, rng.choice(w.M, 245, replace=False)]))
        err = oracle_error(w.form, d, Y[rows], rows=rows)
        assert np.all(np.isfinite(Y))
    else:
        err = oracle_error(w.form, d, Y)
    print(f"{w.name}: normalised error {err:.3e}")
    assert err <= TOL, err


def test_swiglu_outliers_exercise_both_sigmoid_branches():
    # GATE entries far out on both sides (|g| up to 1000): the stable sigmoid
    # must neither overflow nor produce NaN, and the result stays in bound.
    for form in ("matmul_residual_swiglu_a", "matmul_residual_swiglu_a_w16"):
        M, N, K = 130, 72, 96
        d = wl.generate(form, M, N, K, seed=99)
        g = d["GATE"]
        g[::7, ::5] = 1000.0
        g[3::7, 1::5] = -1000.0
        g[5::11, 2::3] = -88.0
        Y = run_device(form, to_device(d), M, N).cpu().numpy()
        assert np.all(np.isfinite(Y))
        assert oracle_error(form, d, Y) <= TOL
