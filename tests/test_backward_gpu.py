"""The backward input gradient dX = dY @ W^T (lin_matmul_t, _acc, _w16) on
the GPU against the oracle.

The backward-linear page is not part of the material; the operation is the
adjoint of the forward product (see the oracle). Shapes use the C ABI's
convention: dY [M,N], W [K,N], dX [M,K]; the contraction runs over N.
"""

import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from tests.gpu_util import TOL, integer_inputs, oracle_error, require_gpu, to_device
from transformer_linear_layer_tcgen05_gb300 import lin
from transformer_linear_layer_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

T_FORMS = wl.T_FORMS
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (M, N, K): ragged tiles, a single row, a contraction shorter than a
# k-block, and an output wide enough for clusters of four with several N
# groups (binary16 W: N % 8 == 0). The last two split K (the contraction)
# across CTAs or clusters.
SHAPES = [(128, 256, 128), (129, 136, 260), (1, 8, 4), (300, 64, 1032), (257, 1024, 2048),
          (300, 2048, 2048), (520, 512, 768)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(form, dd, M, K):
    import torch
    Y = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
    lin.run_form(form, dd, Y)
    torch.cuda.synchronize()
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    return Y


@pytest.mark.parametrize("form", T_FORMS)
@pytest.mark.parametrize("shape", SHAPES)
def test_exact_small_integers(form, shape):
    M, N, K = shape
    d = integer_inputs(form, M, N, K, seed=M + 3 * N + 5 * K)
    Y = _run(form, to_device(d), M, K).cpu().numpy().astype(np.float64)
    Yref, _ = oracle.reference(form, d)
    assert np.array_equal(Y, Yref), f"max |diff| = {np.max(np.abs(Y - Yref))}"


@pytest.mark.parametrize("form", T_FORMS)
@pytest.mark.parametrize("shape", [(300, 392, 200), (513, 264, 1024), (512, 768, 768)])
def test_random_within_bound(form, shape):
    M, N, K = shape
    d = wl.generate(form, M, N, K, seed=29 + M + N)
    Y = _run(form, to_device(d), M, K).cpu().numpy()
    assert oracle_error(form, d, Y) <= TOL


@pytest.mark.parametrize("form", T_FORMS)
def test_empty_contraction_gives_initial_or_zero(form):
    import torch
    M, N, K = 70, 0, 48
    d = to_device(wl.generate(form, M, 8, K, seed=1))
    d["DY"] = torch.empty((M, N), dtype=torch.float32, device="cuda")
    w = "W16" if form.endswith("_w16") else "W"
    d[w] = torch.empty((K, N), dtype=d[w].dtype, device="cuda")
    Y = _run(form, d, M, K)
    want = d["R"] if "R" in d else torch.zeros_like(Y)
    assert torch.equal(Y, want)


def test_adjoint_of_the_forward_kernel():
    # sum(dY * (X @ W)) == sum(dX * X) with both sides computed on the GPU,
    # exactly on small integers
    import torch
    M, N, K = 200, 136, 264
    rng = np.random.default_rng(3)
    X = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    W = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    DY = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    Xd, Wd, DYd = (torch.from_numpy(a).cuda() for a in (X, W, DY))
    Y = torch.empty((M, N), device="cuda")
    DX = torch.empty((M, K), device="cuda")
    lin.lin_matmul(Xd, Wd, Y)
    lin.lin_matmul_t(DYd, Wd, DX)
    torch.cuda.synchronize()
    lhs = float(np.sum(Y.cpu().numpy().astype(np.float64) * DY))
    rhs = float(np.sum(DX.cpu().numpy().astype(np.float64) * X))
    assert lhs == rhs


def test_acc_reads_and_writes_in_place():
    import torch
    M, N, K = 256, 512, 1024
    d = integer_inputs("matmul_t_acc_w16", M, N, K, seed=8)
    dd = to_device(d)
    DX = dd["R"].clone()
    lin.lin_matmul_t_acc_w16(dd["DY"], dd["W16"], DX)
    lin.lin_matmul_t_acc_w16(dd["DY"], dd["W16"], DX)   # twice: dX0 + 2 dY W^T
    torch.cuda.synchronize()
    once = oracle.matmul_t_w16(d["DY"], d["W16"])
    assert np.array_equal(DX.cpu().numpy().astype(np.float64), d["R"] + 2.0 * once)


CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import oracle
from tests.gpu_util import integer_inputs, require_gpu, to_device
from transformer_linear_layer_tcgen05_gb300 import lin
require_gpu()
bad = 0
for form in ("matmul_t_w16", "matmul_t_acc_w16", "matmul_t_swiglu_backward_w16"):
    for (M, N, K) in [(128, 64, 256), (300, 200, 2048), (129, 520, 1032), (1, 1032, 4),
                      (700, 1536, 1024), (4736, 1024, 2048)]:
        d = integer_inputs(form, M, N, K, seed=M + N + K)
        two = "swiglu" in form        # (dGATE, dUP)
        Yd = tuple(torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
                   for _ in range(2 if two else 1))
        lin.run_form(form, to_device(d), Yd if two else Yd[0])
        torch.cuda.synchronize()
        st = lin.lin_get_device_status()
        ref = oracle.reference(form, d)[0]
        refs = ref if two else (ref,)
        nd = sum(int(np.sum(y.cpu().numpy().astype(np.float64) != r)) for y, r in zip(Yd, refs))
        if nd or st != lin.LIN_SUCCESS:
            print(f"{form} {M}x{N}x{K}: status {st}, {nd} mismatches", flush=True)
        bad += nd + (st != lin.LIN_SUCCESS)
sys.exit(1 if bad else 0)
"""

VARIANTS = [{"LIN_F16_KERNEL": "1"}, {"LIN_F16_KERNEL": "2"}, {"LIN_F16_KERNEL": "4"},
            {"LIN_F16_KERNEL": "tile"}, {"LIN_F16_KERNEL": "4", "LIN_F16_PRECONVERT": "0"},
            {"LIN_F16_KERNEL": "1", "LIN_F16_PRECONVERT": "1"}]


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: "-".join(v.values()))
def test_w16_every_kernel_exact(variant):
    env = dict(os.environ, **variant)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-4000:]


# ---------------------------------------------------------------- weight gradient dW = X^T @ dY

AT_FORMS = wl.AT_FORMS
# (M, N, K): dW is [K,N]; the contraction runs over the M tokens, which need
# no alignment (ragged M: 1, 129, 777); the last shapes split M across CTAs
AT_SHAPES = [(128, 128, 128), (129, 136, 260), (1, 8, 4), (777, 264, 132), (512, 768, 768),
             (2048, 256, 128)]


@pytest.mark.parametrize("form", AT_FORMS)
@pytest.mark.parametrize("shape", AT_SHAPES)
def test_weight_gradient_exact_small_integers(form, shape):
    M, N, K = shape
    d = integer_inputs(form, M, N, K, seed=M + 7 * N + 3 * K)
    Y = _run(form, to_device(d), K, N).cpu().numpy().astype(np.float64)
    Yref, _ = oracle.reference(form, d)
    assert np.array_equal(Y, Yref), f"max |diff| = {np.max(np.abs(Y - Yref))}"


@pytest.mark.parametrize("form", AT_FORMS)
@pytest.mark.parametrize("shape", [(300, 392, 200), (512, 3072, 768)])
def test_weight_gradient_random_within_bound(form, shape):
    M, N, K = shape
    d = wl.generate(form, M, N, K, seed=41 + M + N)
    Y = _run(form, to_device(d), K, N).cpu().numpy()
    assert oracle_error(form, d, Y) <= TOL


def test_weight_gradient_is_the_adjoint_in_w():
    # sum(dY * (X @ W)) == sum(dW * W), both products computed on the GPU
    import torch
    M, N, K = 300, 136, 264
    rng = np.random.default_rng(4)
    X = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    W = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    DY = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    Xd, Wd, DYd = (torch.from_numpy(a).cuda() for a in (X, W, DY))
    Y = torch.empty((M, N), device="cuda")
    DW = torch.empty((K, N), device="cuda")
    lin.lin_matmul(Xd, Wd, Y)
    lin.lin_matmul_at(Xd, DYd, DW)
    torch.cuda.synchronize()
    lhs = float(np.sum(Y.cpu().numpy().astype(np.float64) * DY))
    rhs = float(np.sum(DW.cpu().numpy().astype(np.float64) * W))
    assert lhs == rhs


def test_weight_gradient_accumulates_over_micro_batches():
    # dW over two halves of the tokens, accumulated in place, equals dW over
    # all tokens (exact on small integers)
    import torch
    M, N, K = 512, 256, 384
    d = integer_inputs("matmul_at", M, N, K, seed=12)
    X, DY = (torch.from_numpy(d[k]).cuda() for k in ("X", "DY"))
    DW = torch.zeros((K, N), device="cuda")
    for h in range(2):
        rows = slice(h * M // 2, (h + 1) * M // 2)
        lin.lin_matmul_at_acc(X[rows].contiguous(), DY[rows].contiguous(), DW)
    torch.cuda.synchronize()
    assert np.array_equal(DW.cpu().numpy().astype(np.float64), oracle.matmul_at(d["X"], d["DY"]))


def test_swiglu_weight_gradient_is_the_adjoint_of_the_forward_kernel():
    # sum(dY * (silu(G)*U) @ W) == sum(dW_down * W), both sides on the GPU;
    # GATE >= 40 keeps every value an exact small integer in TF32
    import torch
    M, N, K = 333, 136, 264
    rng = np.random.default_rng(6)
    G = rng.integers(40, 61, size=(M, K)).astype(np.float32)
    U = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    W = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    DY = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    Gd, Ud, Wd, DYd = (torch.from_numpy(a).cuda() for a in (G, U, W, DY))
    Y = torch.empty((M, N), device="cuda")
    DW = torch.empty((K, N), device="cuda")
    lin.lin_matmul_residual_swiglu_a(Gd, Ud, Wd, torch.zeros((M, N), device="cuda"), Y)
    lin.lin_matmul_at_swiglu_a(Gd, Ud, DYd, DW)
    torch.cuda.synchronize()
    lhs = float(np.sum(Y.cpu().numpy().astype(np.float64) * DY))
    rhs = float(np.sum(DW.cpu().numpy().astype(np.float64) * W))
    assert lhs == rhs


# ---------------------------------------------------------------- fused SwiGLU backward

SWB_FORMS = wl.SWIGLU_BWD_FORMS


def _run_swb(form, dd, M, K):
    import torch
    DG = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
    DU = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
    lin.run_form(form, dd, (DG, DU))
    torch.cuda.synchronize()
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    return DG.cpu().numpy().astype(np.float64), DU.cpu().numpy().astype(np.float64)


# (M, N, K): dA = dY[M,N] @ W[K,N]^T is [M,K]; the last two split the
# contraction (per-tile split K for the f32 form, the split tail of the
# clustered kernel for binary16 W)
SWB_SHAPES = [(128, 256, 128), (129, 136, 260), (1, 8, 4), (300, 64, 1032), (300, 2048, 2048),
              (777, 512, 768)]


@pytest.mark.parametrize("form", SWB_FORMS)
@pytest.mark.parametrize("shape", SWB_SHAPES)
def test_swiglu_backward_exact_small_integers(form, shape):
    M, N, K = shape
    d = integer_inputs(form, M, N, K, seed=5 * M + N + 3 * K)
    DG, DU = _run_swb(form, to_device(d), M, K)
    (rg, ru), _ = oracle.reference(form, d)
    assert np.array_equal(DG, rg), f"dGATE max |diff| = {np.max(np.abs(DG - rg))}"
    assert np.array_equal(DU, ru), f"dUP max |diff| = {np.max(np.abs(DU - ru))}"


@pytest.mark.parametrize("form", SWB_FORMS)
@pytest.mark.parametrize("shape", [(300, 392, 200), (512, 768, 3072), (1100, 2048, 1024)])
def test_swiglu_backward_random_within_bound(form, shape):
    M, N, K = shape
    d = wl.generate(form, M, N, K, seed=53 + M + N, outlier_frac=0.01)
    DG, DU = _run_swb(form, to_device(d), M, K)
    (rg, ru), (sg, su) = oracle.reference(form, d)
    # Underflow: the pages let exp() of a very negative gate resolve to 0
    # (09_backward_ffn, note 2), so a gradient below binary32's smallest
    # subnormal (2**-149) may come out as 0 or as that subnormal: the
    # comparison allows one subnormal step on top of the relative bound.
    tiny = 2.0 ** -149
    for Y, ref, S in ((DG, rg, sg), (DU, ru, su)):
        assert np.all(np.isfinite(Y))
        nz = S > 0
        dev = np.maximum(np.abs(Y - ref) - tiny, 0.0)
        err = float(np.max(dev[nz] / S[nz])) if np.any(nz) else 0.0
        assert err <= TOL, err
        assert np.all(dev[~nz] == 0.0)


@pytest.mark.parametrize("form", SWB_FORMS)
def test_swiglu_backward_guards_non_finite_values(form):
    # NaN and infinite gates give NaN products, which nan_guard turns into 0;
    # the other elements are untouched
    M, N, K = 130, 64, 136
    d = integer_inputs(form, M, N, K, seed=2)
    d["GATE"][3, 5] = np.nan
    d["GATE"][7, 9] = np.inf
    d["GATE"][11, 13] = -np.inf
    DG, DU = _run_swb(form, to_device(d), M, K)
    (rg, ru), _ = oracle.reference(form, d)
    assert np.array_equal(DG, rg) and np.array_equal(DU, ru)
    for i, k in ((3, 5), (7, 9)):
        assert DG[i, k] == 0.0 and DU[i, k] == 0.0
