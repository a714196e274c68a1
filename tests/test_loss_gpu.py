"""lm_head + the fused cross-entropy of page 07_loss
(lin_lm_head_cross_entropy_w16) on the GPU against the oracle.

The logits part is the matmul_w16 GEMM the other parity tests cover, so the
loss part is checked twice: against the oracle's cross-entropy of the very
logits the GEMM produced (lin_matmul_w16 on the same inputs, the same
kernel without a split, so the same bits), tightly; and end to end against
the fp64 oracle of X @ W16, within what the logits' bound allows.
"""

import math

import numpy as np
import pytest

import oracle
from tests.gpu_util import require_gpu
from transformer_linear_layer_tcgen05_gb300 import lin
from transformer_linear_layer_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _inputs(M, V, K, seed):
    d = wl.generate("matmul_w16", M, V, K, seed=seed, w_var=0.02)
    rng = np.random.default_rng(seed)
    t = rng.integers(0, V, size=M).astype(np.int32)
    t[::7] = -1            # padding rows: ignored
    if M > 3:
        t[3] = V + 5       # beyond the vocabulary: ignored
    return d["X"], d["W16"], t


def _fused(X, W16, t, alpha, beta, inv_norm):
    import torch
    M, V = X.shape[0], W16.shape[1]
    Xd = torch.from_numpy(X).cuda()
    Wd = torch.from_numpy(W16.view(np.int16)).cuda()
    td = torch.from_numpy(t).cuda()
    DL = torch.full((M, V), float("nan"), device="cuda")
    losses = torch.full((M,), float("nan"), device="cuda")
    total = torch.full((1,), float("nan"), device="cuda")
    lin.lin_lm_head_cross_entropy_w16(Xd, Wd, td, DL, losses, total, alpha, beta, inv_norm)
    torch.cuda.synchronize()
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    logits = torch.empty((M, V), device="cuda")
    lin.lin_matmul_w16(Xd, Wd, logits)
    torch.cuda.synchronize()
    return (DL.cpu().numpy().astype(np.float64), losses.cpu().numpy().astype(np.float64),
            float(total.item()), logits.cpu().numpy().astype(np.float64))


# (M, V, K): ragged rows, a vocabulary that is not a multiple of 256 or of a
# cluster's 1024 columns, the lm_head shape of the pages (512 x 16384 x 768),
# and rows longer than the loss kernel stages at once (16384 logits: the
# rest is read chunk by chunk)
SHAPES = [(129, 1032, 64), (300, 2048, 768), (64, 4096, 256), (512, 16384, 768),
          (64, 20488, 128)]
PARAMS = [(0.0, 0.0, 1.0), (0.1, 0.0, 1.0 / 300), (0.0, 1e-4, 0.5), (0.05, 1e-3, 1.0)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("alpha,beta,inv_norm", PARAMS)
def test_loss_of_the_gemm_logits(shape, alpha, beta, inv_norm):
    M, V, K = shape
    X, W16, t = _inputs(M, V, K, seed=M + V)
    DL, losses, total, logits = _fused(X, W16, t, alpha, beta, inv_norm)
    ref_losses, ref_dl = oracle.cross_entropy(logits, t, alpha, beta, inv_norm)
    np.testing.assert_allclose(losses, ref_losses, rtol=2e-5, atol=2e-5)
    np.testing.assert_allclose(DL, ref_dl, rtol=2e-4, atol=2e-7 * max(inv_norm, 1e-3) + 1e-9)
    assert math.isclose(total, float(np.sum(losses)), rel_tol=1e-5, abs_tol=1e-4)
    ignored = (t < 0) | (t >= V)
    assert np.all(losses[ignored] == 0.0) and np.all(DL[ignored] == 0.0)
    # each valid row's gradient sums to 2 beta LSE inv_norm
    for s in np.nonzero(~ignored)[0][:8]:
        row = logits[s]
        mx = row.max()
        lse = mx + math.log(np.sum(np.exp(row - mx)))
        assert abs(DL[s].sum() - 2 * beta * lse * inv_norm) < 1e-4 * max(inv_norm, 1e-2)


@pytest.mark.parametrize("shape", [(300, 2048, 768), (512, 16384, 768)])
def test_end_to_end_against_the_fp64_oracle(shape):
    M, V, K = shape
    X, W16, t = _inputs(M, V, K, seed=7 * M)
    DL, losses, total, _ = _fused(X, W16, t, 0.1, 1e-4, 1.0 / M)
    ref_losses, ref_dl, ref_total = oracle.lm_head_cross_entropy_w16(X, W16, t, 0.1, 1e-4, 1.0 / M)
    # the logits carry the GEMM's error (normalised bound 4e-3 of S = |X||W|,
    # measured far below it); the loss moves by at most a few times the
    # largest logit error of its row
    S = np.abs(X.astype(np.float64)) @ np.abs(W16.view(np.float16).astype(np.float64))
    dmax = 4e-3 * S.max(axis=1)
    assert np.all(np.abs(losses - ref_losses) <= 4 * dmax + 1e-5)
    assert abs(total - ref_total) <= 4 * dmax.sum() + 1e-3
    assert np.max(np.abs(DL - ref_dl)) <= 1e-2 / M


def test_no_contraction_gives_uniform_softmax():
    # K == 0: every logit is 0 (no partials from the GEMM: the loss kernel
    # reads the row itself), so every valid row's loss is log V
    import torch
    M, V = 40, 1024
    X = torch.empty((M, 0), device="cuda")
    W = torch.empty((0, V), dtype=torch.int16, device="cuda")
    t = torch.arange(M, dtype=torch.int32, device="cuda")
    t[5] = -1
    DL = torch.empty((M, V), device="cuda")
    losses = torch.empty((M,), device="cuda")
    total = torch.empty((1,), device="cuda")
    lin.lin_lm_head_cross_entropy_w16(X, W, t, DL, losses, total)
    torch.cuda.synchronize()
    want = np.full(M, math.log(V))
    want[5] = 0.0
    np.testing.assert_allclose(losses.cpu().numpy(), want, rtol=1e-6)
    # one kernel: the loss, whose last CTA also adds the losses (the GEMM
    # only zeroes the logits, and a memset the loss kernel's count of rows)
    assert lin.lin_last_launch_info()[0] == 1
