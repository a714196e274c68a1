"""The checked build (liblin_checked.so: the kernels compiled with
LIN_DEVICE_CHECKS=1 check their shared-memory stages and buffers, TMEM
columns, TMA coordinate alignment, cluster peer ranks and non-TMA global
indices, and report LIN_ERROR_DEVICE_CHECK instead of making a bad access)
run over every entry point and kernel variant on ragged shapes: every
result bit-exact against the oracle on small-integer inputs and no check
failing. This stands in for an external memory checker, which the GPUs here
do not offer. The check record itself is exercised by its self-test, which
reports a failure without touching memory."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_device_check_record_self_test():
    from tests.gpu_util import require_gpu
    from transformer_linear_layer_tcgen05_gb300 import lin
    require_gpu()
    assert lin.lin_selftest_device_check(123456789) == lin.LIN_ERROR_DEVICE_CHECK
    assert lin.lin_last_device_check() == (99, 123456789)
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS   # read and cleared


CHILD = r"""
import sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import torch
import oracle
from transformer_linear_layer_tcgen05_gb300 import build, lin
from transformer_linear_layer_tcgen05_gb300 import workloads as wl
build.build_library(checked=True)
assert lin.LIB_PATH.endswith("liblin_checked.so"), lin.LIB_PATH
from tests.gpu_util import integer_inputs, run_device, to_device
from tests.test_gate_up_gpu import _int_inputs, _run
bad = 0

def report(what, nd):
    global bad
    st = lin.lin_get_device_status()
    if nd or st != lin.LIN_SUCCESS:
        print(f"{what}: status {lin.STATUS.get(st, st)} {lin.lin_last_device_check()}, "
              f"{nd} mismatches", flush=True)
    bad += nd + (st != lin.LIN_SUCCESS)

def exact(form, M, N, K):
    d = integer_inputs(form, M, N, K, seed=M + 3 * N + 5 * K)
    dd = to_device(d)
    if wl.form_is_swiglu_bwd(form):
        Y = (torch.full((M, K), float("nan"), device="cuda"),
             torch.full((M, K), float("nan"), device="cuda"))
        lin.run_form(form, dd, Y)
        torch.cuda.synchronize()
        (rg, ru), _ = oracle.reference(form, d)
        nd = int(np.sum(Y[0].cpu().numpy() != rg)) + int(np.sum(Y[1].cpu().numpy() != ru))
    else:
        shape = wl.output_shape(form, M, N, K)
        Y = torch.full(shape, float("nan"), device="cuda")
        lin.run_form(form, dd, Y)
        torch.cuda.synchronize()
        Yref, _ = oracle.reference(form, d)
        nd = int(np.sum(Y.cpu().numpy().astype(np.float64) != Yref))
    report(f"{form} {M}x{N}x{K}", nd)

# forward and backward forms: ragged tiles, a single row, splits of the
# per-tile kernel (cluster sum and workspace), persistent clusters with a
# split tail, pre-converted binary16 A (single CTAs and CTA pairs)
SHAPES = [(129, 136, 68), (1, 8, 4), (300, 264, 256), (257, 136, 1028), (300, 2048, 2048),
          (700, 1536, 1024)]
for form in wl.FORMS:
    for (M, N, K) in SHAPES:
        if form.startswith("matmul_at") and M * N * K > 2e8:
            continue
        exact(form, M, N, K)
for (M, N, K) in [(129, 136, 64), (300, 2048, 200), (513, 8192, 512)]:
    X, WG, WU = _int_inputs(M, N, K, seed=M + N + K)
    G, U = _run(X, WG, WU)
    rg, ru = oracle.gate_up_w16(X, WG, WU)
    report(f"gate_up {M}x{N}x{K}", int(np.sum(G != rg)) + int(np.sum(U != ru)))
# the loss path (GEMM partials, the loss kernel's staged row, its in-kernel sum)
M, V, K = 64, 20488, 128
d = wl.generate("matmul_w16", M, V, K, seed=5, w_var=0.02)
t = np.random.default_rng(5).integers(0, V, size=M).astype(np.int32)
t[::7] = -1
Xd = torch.from_numpy(d["X"]).cuda()
Wd = torch.from_numpy(d["W16"].view(np.int16)).cuda()
DL = torch.empty((M, V), device="cuda")
losses = torch.empty((M,), device="cuda")
total = torch.empty((1,), device="cuda")
lin.lin_lm_head_cross_entropy_w16(Xd, Wd, torch.from_numpy(t).cuda(), DL, losses, total, 0.1,
                                  1e-4, 1.0 / M)
torch.cuda.synchronize()
logits = torch.empty((M, V), device="cuda")
lin.lin_matmul_w16(Xd, Wd, logits)
torch.cuda.synchronize()
ref_losses, _ = oracle.cross_entropy(logits.cpu().numpy().astype(np.float64), t, 0.1, 1e-4, 1.0 / M)
nd = int(np.sum(np.abs(losses.cpu().numpy() - ref_losses) > 2e-5 + 2e-5 * np.abs(ref_losses)))
report("lm_head_cross_entropy_w16", nd)
sys.exit(1 if bad else 0)
"""

VARIANTS = [{}, {"LIN_F16_PAIR": "1", "LIN_F16_PRECONVERT": "1"}]


@pytest.mark.parametrize("variant", VARIANTS, ids=["default", "pairs"])
def test_checked_build_every_form(variant):
    env = dict(os.environ, LIN_CHECKED="1", **variant)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:]
