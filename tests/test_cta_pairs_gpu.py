"""The pre-converted binary16 forms (A rounded by the pre-pass and copied by
TMA) run as CTA pairs -- one UMMA of M = 256 over the two CTAs of a cluster
of two (tcgen05 .cta_group::2), each CTA loading 128 rows of A and half of
the tile's W columns -- or as single CTAs. Both, bit-exact against the
oracle on small-integer inputs, for every form that takes that path: the
forward products, the transposed product dY · W^T (K-major W, half the W
rows per CTA), its accumulating form, the fused SwiGLU backward, and the
gate/up pair (the even CTA loads the W_gate tile, the odd one W_up's).

Each setting runs in a child process of its own (the library reads
LIN_F16_PAIR and LIN_F16_PRECONVERT once per process); the pre-pass is
forced on, so that narrow outputs take this path too. The shapes put the
odd CTA's rows wholly or partly past M, leave N and the contraction
ragged, and split the last round along K after whole rounds and alone.
A child also fails on a device status other than success.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import torch
import oracle
from tests.gpu_util import integer_inputs, require_gpu, to_device
from tests.test_gate_up_gpu import _int_inputs, _run
from transformer_linear_layer_tcgen05_gb300 import lin
require_gpu()
bad = 0

def report(what, nd, st):
    global bad
    if nd or st != lin.LIN_SUCCESS:
        print(f"{what}: status {st}, {nd} mismatches", flush=True)
    bad += nd + (st != lin.LIN_SUCCESS)

# (M, N, K) of the forward products: rows 1, 129 and 300 leave the odd CTA
# of the last pair tile with no or some rows; 2560 x 2048 x 1024 makes 80
# pair tiles (76 pairs: a split tail after a whole round); 512 x 2048 x 2048
# 16 tiles (a split alone)
FWD = [(1, 1032, 8), (129, 520, 200), (300, 2048, 256), (256, 136, 64), (700, 1536, 1024),
       (2560, 2048, 1024), (512, 2048, 2048)]
for form in ("matmul_w16", "matmul_residual_w16"):
    for (M, N, K) in FWD:
        d = integer_inputs(form, M, N, K, seed=M + N + K)
        Yd = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        lin.run_form(form, to_device(d), Yd)
        torch.cuda.synchronize()
        Yref, _ = oracle.reference(form, d)
        report(f"{form} {M}x{N}x{K}", int(np.sum(Yd.cpu().numpy().astype(np.float64) != Yref)),
               lin.lin_get_device_status())

# transposed products: dY [M,N], W [K,N], dX [M,K] (the output has K columns)
BT = [(129, 136, 520), (300, 1032, 2048), (1, 8, 1024), (2560, 1024, 2048), (512, 2048, 2048)]
for form in ("matmul_t_w16", "matmul_t_acc_w16"):
    for (M, N, K) in BT:
        d = integer_inputs(form, M, N, K, seed=M + 3 * N + 5 * K)
        Yd = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
        lin.run_form(form, to_device(d), Yd)
        torch.cuda.synchronize()
        Yref, _ = oracle.reference(form, d)
        report(f"{form} {M}x{N}x{K}", int(np.sum(Yd.cpu().numpy().astype(np.float64) != Yref)),
               lin.lin_get_device_status())

form = "matmul_t_swiglu_backward_w16"
for (M, N, K) in [(129, 136, 520), (300, 2048, 2048), (777, 512, 768)]:
    d = integer_inputs(form, M, N, K, seed=5 * M + N + 3 * K)
    DG = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
    DU = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
    lin.run_form(form, to_device(d), (DG, DU))
    torch.cuda.synchronize()
    (rg, ru), _ = oracle.reference(form, d)
    nd = int(np.sum(DG.cpu().numpy().astype(np.float64) != rg))
    nd += int(np.sum(DU.cpu().numpy().astype(np.float64) != ru))
    report(f"{form} {M}x{N}x{K}", nd, lin.lin_get_device_status())

for (M, N, K) in [(129, 136, 64), (300, 2048, 200), (513, 8192, 512), (4736, 1024, 1024)]:
    X, WG, WU = _int_inputs(M, N, K, seed=M + N + K)
    G, U = _run(X, WG, WU)
    rg, ru = oracle.gate_up_w16(X, WG, WU)
    report(f"gate_up {M}x{N}x{K}", int(np.sum(G != rg)) + int(np.sum(U != ru)),
           lin.lin_get_device_status())
sys.exit(1 if bad else 0)
"""

VARIANTS = [{"LIN_F16_PAIR": "1", "LIN_F16_PRECONVERT": "1"},
            {"LIN_F16_PAIR": "0", "LIN_F16_PRECONVERT": "1"}]


@pytest.mark.parametrize("variant", VARIANTS, ids=["pairs", "single"])
def test_preconverted_forms_exact(variant):
    env = dict(os.environ, **variant)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:]
