"""The f32 forms that copy X (or dY) as is (matmul, matmul_residual, and the
input gradient matmul_t, whose W tile is K-major) in the per-tile kernel
with both of their tile widths (96 and 128 columns; the library takes 96
while 96-column tiles fit one wave on the SMs), bit-exact
against the oracle on small-integer inputs: ragged rows and columns (a last
column tile narrower than the tile, or than a 32-column W box), the K split
in clusters and through one tile. Each width runs in a child process of its
own (LIN_F32_BN is read once per process). A child also fails on a device
status other than success."""

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
from transformer_linear_layer_tcgen05_gb300 import lin
from transformer_linear_layer_tcgen05_gb300 import workloads as wl
require_gpu()
bad = 0
for form in ("matmul", "matmul_residual", "matmul_t"):
    # (M, N, K); matmul_t's output is [M, K]
    for (M, N, K) in [(512, 3072, 768), (512, 768, 3072), (300, 264, 68), (129, 100, 256),
                      (512, 768, 768), (1, 1000, 64), (640, 2984, 132)]:
        d = integer_inputs(form, M, N, K, seed=M + N + K)
        Yd = torch.full(wl.output_shape(form, M, N, K), float("nan"), device="cuda")
        lin.run_form(form, to_device(d), Yd)
        torch.cuda.synchronize()
        Y = Yd.cpu().numpy().astype(np.float64)
        Yref, _ = oracle.reference(form, d)
        st = lin.lin_get_device_status()
        nd = int(np.sum(Y != Yref))
        if nd or st != lin.LIN_SUCCESS:
            print(f"{form} {M}x{N}x{K}: status {st}, {nd} mismatches", flush=True)
        bad += nd + (st != lin.LIN_SUCCESS)
sys.exit(1 if bad else 0)
"""


@pytest.mark.parametrize("bn", ["96", "128"])
def test_f32_x_tile_widths_exact(bn):
    env = dict(os.environ, LIN_F32_BN=bn)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-4000:]
