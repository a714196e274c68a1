"""Every cluster size of the binary16 kernels, bit-exact against the oracle.

The library picks the cluster size from N; LIN_F16_KERNEL overrides it for a
process ("1", "2", "4", or "tile" for the per-tile kernel), so each size runs
in a child process of its own. The override applies where the transform
warps build A on chip; the pre-converted binary16 A (a TMA-loaded operand)
always runs as single CTAs, so under every variant those shapes check the
single-CTA path beside the forced cluster size. The shapes cover ragged M, N and K, a single
row, and launches whose last round is split along K after whole rounds or
alone. A child also fails on a device status other than success (a bounded
wait that ran out), even when the output is right.
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
from transformer_linear_layer_tcgen05_gb300 import lin
require_gpu()
bad = 0
shapes = [(128, 256, 64), (300, 2048, 200), (129, 520, 68), (1, 1032, 4), (700, 1536, 256),
          (300, 2048, 2048), (1100, 1024, 1024), (4736, 2048, 1024), (5000, 1032, 520)]
for form in ("matmul_residual_swiglu_a_w16", "matmul_w16", "matmul_residual_w16"):
    for (M, N, K) in shapes:
        d = integer_inputs(form, M, N, K, seed=M + N + K)
        Yd = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        lin.run_form(form, to_device(d), Yd)
        torch.cuda.synchronize()
        st = lin.lin_get_device_status()
        Y = Yd.cpu().numpy().astype(np.float64)
        Yref, _ = oracle.reference(form, d)
        nd = int(np.sum(Y != Yref))
        if nd or st != lin.LIN_SUCCESS:
            print(f"{form} {M}x{N}x{K}: status {st}, {nd} mismatches", flush=True)
        bad += nd + (st != lin.LIN_SUCCESS)
sys.exit(1 if bad else 0)
"""


VARIANTS = [{"LIN_F16_KERNEL": "1"}, {"LIN_F16_KERNEL": "2"}, {"LIN_F16_KERNEL": "4"},
            {"LIN_F16_KERNEL": "tile"}]


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: "-".join(v.values()))
def test_cluster_size_exact(variant):
    env = dict(os.environ, **variant)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-4000:]
