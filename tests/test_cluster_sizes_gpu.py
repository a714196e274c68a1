"""Every cluster size of the binary16 kernels, bit-exact against the oracle.

The library picks the cluster size from N; LIN_F16_KERNEL overrides it for a
process ("1", "2", "4", or "tile" for the per-tile kernel), so each size runs
in a child process of its own. The shapes cover ragged M, N and K, a single
row, and launches whose last round is split along K.
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
import oracle
from tests.gpu_util import integer_inputs, require_gpu, run_device, to_device
require_gpu()
bad = 0
shapes = [(128, 256, 64), (300, 2048, 200), (129, 520, 68), (1, 1032, 4), (700, 1536, 256),
          (300, 2048, 2048), (1100, 1024, 1024)]
for form in ("matmul_residual_swiglu_a_w16", "matmul_w16", "matmul_residual_w16"):
    for (M, N, K) in shapes:
        d = integer_inputs(form, M, N, K, seed=M + N + K)
        Y = run_device(form, to_device(d), M, N).cpu().numpy().astype(np.float64)
        Yref, _ = oracle.reference(form, d)
        nd = int(np.sum(Y != Yref))
        if nd:
            print(f"{form} {M}x{N}x{K}: {nd} mismatches", flush=True)
        bad += nd
sys.exit(1 if bad else 0)
"""


@pytest.mark.parametrize("cn", ["1", "2", "4", "tile"])
def test_cluster_size_exact(cn):
    env = dict(os.environ, LIN_F16_KERNEL=cn)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-4000:]
