"""lin_gate_up_w16: GATE = X @ W_gate and UP = X @ W_up in one launch, on the
GPU against the oracle, for every cluster size and both ways of rounding X
to binary16 (each in a child process, since the choice is made once per
process)."""

import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from tests.gpu_util import TOL, require_gpu
from transformer_linear_layer_tcgen05_gb300 import lin
from transformer_linear_layer_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(X, WG, WU):
    import torch
    M, N = X.shape[0], WG.shape[1]
    t = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    G = torch.full((M, N), float("nan"), device="cuda")
    U = torch.full((M, N), float("nan"), device="cuda")
    lin.lin_gate_up_w16(t(X), t(WG), t(WU), G, U)
    torch.cuda.synchronize()
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    return G.cpu().numpy().astype(np.float64), U.cpu().numpy().astype(np.float64)


def _int_inputs(M, N, K, seed):
    rng = np.random.default_rng(seed)
    X = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    WG = rng.integers(-4, 5, size=(K, N)).astype(np.float16).view(np.uint16)
    WU = rng.integers(-4, 5, size=(K, N)).astype(np.float16).view(np.uint16)
    return X, WG, WU


CHILD = r"""
import sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import oracle
from tests.gpu_util import require_gpu
from tests.test_gate_up_gpu import _int_inputs, _run
require_gpu()
bad = 0
for (M, N, K) in [(128, 128, 64), (129, 136, 68), (1, 1032, 4), (300, 2048, 200),
                  (700, 1536, 256), (4736, 1024, 1024), (513, 8192, 512), (257, 8192, 4096)]:
    X, WG, WU = _int_inputs(M, N, K, seed=M + N + K)
    G, U = _run(X, WG, WU)
    rg, ru = oracle.gate_up_w16(X, WG, WU)
    nd = int(np.sum(G != rg)) + int(np.sum(U != ru))
    if nd:
        print(f"{M}x{N}x{K}: {nd} mismatches", flush=True)
    bad += nd
sys.exit(1 if bad else 0)
"""

VARIANTS = [{"LIN_F16_KERNEL": "1"}, {"LIN_F16_KERNEL": "2"}, {"LIN_F16_KERNEL": "4"},
            {"LIN_F16_KERNEL": "tile"}, {"LIN_F16_KERNEL": "4", "LIN_F16_PRECONVERT": "0"},
            {"LIN_F16_KERNEL": "2", "LIN_F16_PRECONVERT": "1"}]


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: "-".join(v.values()))
def test_every_kernel_exact(variant):
    env = dict(os.environ, **variant)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-4000:]


@pytest.mark.parametrize("shape", [(300, 392, 200), (512, 3072, 768), (1100, 2048, 2048)])
def test_random_within_bound(shape):
    M, N, K = shape
    d = wl.generate("matmul_w16", M, N, K, seed=61 + M)
    WU = wl.generate("matmul_w16", M, N, K, seed=62 + M)["W16"]
    G, U = _run(d["X"], d["W16"], WU)
    rg, ru = oracle.gate_up_w16(d["X"], d["W16"], WU)
    for Y, ref, W in ((G, rg, d["W16"]), (U, ru, WU)):
        S = oracle.normaliser(d["X"], oracle.f16_bits_to_f64(W))
        assert oracle.normalised_error(Y, ref, S) <= TOL


def test_matches_two_single_products():
    # bit for bit the two lin_matmul_w16 calls it replaces (same rounding of
    # X, same order of the K loop) where those run unsplit (K = 512: 8
    # k-blocks, too few to split a tail)
    import torch
    M, N, K = 640, 2048, 512
    d = wl.generate("matmul_w16", M, N, K, seed=3)
    WU = wl.generate("matmul_w16", M, N, K, seed=4)["W16"]
    G, U = _run(d["X"], d["W16"], WU)
    t = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    Y = torch.empty((M, N), device="cuda")
    lin.lin_matmul_w16(t(d["X"]), t(d["W16"]), Y)
    torch.cuda.synchronize()
    assert lin.lin_last_launch_info()[0] == 2          # pre-pass + GEMM, no split sum
    assert np.array_equal(Y.cpu().numpy().astype(np.float64), G)
    lin.lin_matmul_w16(t(d["X"]), t(WU), Y)
    torch.cuda.synchronize()
    assert np.array_equal(Y.cpu().numpy().astype(np.float64), U)


def test_pairs_run_as_the_two_single_products():
    # where the products run as CTA pairs the call is the binary16 pre-pass
    # and the single-product kernel once per weight matrix, so it equals the
    # two lin_matmul_w16 calls bit for bit
    import torch
    M, N, K = 513, 8192, 512
    d = wl.generate("matmul_w16", M, N, K, seed=5)
    WU = wl.generate("matmul_w16", M, N, K, seed=6)["W16"]
    G, U = _run(d["X"], d["W16"], WU)
    assert lin.lin_last_launch_info()[0] == 3
    t = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
    Y = torch.empty((M, N), device="cuda")
    for W, ref in ((d["W16"], G), (WU, U)):
        lin.lin_matmul_w16(t(d["X"]), t(W), Y)
        torch.cuda.synchronize()
        assert np.array_equal(Y.cpu().numpy().astype(np.float64), ref)
