"""The clustered kernels' banded tile order on the GPU: where the weights of
all column groups exceed what the L2 is left to hold, the tiles run in bands
of column groups (the last band narrower). Integer inputs make every result
exact, so each output element is compared for equality with the oracle;
outputs start as NaN, so an element no tile wrote shows up too. The shapes
include a split tail inside the last band and a ragged last band."""

import numpy as np
import pytest

import oracle
from tests.gpu_util import integer_inputs, require_gpu, run_device, to_device
from transformer_linear_layer_tcgen05_gb300 import lin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


# (form, M, N, K): weights per column group of four CTAs = contraction x 1024
# x 2 bytes; band = 32 MiB / that.
CASES = [
    ("matmul_w16", 640, 16384, 4096),        # 4 bands of 4; 80 tiles: split tail
    ("matmul_w16", 300, 9000, 2056),         # bands of 7 and 2 (ragged N)
    ("matmul_residual_w16", 129, 12288, 4096),
    ("matmul_residual_swiglu_a_w16", 256, 8192, 8192),   # 4 bands of 2
    ("matmul_t_w16", 384, 4096, 16384),      # output 16384 columns, contraction 4096
]


@pytest.mark.parametrize("form,M,N,K", CASES, ids=lambda v: str(v))
def test_banded_order_exact(form, M, N, K):
    from transformer_linear_layer_tcgen05_gb300 import workloads as wl
    d = integer_inputs(form, M, N, K, seed=M + K)
    out_cols = K if wl.form_is_t(form) else N
    Y = run_device(form, to_device(d), M, out_cols).cpu().numpy().astype(np.float64)
    ref, _ = oracle.reference(form, d)
    assert np.array_equal(Y, ref)


def test_gate_up_banded_exact():
    import torch
    M, N, K = 257, 8192, 4096      # 16 column groups of 512 per output, bands of 4
    rng = np.random.default_rng(5)
    X = rng.integers(-4, 5, size=(M, K)).astype(np.float32)
    WG = rng.integers(-4, 5, size=(K, N)).astype(np.float16)
    WU = rng.integers(-4, 5, size=(K, N)).astype(np.float16)
    G = torch.full((M, N), float("nan"), device="cuda")
    U = torch.full((M, N), float("nan"), device="cuda")
    lin.lin_gate_up_w16(torch.from_numpy(X).cuda(), torch.from_numpy(WG.view(np.int16)).cuda(),
                        torch.from_numpy(WU.view(np.int16)).cuda(), G, U)
    torch.cuda.synchronize()
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    rg, ru = oracle.gate_up_w16(X, WG.view(np.uint16), WU.view(np.uint16))
    assert np.array_equal(G.cpu().numpy().astype(np.float64), rg)
    assert np.array_equal(U.cpu().numpy().astype(np.float64), ru)
