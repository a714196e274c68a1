"""The host-operand forms (lin_*_host) on the GPU against the oracle: every
forward form with its operands in pinned or pageable host memory, split into
many row blocks (the staging buffers are reused several times, and the last
block is ragged), exactly on integer inputs; random inputs within the bound
with the default blocks; the empty contraction; and the memory-type rule."""

import numpy as np
import pytest

import oracle
from tests.gpu_util import TOL, integer_inputs, require_gpu
from transformer_linear_layer_tcgen05_gb300 import lin
from transformer_linear_layer_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

FORMS = list(lin.HOST_FORM_FUNCS)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    yield
    lin.lin_set_host_block_bytes(0)


def _host_dict(d, pinned):
    import torch
    out = {}
    for k, v in d.items():
        t = torch.from_numpy(np.ascontiguousarray(v.view(np.int16) if v.dtype == np.uint16 else v))
        out[k] = t.pin_memory() if pinned else t
    return out


def _run(form, d, M, N, pinned):
    import torch
    Y = torch.full((M, N), float("nan"))
    if pinned:
        Y = Y.pin_memory()
    lin.run_form_host(form, _host_dict(d, pinned), Y)
    torch.cuda.synchronize()
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    return Y.numpy().astype(np.float64)


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("form", FORMS)
def test_many_blocks_exact(form, pinned):
    M, N, K = 1000, 264, 200          # 128-row blocks: 8 of them, the last 104 rows
    lin.lin_set_host_block_bytes(1 << 16)
    try:
        d = integer_inputs(form, M, N, K, seed=M + N + K)
        Y = _run(form, d, M, N, pinned)
        kernels, _ = lin.lin_last_launch_info()
        assert kernels >= 8
    finally:
        lin.lin_set_host_block_bytes(0)
    ref, _ = oracle.reference(form, d)
    assert np.array_equal(Y, ref)


@pytest.mark.parametrize("form", ["matmul_residual_swiglu_a_w16", "matmul_w16", "matmul_residual"])
def test_random_within_bound(form):
    M, N, K = 700, 1024, 768
    d = wl.generate(form, M, N, K, seed=77)
    Y = _run(form, d, M, N, True)
    Yref, S = oracle.reference(form, d)
    assert oracle.normalised_error(Y, Yref, S, d.get("R")) <= TOL


def test_empty_contraction_copies_r():
    import torch
    M, N = 300, 64
    R = torch.arange(M * N, dtype=torch.float32).reshape(M, N).pin_memory()
    Y = torch.full((M, N), float("nan")).pin_memory()
    X = torch.empty((M, 0)).pin_memory()
    W = torch.empty((0, N), dtype=torch.int16).pin_memory()
    lin.lin_matmul_residual_w16_host(X, W, R, Y)
    torch.cuda.synchronize()
    assert torch.equal(Y, R)


def test_device_memory_is_rejected():
    import torch
    M, N, K = 128, 64, 64
    X = torch.zeros((M, K), device="cuda")
    W = torch.zeros((K, N)).pin_memory()
    Y = torch.zeros((M, N)).pin_memory()
    st = lin.lib().lin_matmul_host(X.data_ptr(), W.data_ptr(), Y.data_ptr(), M, N, K,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == lin.LIN_ERROR_INVALID_VALUE


def test_rejected_under_stream_capture():
    import torch
    M, N, K = 128, 64, 64
    X = torch.zeros((M, K)).pin_memory()
    W = torch.zeros((K, N)).pin_memory()
    Y = torch.zeros((M, N)).pin_memory()
    Z = torch.zeros(16, device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            Z.add_(1.0)     # the graph is not empty
            st = lin.lib().lin_matmul_host(X.data_ptr(), W.data_ptr(), Y.data_ptr(), M, N, K,
                                           s.cuda_stream)
    torch.cuda.current_stream().wait_stream(s)
    assert st == lin.LIN_ERROR_INVALID_VALUE
