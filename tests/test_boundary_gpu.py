"""The C ABI on a GPU: degenerate dims, validation of real buffers, no
writes outside Y, invariants between entry points, determinism, and the
bounded-wait timeout path."""

import numpy as np
import pytest

from tests.gpu_util import TOL, integer_inputs, oracle_error, require_gpu, run_device, to_device
import oracle
from transformer_linear_layer_tcgen05_gb300 import lin
from transformer_linear_layer_tcgen05_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _torch():
    import torch
    return torch


@pytest.mark.parametrize("form", wl.FORWARD_FORMS)
def test_k_zero_gives_residual_or_zero(form):
    torch = _torch()
    M, N = 70, 48
    d = to_device(wl.generate(form, M, N, 4, seed=1))
    for k in list(d):
        if k in ("X", "GATE", "UP"):
            d[k] = torch.empty((M, 0), dtype=torch.float32, device="cuda")
        if k in ("W", "W16"):
            d[k] = torch.empty((0, N), dtype=d[k].dtype, device="cuda")
    Y = run_device(form, d, M, N)
    want = d["R"] if "R" in d else torch.zeros_like(Y)
    assert torch.equal(Y, want)


def test_empty_m_leaves_y_untouched():
    torch = _torch()
    X = torch.empty((0, 16), device="cuda")
    W = torch.randn(16, 8, device="cuda")
    Y = torch.empty((0, 8), device="cuda")
    lin.lin_matmul(X, W, Y)
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS


def test_no_writes_outside_y():
    torch = _torch()
    M, N, K = 131, 136, 36
    for form in ("matmul_residual", "matmul_w16", "matmul_residual_swiglu_a_w16"):
        d = wl.generate(form, M, N, K, seed=5)
        dd = to_device(d)
        big = torch.full((M + 64, N), 12345.0, device="cuda")
        Y = big[32:32 + M]                       # a contiguous view inside a larger buffer
        lin.run_form(form, dd, Y)
        torch.cuda.synchronize()
        assert torch.all(big[:32] == 12345.0) and torch.all(big[32 + M:] == 12345.0)
        assert oracle_error(form, d, Y.cpu().numpy()) <= TOL


def test_validation_with_real_buffers():
    torch = _torch()
    L = lin.lib()
    M, N, K = 64, 64, 64
    X = torch.randn(M, K, device="cuda")
    W = torch.randn(K, N, device="cuda")
    R = torch.randn(M, N, device="cuda")
    Y = torch.empty(M, N, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # in-place residual is aliasing
    assert L.lin_matmul_residual(X.data_ptr(), W.data_ptr(), R.data_ptr(), R.data_ptr(),
                                 M, N, K, s) == lin.LIN_ERROR_ALIASING
    # misaligned by one element
    assert L.lin_matmul(X.data_ptr() + 4, W.data_ptr(), Y.data_ptr(), M, N, K - 4, s) == \
        lin.LIN_ERROR_MISALIGNED
    # host memory is not accepted
    host = np.zeros((M, K), dtype=np.float32)
    assert L.lin_matmul(host.ctypes.data, W.data_ptr(), Y.data_ptr(), M, N, K, s) == \
        lin.LIN_ERROR_INVALID_VALUE
    # w16 needs N % 8 == 0
    W16 = torch.zeros((K, 12), dtype=torch.int16, device="cuda")
    Y12 = torch.empty((M, 12), device="cuda")
    with pytest.raises(lin.LinError) as e:
        lin.lin_matmul_w16(X, W16, Y12)
    assert e.value.status == lin.LIN_ERROR_UNSUPPORTED_SHAPE
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS


def test_residual_minus_plain_is_r():
    torch = _torch()
    M, N, K = 200, 264, 132
    for plain, resid in (("matmul", "matmul_residual"), ("matmul_w16", "matmul_residual_w16")):
        d = wl.generate(resid, M, N, K, seed=3)
        dd = to_device(d)
        Yr = run_device(resid, dd, M, N)
        Yp = run_device(plain, dd, M, N)
        # Y_r = fl(acc + R) and Y_p = fl(acc): they differ from R by at most
        # one float32 rounding of Y_r
        diff = (Yr - Yp - dd["R"]).abs()
        bound = torch.finfo(torch.float32).eps * Yr.abs()
        assert torch.all(diff <= bound + 1e-30)


def test_swiglu_matches_residual_on_materialised_a():
    torch = _torch()
    M, N, K = 150, 136, 260
    for fused, staged in (("matmul_residual_swiglu_a", "matmul_residual"),
                          ("matmul_residual_swiglu_a_w16", "matmul_residual_w16")):
        d = wl.generate(fused, M, N, K, seed=8)
        A = oracle.swiglu_a(d["GATE"], d["UP"]).astype(np.float32)
        dd = to_device(d)
        Yf = run_device(fused, dd, M, N).cpu().numpy()
        ds = {"X": torch.from_numpy(A).cuda(), "R": dd["R"]}
        ds["W16" if fused.endswith("_w16") else "W"] = dd["W16" if fused.endswith("_w16") else "W"]
        Ys = run_device(staged, ds, M, N).cpu().numpy()
        Yref, S = oracle.reference(fused, d)
        assert np.max(np.abs(Yf - Ys) / S) <= 2 * TOL


@pytest.mark.parametrize("form", wl.FORWARD_FORMS)
def test_deterministic(form):
    M, N, K = 260, 264, 300
    dd = to_device(wl.generate(form, M, N, K, seed=4))
    Y1 = run_device(form, dd, M, N)
    Y2 = run_device(form, dd, M, N)
    assert _torch().equal(Y1, Y2)


def test_exact_on_a_side_stream():
    torch = _torch()
    M, N, K = 256, 256, 128
    d = integer_inputs("matmul_residual", M, N, K, seed=2)
    dd = to_device(d)
    Y = torch.empty(M, N, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.current_stream().synchronize()
    with torch.cuda.stream(s):
        lin.lin_matmul_residual(dd["X"], dd["W"], dd["R"], Y)
    s.synchronize()
    Yref, _ = oracle.reference("matmul_residual", d)
    assert np.array_equal(Y.cpu().numpy().astype(np.float64), Yref)


def test_bounded_wait_times_out_cleanly():
    torch = _torch()
    rc = lin.lin_selftest_wait_timeout(20000)      # 20 ms per wait
    assert rc == lin.LIN_ERROR_TIMEOUT
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS   # cleared by the self-test
    # the context is still usable afterwards
    d = integer_inputs("matmul", 128, 128, 64, seed=1)
    Y = run_device("matmul", to_device(d), 128, 128).cpu().numpy().astype(np.float64)
    assert np.array_equal(Y, oracle.reference("matmul", d)[0])
    assert torch.cuda.is_available()


# (form, shape, kernels, workspace): the per-tile f32 kernel splits K inside
# a cluster (one kernel, no workspace); the clustered binary16 kernel splits
# its last round (GEMM + split sum, a workspace)
@pytest.mark.parametrize("form,shape,kernels,workspace",
                         [("matmul", (512, 768, 768), 1, False),
                          ("matmul_residual_swiglu_a_w16", (300, 2048, 2048), 2, True)])
def test_split_inside_a_cuda_graph(form, shape, kernels, workspace):
    # A split launch captured into a graph takes its workspace (if any) as a
    # graph memory node; replays must equal a direct call bit for bit.
    torch = _torch()
    M, N, K = shape
    dd = to_device(wl.generate(form, M, N, K, seed=9))
    direct = run_device(form, dd, M, N)
    assert lin.lin_last_launch_info()[0] == kernels   # the problem splits on a GB300
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            lin.run_form(form, dd, Y)
            captured = lin.lin_last_launch_info()
    torch.cuda.current_stream().wait_stream(s)
    assert captured[0] == kernels and (captured[1] > 0) == workspace
    for _ in range(2):
        Y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert lin.lin_get_device_status() == lin.LIN_SUCCESS
        assert torch.equal(Y, direct)
    del g
