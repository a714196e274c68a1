"""Thin ctypes binding of the C ABI in include/lin.h.

Argument marshalling only: every function here forwards to the function of
the same name in ``liblin.so``; all arithmetic runs in the library's CUDA
kernels. There is no fallback: if the library is missing or fails to load,
every call raises.

Two layers:

* ``lib()`` returns the ``ctypes.CDLL`` with typed signatures; its functions
  take raw device pointers (ints), int64 dims and a stream handle, and return
  the ``lin_status`` code.
* ``lin_matmul(X, W, Y)`` and friends take torch CUDA tensors, derive
  (M, N, K) from their shapes, call the C function on the current torch
  stream (or ``stream=``) and raise ``LinError`` on a non-zero status.
  Binary16 weights may be given as ``torch.float16``, ``torch.int16`` or
  ``torch.uint16`` tensors (only the bit patterns are read).
"""

from __future__ import annotations

import ctypes
import os

# LIN_CHECKED=1 loads the checked build (liblin_checked.so: the kernels check
# their indices and report LIN_ERROR_DEVICE_CHECK; see include/lin.h).
_LIB_NAME = "liblin_checked.so" if os.environ.get("LIN_CHECKED") == "1" else "liblin.so"
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), _LIB_NAME)

STATUS = {
    0: "LIN_SUCCESS",
    1: "LIN_ERROR_INVALID_VALUE",
    2: "LIN_ERROR_UNSUPPORTED_SHAPE",
    3: "LIN_ERROR_MISALIGNED",
    4: "LIN_ERROR_ALIASING",
    5: "LIN_ERROR_UNSUPPORTED_DEVICE",
    6: "LIN_ERROR_CUDA",
    7: "LIN_ERROR_TIMEOUT",
    8: "LIN_ERROR_DEVICE_CHECK",
}
LIN_SUCCESS = 0
LIN_ERROR_INVALID_VALUE = 1
LIN_ERROR_UNSUPPORTED_SHAPE = 2
LIN_ERROR_MISALIGNED = 3
LIN_ERROR_ALIASING = 4
LIN_ERROR_UNSUPPORTED_DEVICE = 5
LIN_ERROR_CUDA = 6
LIN_ERROR_TIMEOUT = 7
LIN_ERROR_DEVICE_CHECK = 8

_P = ctypes.c_void_p
_I = ctypes.c_int64
_S = ctypes.c_void_p  # lin_stream_t
_F = ctypes.c_float

# name -> argument types (all compute entry points return lin_status as int)
SIGNATURES = {
    "lin_matmul": [_P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_residual": [_P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_residual_swiglu_a": [_P, _P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_w16": [_P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_residual_w16": [_P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_residual_swiglu_a_w16": [_P, _P, _P, _P, _P, _I, _I, _I, _S],
    "lin_get_device_status": [_S],
    "lin_selftest_wait_timeout": [_I, _S],
    "lin_selftest_device_check": [_I, _S],
    "lin_matmul_residual_swiglu_a_w16_noalloc": [_P, _P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_t": [_P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_t_acc": [_P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_t_w16": [_P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_t_acc_w16": [_P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_at": [_P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_at_acc": [_P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_at_swiglu_a": [_P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_at_swiglu_a_acc": [_P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_t_swiglu_backward": [_P, _P, _P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_t_swiglu_backward_w16": [_P, _P, _P, _P, _P, _P, _I, _I, _I, _S],
    "lin_lm_head_cross_entropy_w16": [_P, _P, _P, _P, _P, _P, _I, _I, _I, _F, _F, _F, _S],
    "lin_gate_up_w16": [_P, _P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_host": [_P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_residual_host": [_P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_residual_swiglu_a_host": [_P, _P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_w16_host": [_P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_residual_w16_host": [_P, _P, _P, _P, _I, _I, _I, _S],
    "lin_matmul_residual_swiglu_a_w16_host": [_P, _P, _P, _P, _P, _I, _I, _I, _S],
    "lin_set_host_block_bytes": [ctypes.c_uint64],
}

_lib = None


class LinError(RuntimeError):
    """A non-zero lin_status returned by the library."""

    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{fn} returned {STATUS.get(status, status)}"
        if status == LIN_ERROR_CUDA:
            msg += f" (cudaError_t {cuda_error})"
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """Load liblin.so (once) and declare its signatures. Raises if missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; build it with "
                "transformer_linear_layer_tcgen05_gb300.build.build_library()")
        L = ctypes.CDLL(LIB_PATH)
        for name, argtypes in SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = argtypes
            f.restype = ctypes.c_int
        L.lin_status_string.argtypes = [ctypes.c_int]
        L.lin_status_string.restype = ctypes.c_char_p
        L.lin_last_cuda_error.argtypes = []
        L.lin_last_cuda_error.restype = ctypes.c_int
        L.lin_version.argtypes = []
        L.lin_version.restype = ctypes.c_int
        L.lin_last_launch_info.argtypes = [ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_uint64)]
        L.lin_last_launch_info.restype = None
        L.lin_last_device_check.argtypes = [ctypes.POINTER(ctypes.c_int),
                                            ctypes.POINTER(ctypes.c_int64)]
        L.lin_last_device_check.restype = None
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().lin_status_string(int(status)).decode()


def check(fn: str, status: int) -> None:
    if status != LIN_SUCCESS:
        raise LinError(fn, status, lib().lin_last_cuda_error() if status == LIN_ERROR_CUDA else 0)


# ----------------------------------------------------------------- tensor layer

def _stream_handle(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _f32(t, name):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda:
        raise TypeError(f"{name} must be a float32 CUDA tensor")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D tensor")
    return t


def _w16(t, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.element_size() != 2 or \
            t.dtype not in (torch.float16, torch.int16, getattr(torch, "uint16", torch.int16)):
        raise TypeError(f"{name} must be a 16-bit (binary16 bits) CUDA tensor")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D tensor")
    return t


def _dims(A, W, Y):
    M, K = A.shape
    K2, N = W.shape
    if K2 != K or tuple(Y.shape) != (M, N):
        raise ValueError(f"shape mismatch: A{tuple(A.shape)} W{tuple(W.shape)} Y{tuple(Y.shape)}")
    return M, N, K


def _call(name, *args):
    check(name, getattr(lib(), name)(*args))


def lin_matmul(X, W, Y, stream=None):
    """Y = X @ W (f32; TF32 tensor cores, f32 accumulate)."""
    M, N, K = _dims(_f32(X, "X"), _f32(W, "W"), _f32(Y, "Y"))
    _call("lin_matmul", X.data_ptr(), W.data_ptr(), Y.data_ptr(), M, N, K,
          _stream_handle(stream))
    return Y


def lin_matmul_residual(X, W, R, Y, stream=None):
    """Y = X @ W + R."""
    M, N, K = _dims(_f32(X, "X"), _f32(W, "W"), _f32(Y, "Y"))
    if tuple(_f32(R, "R").shape) != (M, N):
        raise ValueError("R must be [M, N]")
    _call("lin_matmul_residual", X.data_ptr(), W.data_ptr(), R.data_ptr(), Y.data_ptr(),
          M, N, K, _stream_handle(stream))
    return Y


def lin_matmul_residual_swiglu_a(GATE, UP, W, R, Y, stream=None):
    """Y = (silu(GATE) * UP) @ W + R."""
    M, N, K = _dims(_f32(GATE, "GATE"), _f32(W, "W"), _f32(Y, "Y"))
    if tuple(_f32(UP, "UP").shape) != (M, K) or tuple(_f32(R, "R").shape) != (M, N):
        raise ValueError("UP must be [M, K] and R [M, N]")
    _call("lin_matmul_residual_swiglu_a", GATE.data_ptr(), UP.data_ptr(), W.data_ptr(),
          R.data_ptr(), Y.data_ptr(), M, N, K, _stream_handle(stream))
    return Y


def lin_matmul_w16(X, W16, Y, stream=None):
    """Y = X @ W16 with binary16 weights."""
    M, N, K = _dims(_f32(X, "X"), _w16(W16, "W16"), _f32(Y, "Y"))
    _call("lin_matmul_w16", X.data_ptr(), W16.data_ptr(), Y.data_ptr(), M, N, K,
          _stream_handle(stream))
    return Y


def lin_matmul_residual_w16(X, W16, R, Y, stream=None):
    """Y = X @ W16 + R with binary16 weights."""
    M, N, K = _dims(_f32(X, "X"), _w16(W16, "W16"), _f32(Y, "Y"))
    if tuple(_f32(R, "R").shape) != (M, N):
        raise ValueError("R must be [M, N]")
    _call("lin_matmul_residual_w16", X.data_ptr(), W16.data_ptr(), R.data_ptr(),
          Y.data_ptr(), M, N, K, _stream_handle(stream))
    return Y


def lin_matmul_residual_swiglu_a_w16(GATE, UP, W16, R, Y, stream=None):
    """Y = (silu(GATE) * UP) @ W16 + R with binary16 W_down."""
    M, N, K = _dims(_f32(GATE, "GATE"), _w16(W16, "W16"), _f32(Y, "Y"))
    if tuple(_f32(UP, "UP").shape) != (M, K) or tuple(_f32(R, "R").shape) != (M, N):
        raise ValueError("UP must be [M, K] and R [M, N]")
    _call("lin_matmul_residual_swiglu_a_w16", GATE.data_ptr(), UP.data_ptr(),
          W16.data_ptr(), R.data_ptr(), Y.data_ptr(), M, N, K, _stream_handle(stream))
    return Y


def lin_matmul_residual_swiglu_a_w16_noalloc(GATE, UP, W16, R, Y, stream=None):
    """lin_matmul_residual_swiglu_a_w16 with its split-tail workspace in the
    library's static device array: allocates no device memory. Calls whose
    execution can overlap (different streams) must not be issued."""
    M, K = _f32(GATE, "GATE").shape
    N = W16.shape[1]
    if tuple(W16.shape) != (K, N) or tuple(_f32(Y, "Y").shape) != (M, N):
        raise ValueError("W16 must be [K, N] and Y [M, N]")
    if tuple(_f32(UP, "UP").shape) != (M, K) or tuple(_f32(R, "R").shape) != (M, N):
        raise ValueError("UP must be [M, K] and R [M, N]")
    _call("lin_matmul_residual_swiglu_a_w16_noalloc", GATE.data_ptr(), UP.data_ptr(),
          W16.data_ptr(), R.data_ptr(), Y.data_ptr(), M, N, K, _stream_handle(stream))
    return Y


def _dims_t(DY, W, DX):
    M, N = DY.shape
    K, N2 = W.shape
    if N2 != N or tuple(DX.shape) != (M, K):
        raise ValueError(f"shape mismatch: dY{tuple(DY.shape)} W{tuple(W.shape)} dX{tuple(DX.shape)}")
    return M, N, K


def lin_matmul_t(DY, W, DX, stream=None):
    """dX = dY @ W^T (dY [M,N], W [K,N], dX [M,K]; TF32, f32 accumulate)."""
    M, N, K = _dims_t(_f32(DY, "dY"), _f32(W, "W"), _f32(DX, "dX"))
    _call("lin_matmul_t", DY.data_ptr(), W.data_ptr(), DX.data_ptr(), M, N, K,
          _stream_handle(stream))
    return DX


def lin_matmul_t_acc(DY, W, DX, stream=None):
    """dX += dY @ W^T."""
    M, N, K = _dims_t(_f32(DY, "dY"), _f32(W, "W"), _f32(DX, "dX"))
    _call("lin_matmul_t_acc", DY.data_ptr(), W.data_ptr(), DX.data_ptr(), M, N, K,
          _stream_handle(stream))
    return DX


def lin_matmul_t_w16(DY, W16, DX, stream=None):
    """dX = dY @ W16^T with binary16 weights (dY rounded to binary16)."""
    M, N, K = _dims_t(_f32(DY, "dY"), _w16(W16, "W16"), _f32(DX, "dX"))
    _call("lin_matmul_t_w16", DY.data_ptr(), W16.data_ptr(), DX.data_ptr(), M, N, K,
          _stream_handle(stream))
    return DX


def lin_matmul_t_acc_w16(DY, W16, DX, stream=None):
    """dX += dY @ W16^T with binary16 weights."""
    M, N, K = _dims_t(_f32(DY, "dY"), _w16(W16, "W16"), _f32(DX, "dX"))
    _call("lin_matmul_t_acc_w16", DY.data_ptr(), W16.data_ptr(), DX.data_ptr(), M, N, K,
          _stream_handle(stream))
    return DX


def _dims_at(X, DY, DW):
    M, K = X.shape
    M2, N = DY.shape
    if M2 != M or tuple(DW.shape) != (K, N):
        raise ValueError(f"shape mismatch: X{tuple(X.shape)} dY{tuple(DY.shape)} dW{tuple(DW.shape)}")
    return M, N, K


def lin_matmul_at(X, DY, DW, stream=None):
    """dW = X^T @ dY (X [M,K], dY [M,N], dW [K,N]; TF32, f32 accumulate)."""
    M, N, K = _dims_at(_f32(X, "X"), _f32(DY, "dY"), _f32(DW, "dW"))
    _call("lin_matmul_at", X.data_ptr(), DY.data_ptr(), DW.data_ptr(), M, N, K,
          _stream_handle(stream))
    return DW


def lin_matmul_at_acc(X, DY, DW, stream=None):
    """dW += X^T @ dY."""
    M, N, K = _dims_at(_f32(X, "X"), _f32(DY, "dY"), _f32(DW, "dW"))
    _call("lin_matmul_at_acc", X.data_ptr(), DY.data_ptr(), DW.data_ptr(), M, N, K,
          _stream_handle(stream))
    return DW


def lin_matmul_at_swiglu_a(GATE, UP, DY, DW, stream=None):
    """dW = (silu(GATE) * UP)^T @ dY (GATE, UP [M,K], dY [M,N], dW [K,N])."""
    M, N, K = _dims_at(_f32(GATE, "GATE"), _f32(DY, "dY"), _f32(DW, "dW"))
    if tuple(_f32(UP, "UP").shape) != (M, K):
        raise ValueError("UP must be [M, K]")
    _call("lin_matmul_at_swiglu_a", GATE.data_ptr(), UP.data_ptr(), DY.data_ptr(),
          DW.data_ptr(), M, N, K, _stream_handle(stream))
    return DW


def lin_matmul_at_swiglu_a_acc(GATE, UP, DY, DW, stream=None):
    """dW += (silu(GATE) * UP)^T @ dY."""
    M, N, K = _dims_at(_f32(GATE, "GATE"), _f32(DY, "dY"), _f32(DW, "dW"))
    if tuple(_f32(UP, "UP").shape) != (M, K):
        raise ValueError("UP must be [M, K]")
    _call("lin_matmul_at_swiglu_a_acc", GATE.data_ptr(), UP.data_ptr(), DY.data_ptr(),
          DW.data_ptr(), M, N, K, _stream_handle(stream))
    return DW


def _swiglu_bwd(name, DY, W, GATE, UP, DGATE, DUP, stream):
    M, N, K = _dims_t(_f32(DY, "dY"), W, _f32(DGATE, "dGATE"))
    for t, nm in ((GATE, "GATE"), (UP, "UP"), (DUP, "dUP")):
        if tuple(_f32(t, nm).shape) != (M, K):
            raise ValueError(f"{nm} must be [M, K]")
    _call(name, DY.data_ptr(), W.data_ptr(), GATE.data_ptr(), UP.data_ptr(), DGATE.data_ptr(),
          DUP.data_ptr(), M, N, K, _stream_handle(stream))
    return DGATE, DUP


def lin_matmul_t_swiglu_backward(DY, W, GATE, UP, DGATE, DUP, stream=None):
    """dA = dY @ W^T on chip; dGATE = nan_guard(dA * UP * silu'(GATE)),
    dUP = nan_guard(dA * silu(GATE)) (TF32)."""
    return _swiglu_bwd("lin_matmul_t_swiglu_backward", DY, _f32(W, "W"), GATE, UP, DGATE, DUP,
                       stream)


def lin_matmul_t_swiglu_backward_w16(DY, W16, GATE, UP, DGATE, DUP, stream=None):
    """lin_matmul_t_swiglu_backward with binary16 W_down."""
    return _swiglu_bwd("lin_matmul_t_swiglu_backward_w16", DY, _w16(W16, "W16"), GATE, UP,
                       DGATE, DUP, stream)


def lin_lm_head_cross_entropy_w16(X, W16, targets, DLOGITS, losses, loss_sum, alpha=0.0,
                                  beta=0.0, inv_norm=1.0, stream=None):
    """Logits X @ W16 into DLOGITS, then the fused cross-entropy in place:
    DLOGITS becomes dLogits, losses [M] the per-row losses, loss_sum [1]
    their sum. targets: int32 [M] (outside [0, V): ignored row)."""
    import torch
    M, V, K = _dims(_f32(X, "X"), _w16(W16, "W16"), _f32(DLOGITS, "dLogits"))
    if not isinstance(targets, torch.Tensor) or targets.dtype != torch.int32 or \
            not targets.is_cuda or targets.numel() != M or not targets.is_contiguous():
        raise TypeError("targets must be a contiguous int32 CUDA tensor of M entries")
    for t, nm, n in ((losses, "losses", M), (loss_sum, "loss_sum", 1)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda or \
                t.numel() != n or not t.is_contiguous():
            raise TypeError(f"{nm} must be a contiguous float32 CUDA tensor of {n} entries")
    _call("lin_lm_head_cross_entropy_w16", X.data_ptr(), W16.data_ptr(), targets.data_ptr(),
          DLOGITS.data_ptr(), losses.data_ptr(), loss_sum.data_ptr(), M, V, K, float(alpha),
          float(beta), float(inv_norm), _stream_handle(stream))
    return DLOGITS, losses, loss_sum


def lin_gate_up_w16(X, WG16, WU16, GATE, UP, stream=None):
    """GATE = X @ WG16 and UP = X @ WU16 (binary16 weights) in one launch."""
    M, N, K = _dims(_f32(X, "X"), _w16(WG16, "WG16"), _f32(GATE, "GATE"))
    if tuple(_w16(WU16, "WU16").shape) != (K, N) or tuple(_f32(UP, "UP").shape) != (M, N):
        raise ValueError("WU16 must be [K, N] and UP [M, N]")
    _call("lin_gate_up_w16", X.data_ptr(), WG16.data_ptr(), WU16.data_ptr(), GATE.data_ptr(),
          UP.data_ptr(), M, N, K, _stream_handle(stream))
    return GATE, UP


def lin_last_launch_info() -> tuple:
    """(kernels launched, workspace bytes taken) by the last compute call made
    on this thread."""
    k = ctypes.c_int(0)
    b = ctypes.c_uint64(0)
    lib().lin_last_launch_info(ctypes.byref(k), ctypes.byref(b))
    return k.value, b.value


def lin_get_device_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status word."""
    return lib().lin_get_device_status(_stream_handle(stream))


def lin_selftest_wait_timeout(timeout_us: int, stream=None) -> int:
    """Run the bounded-wait self-test; LIN_ERROR_TIMEOUT means it works."""
    return lib().lin_selftest_wait_timeout(int(timeout_us), _stream_handle(stream))


def lin_selftest_device_check(value: int, stream=None) -> int:
    """Run the device-check record self-test; LIN_ERROR_DEVICE_CHECK means it
    works (lin_last_device_check() then gives (99, value))."""
    return lib().lin_selftest_device_check(int(value), _stream_handle(stream))


def lin_last_device_check() -> tuple:
    """(site, value) of the calling thread's last LIN_ERROR_DEVICE_CHECK."""
    site = ctypes.c_int(0)
    value = ctypes.c_int64(0)
    lib().lin_last_device_check(ctypes.byref(site), ctypes.byref(value))
    return site.value, value.value


# ------------------------------------------------- host-operand forms (CPU tensors)

def _host(t, name, w16=False):
    import torch
    ok = isinstance(t, torch.Tensor) and not t.is_cuda and (
        t.element_size() == 2 and t.dtype in (torch.float16, torch.int16,
                                              getattr(torch, "uint16", torch.int16))
        if w16 else t.dtype == torch.float32)
    if not ok:
        raise TypeError(f"{name} must be a {'16-bit' if w16 else 'float32'} CPU tensor")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D tensor")
    return t


def _host_call(name, A, U, W, R, Y, w16, stream):
    M, N, K = _dims(_host(A, "A"), _host(W, "W", w16), _host(Y, "Y"))
    if U is not None and tuple(_host(U, "UP").shape) != (M, K):
        raise ValueError("UP must be [M, K]")
    if R is not None and tuple(_host(R, "R").shape) != (M, N):
        raise ValueError("R must be [M, N]")
    ptrs = [A.data_ptr()] + ([U.data_ptr()] if U is not None else []) + [W.data_ptr()] + \
        ([R.data_ptr()] if R is not None else []) + [Y.data_ptr()]
    _call(name, *ptrs, M, N, K, _stream_handle(stream))
    return Y


def lin_matmul_host(X, W, Y, stream=None):
    """lin_matmul on host (CPU) tensors; pinned memory lets the copies overlap."""
    return _host_call("lin_matmul_host", X, None, W, None, Y, False, stream)


def lin_matmul_residual_host(X, W, R, Y, stream=None):
    return _host_call("lin_matmul_residual_host", X, None, W, R, Y, False, stream)


def lin_matmul_residual_swiglu_a_host(GATE, UP, W, R, Y, stream=None):
    return _host_call("lin_matmul_residual_swiglu_a_host", GATE, UP, W, R, Y, False, stream)


def lin_matmul_w16_host(X, W16, Y, stream=None):
    return _host_call("lin_matmul_w16_host", X, None, W16, None, Y, True, stream)


def lin_matmul_residual_w16_host(X, W16, R, Y, stream=None):
    return _host_call("lin_matmul_residual_w16_host", X, None, W16, R, Y, True, stream)


def lin_matmul_residual_swiglu_a_w16_host(GATE, UP, W16, R, Y, stream=None):
    return _host_call("lin_matmul_residual_swiglu_a_w16_host", GATE, UP, W16, R, Y, True, stream)


def lin_set_host_block_bytes(nbytes: int) -> None:
    """Operand-plus-result bytes per block of the host-operand forms (0: default)."""
    check("lin_set_host_block_bytes", lib().lin_set_host_block_bytes(int(nbytes)))


HOST_FORM_FUNCS = {
    "matmul": lin_matmul_host,
    "matmul_residual": lin_matmul_residual_host,
    "matmul_residual_swiglu_a": lin_matmul_residual_swiglu_a_host,
    "matmul_w16": lin_matmul_w16_host,
    "matmul_residual_w16": lin_matmul_residual_w16_host,
    "matmul_residual_swiglu_a_w16": lin_matmul_residual_swiglu_a_w16_host,
}


def run_form_host(form: str, d: dict, Y, stream=None):
    """run_form for the forward forms with host (CPU) tensors throughout."""
    f = HOST_FORM_FUNCS[form]
    w = d["W16"] if form.endswith("_w16") else d["W"]
    if "swiglu" in form:
        return f(d["GATE"], d["UP"], w, d["R"], Y, stream=stream)
    if "residual" in form:
        return f(d["X"], w, d["R"], Y, stream=stream)
    return f(d["X"], w, Y, stream=stream)


FORM_FUNCS = {
    "matmul": lin_matmul,
    "matmul_residual": lin_matmul_residual,
    "matmul_residual_swiglu_a": lin_matmul_residual_swiglu_a,
    "matmul_w16": lin_matmul_w16,
    "matmul_residual_w16": lin_matmul_residual_w16,
    "matmul_residual_swiglu_a_w16": lin_matmul_residual_swiglu_a_w16,
    "matmul_t": lin_matmul_t,
    "matmul_t_acc": lin_matmul_t_acc,
    "matmul_t_w16": lin_matmul_t_w16,
    "matmul_t_acc_w16": lin_matmul_t_acc_w16,
    "matmul_at": lin_matmul_at,
    "matmul_at_acc": lin_matmul_at_acc,
    "matmul_at_swiglu_a": lin_matmul_at_swiglu_a,
    "matmul_at_swiglu_a_acc": lin_matmul_at_swiglu_a_acc,
    "matmul_t_swiglu_backward": lin_matmul_t_swiglu_backward,
    "matmul_t_swiglu_backward_w16": lin_matmul_t_swiglu_backward_w16,
}

# entry points whose outputs are not a single [M, N] product (no run_form)
OTHER_FUNCS = {
    "lm_head_cross_entropy_w16": lin_lm_head_cross_entropy_w16,
    "gate_up_w16": lin_gate_up_w16,
}


def run_form(form: str, d: dict, Y, stream=None):
    """Call the entry point of ``form`` with the device tensors of dict ``d``
    (keys as produced by ``workloads.generate``: X or GATE/UP, W or W16, R;
    DY for the backward forms). For the SwiGLU-backward forms Y is the pair
    (dGATE, dUP)."""
    f = FORM_FUNCS[form]
    if form.startswith("matmul_at"):
        # dW = X^T @ dY; the accumulating form adds into Y (initial dW = d["R"])
        if "_acc" in form:
            Y.copy_(d["R"])
        if "swiglu" in form:
            return f(d["GATE"], d["UP"], d["DY"], Y, stream=stream)
        return f(d["X"], d["DY"], Y, stream=stream)
    w = d["W16"] if form.endswith("_w16") else d["W"]
    if "swiglu_backward" in form:   # two outputs: Y is the pair (dGATE, dUP)
        return f(d["DY"], w, d["GATE"], d["UP"], Y[0], Y[1], stream=stream)
    if form.startswith("matmul_t"):
        # dX = dY @ W^T; the accumulating forms add into Y, which must hold
        # the initial dX (d["R"]) when called
        if "_acc" in form:
            Y.copy_(d["R"])
        return f(d["DY"], w, Y, stream=stream)
    if "swiglu" in form:
        return f(d["GATE"], d["UP"], w, d["R"], Y, stream=stream)
    if "residual" in form:
        return f(d["X"], w, d["R"], Y, stream=stream)
    return f(d["X"], w, Y, stream=stream)
