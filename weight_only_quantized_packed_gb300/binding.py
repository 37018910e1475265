"""Thin ctypes binding over libwqp.so (the C ABI declared in include/wqp.h).

Argument marshalling only. torch supplies device memory and the current
stream, and every step of the computation runs in the library's CUDA
kernels. There is no CPU or PyTorch fallback: if libwqp.so is missing or a
call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "WqpError", "lib", "lib_path", "q2_gemv", "q2_gemm_tc", "q2_gemm_mma", "w4a16_gemv", "w4a16_gemm_tc",
    "w4a16_gemm_mma", "w8a16_gemm", "w8a16_gemm_tc", "w8a16_gemm_mma",
    "q2_dequant", "w4a16_dequant", "w8a16_dequant", "row_chunks", "set_pdl",
    "get_device_error", "selftest_wait_timeout", "status_string", "EXPORTS", "MAX_M_PER_LAUNCH",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libwqp.so")
MAX_M_PER_LAUNCH = 16

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float

# name -> argtypes; every symbol declared in include/wqp.h.
EXPORTS = {
    "q2_gemv": [_P, _P, _P, _P, _I, _I, _I, _P],
    "q2_gemv_strided": [_P, _I, _P, _P, _I, _I, _I, _I, _P],
    "q2_gemm_tc": [_P, _P, _P, _I, _I, _I, _P],
    "q2_gemm_tc_strided": [_P, _I, _P, _P, _I, _I, _I, _I, _P],
    "q2_gemm_mma": [_P, _P, _P, _I, _I, _I, _P],
    "q2_gemm_mma_strided": [_P, _I, _P, _P, _I, _I, _I, _I, _P],
    "w4a16_gemv": [_P, _P, _P, _P, _I, _I, _I, _P],
    "w4a16_gemv_ex": [_P, _I, _P, _P, _F, _P, _I, _I, _I, _I, _P],
    "w4a16_gemm_tc": [_P, _P, _P, _P, _I, _I, _I, _P],
    "w4a16_gemm_tc_ex": [_P, _I, _P, _P, _F, _P, _I, _I, _I, _I, _P],
    "w4a16_gemm_mma": [_P, _P, _P, _P, _I, _I, _I, _P],
    "w4a16_gemm_mma_ex": [_P, _I, _P, _P, _F, _P, _I, _I, _I, _I, _P],
    "w8a16_gemm": [_P, _P, _P, _P, _I, _I, _I, _P],
    "w8a16_gemm_strided": [_P, _I, _P, _P, _P, _I, _I, _I, _I, _P],
    "w8a16_gemm_tc": [_P, _P, _P, _P, _I, _I, _I, _P],
    "w8a16_gemm_tc_strided": [_P, _I, _P, _P, _P, _I, _I, _I, _I, _P],
    "w8a16_gemm_mma": [_P, _P, _P, _P, _I, _I, _I, _P],
    "w8a16_gemm_mma_strided": [_P, _I, _P, _P, _P, _I, _I, _I, _I, _P],
    "q2_dequant": [_P, _P, _I, _I, _P],
    "w4a16_dequant": [_P, _P, _F, _P, _I, _I, _P],
    "w8a16_dequant": [_P, _P, _P, _I, _I, _P],
    "wqp_row_chunks": [_I, _I, _I, _I, ctypes.POINTER(ctypes.c_longlong), _I],
    "wqp_set_pdl": [_I],
    "wqp_get_device_error": [],
    "wqp_selftest_wait_timeout": [_I, _P],
    "wqp_status_string": [_I],
    "wqp_last_error": [],
    "wqp_abi_version": [],
}

_lock = threading.Lock()
_lib = None


class WqpError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}" + (f" ({detail})" if detail else ""))


def lib() -> ctypes.CDLL:
    """Load libwqp.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(lib_path):
                raise ImportError(
                    f"libwqp.so not found at {lib_path}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(lib_path)
            for name, args in EXPORTS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = _I
            L.wqp_status_string.restype = ctypes.c_char_p
            L.wqp_last_error.restype = ctypes.c_char_p
            _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().wqp_status_string(int(status)).decode()
    except ImportError:
        return f"status {status}"


def _check(status: int, where: str):
    if status != 0:
        raise WqpError(status, where, lib().wqp_last_error().decode())


_current_stream = None   # () -> raw handle of this thread's current stream, set on first use
_BF16 = None


def _stream(stream):
    """The stream argument as an integer handle (ctypes converts it)."""
    global _current_stream
    if stream is None:
        if _current_stream is None:
            import torch

            # The current stream's raw handle; torch.cuda.current_stream()
            # builds a Python stream object, which costs about as much host
            # time as a launch.
            raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
            if raw is not None:
                dev = torch._C._cuda_getDevice
                _current_stream = lambda: raw(dev())
            else:
                _current_stream = lambda: torch.cuda.current_stream().cuda_stream
        return _current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    """A tensor's device address as an integer (None for no tensor)."""
    return t.data_ptr() if t is not None else None


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (no CPU fallback)")


def _out(A, M, N, out):
    import torch

    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    return out


def _rows(A, K):
    global _BF16
    if _BF16 is None:
        import torch

        _BF16 = torch.bfloat16
    if A.dtype is not _BF16:
        raise TypeError("A must be torch.bfloat16")
    if A.dim() != 2 or A.shape[1] != K or A.stride(1) != 1:
        raise ValueError(f"A must be [M, {K}] with unit column stride")
    return A.shape[0], A.stride(0)


def q2_gemv(A, W, N: int, K: int, out=None, stream=None):
    """C[M, N] = A @ dequant_q2(W)^T. W is uint8 Q2_0 blocks (34*K/128 B per row)."""
    _need_cuda(A, W, out)
    M, lda = _rows(A, K)
    C = _out(A, M, N, out)
    _check(lib().q2_gemv_strided(_ptr(A), lda, _ptr(W), _ptr(C), C.stride(0), M, N, K,
                                 _stream(stream)), "q2_gemv")
    return C


def q2_gemm_tc(A, W, N: int, K: int, out=None, stream=None):
    """Tensor-core (tcgen05 swap-AB) form of q2_gemv, 1 <= M <= 16, K % 1024 == 0."""
    _need_cuda(A, W, out)
    M, lda = _rows(A, K)
    C = _out(A, M, N, out)
    _check(lib().q2_gemm_tc_strided(_ptr(A), lda, _ptr(W), _ptr(C), C.stride(0), M, N, K,
                                    _stream(stream)), "q2_gemm_tc")
    return C


def q2_gemm_mma(A, W, N: int, K: int, out=None, stream=None):
    """Warp-level tensor-core (mma.sync swap-AB) form of q2_gemv, 1 <= M <= 16, K % 1024 == 0."""
    _need_cuda(A, W, out)
    M, lda = _rows(A, K)
    C = _out(A, M, N, out)
    _check(lib().q2_gemm_mma_strided(_ptr(A), lda, _ptr(W), _ptr(C), C.stride(0), M, N, K,
                                     _stream(stream)), "q2_gemm_mma")
    return C


def w4a16_gemv(A, W, scales, N: int, K: int, global_scale: float = 1.0, out=None, stream=None):
    """C = A @ dequant_w4(W, scales, global_scale)^T."""
    _need_cuda(A, W, scales, out)
    M, lda = _rows(A, K)
    C = _out(A, M, N, out)
    _check(lib().w4a16_gemv_ex(_ptr(A), lda, _ptr(W), _ptr(scales), float(global_scale), _ptr(C),
                               C.stride(0), M, N, K, _stream(stream)), "w4a16_gemv")
    return C


def w4a16_gemm_tc(A, W, scales, N: int, K: int, global_scale: float = 1.0, out=None, stream=None):
    """Tensor-core (tcgen05 swap-AB) form of w4a16_gemv, 1 <= M <= 16, K % 256 == 0."""
    _need_cuda(A, W, scales, out)
    M, lda = _rows(A, K)
    C = _out(A, M, N, out)
    _check(lib().w4a16_gemm_tc_ex(_ptr(A), lda, _ptr(W), _ptr(scales), float(global_scale), _ptr(C),
                                  C.stride(0), M, N, K, _stream(stream)), "w4a16_gemm_tc")
    return C


def w4a16_gemm_mma(A, W, scales, N: int, K: int, global_scale: float = 1.0, out=None, stream=None):
    """Warp-level tensor-core (mma.sync swap-AB) form of w4a16_gemv, K % 1024 == 0."""
    _need_cuda(A, W, scales, out)
    M, lda = _rows(A, K)
    C = _out(A, M, N, out)
    _check(lib().w4a16_gemm_mma_ex(_ptr(A), lda, _ptr(W), _ptr(scales), float(global_scale), _ptr(C),
                                   C.stride(0), M, N, K, _stream(stream)), "w4a16_gemm_mma")
    return C


def w8a16_gemm_mma(A, W, scales, N: int, K: int, out=None, stream=None):
    """Warp-level tensor-core (mma.sync swap-AB) form of w8a16_gemm, K % 1024 == 0."""
    _need_cuda(A, W, scales, out)
    M, lda = _rows(A, K)
    C = _out(A, M, N, out)
    _check(lib().w8a16_gemm_mma_strided(_ptr(A), lda, _ptr(W), _ptr(scales), _ptr(C), C.stride(0),
                                        M, N, K, _stream(stream)), "w8a16_gemm_mma")
    return C


def w8a16_gemm(A, W, scales, N: int, K: int, out=None, stream=None):
    """C = A @ (e4m3(W) * block_scales)^T, scalar-FMA kernels."""
    _need_cuda(A, W, scales, out)
    M, lda = _rows(A, K)
    C = _out(A, M, N, out)
    _check(lib().w8a16_gemm_strided(_ptr(A), lda, _ptr(W), _ptr(scales), _ptr(C), C.stride(0),
                                    M, N, K, _stream(stream)), "w8a16_gemm")
    return C


def w8a16_gemm_tc(A, W, scales, N: int, K: int, out=None, stream=None):
    """Tensor-core (tcgen05 swap-AB) form of w8a16_gemm, 1 <= M <= 16."""
    _need_cuda(A, W, scales, out)
    M, lda = _rows(A, K)
    C = _out(A, M, N, out)
    _check(lib().w8a16_gemm_tc_strided(_ptr(A), lda, _ptr(W), _ptr(scales), _ptr(C), C.stride(0),
                                       M, N, K, _stream(stream)), "w8a16_gemm_tc")
    return C


def _deq_out(W, N, K, out):
    import torch

    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=W.device)
    return out


def q2_dequant(W, N: int, K: int, out=None, stream=None):
    _need_cuda(W, out)
    o = _deq_out(W, N, K, out)
    _check(lib().q2_dequant(_ptr(W), _ptr(o), N, K, _stream(stream)), "q2_dequant")
    return o


def w4a16_dequant(W, scales, N: int, K: int, global_scale: float = 1.0, out=None, stream=None):
    _need_cuda(W, scales, out)
    o = _deq_out(W, N, K, out)
    _check(lib().w4a16_dequant(_ptr(W), _ptr(scales), float(global_scale), _ptr(o), N, K,
                               _stream(stream)), "w4a16_dequant")
    return o


def w8a16_dequant(W, scales, N: int, K: int, out=None, stream=None):
    _need_cuda(W, scales, out)
    o = _deq_out(W, N, K, out)
    _check(lib().w8a16_dequant(_ptr(W), _ptr(scales), _ptr(o), N, K, _stream(stream)),
           "w8a16_dequant")
    return o


def row_chunks(M: int, K: int, N: int, max_rows: int):
    """Host-side row chunking: list of (a_byte_offset, c_byte_offset, rows)."""
    cap = max(1, (M + max(max_rows, 1) - 1) // max(max_rows, 1))
    buf = (ctypes.c_longlong * (3 * cap))()
    n = lib().wqp_row_chunks(M, K, N, max_rows, buf, cap)
    if n < 0:
        raise ValueError("invalid row_chunks arguments")
    return [(buf[3 * i], buf[3 * i + 1], buf[3 * i + 2]) for i in range(n)]


def set_pdl(enable: bool) -> bool:
    """Process-wide programmatic-dependent-launch policy; returns the old one."""
    return bool(lib().wqp_set_pdl(1 if enable else 0))


def get_device_error() -> int:
    """Read and clear the device error word (synchronises the device)."""
    return lib().wqp_get_device_error()


def selftest_wait_timeout(limit_us: int = 2000, stream=None) -> None:
    """Launch the failure-path self-test: a kernel whose bounded wait on a
    barrier nothing completes gives up after limit_us microseconds and records
    the timeout in the device error word (read it with get_device_error())."""
    _check(lib().wqp_selftest_wait_timeout(int(limit_us), _stream(stream)), "wqp_selftest_wait_timeout")
