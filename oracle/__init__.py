"""ctypes front end of the CPU oracle (``oracle.c`` -> ``liboracle.so``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg use it; the product package never imports it.

All arrays are numpy; BF16 values travel as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
          "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (fp contraction off) if it is stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            F = ctypes.c_float
            for name, args in {
                "oracle_q2_gemv": [P, P, I, I, I, P, P, P],
                "oracle_w4_gemv": [P, P, P, F, I, I, I, P, P, P],
                "oracle_w8_gemm": [P, P, P, I, I, I, P, P, P],
                "oracle_q2_dequant": [P, I, I, P],
                "oracle_w4_dequant": [P, P, F, I, I, P],
                "oracle_w8_dequant": [P, P, I, I, P],
                "oracle_set_threads": [I],
            }.items():
                getattr(lib, name).argtypes = args
                getattr(lib, name).restype = None
            lib.oracle_max_threads.restype = I
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f32.restype = F
            lib.oracle_f32_to_bf16.argtypes = [F]
            lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f32.restype = F
            lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_f32.restype = F
            lib.oracle_e2m1_to_f32.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_to_f32.restype = F
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return _load().oracle_max_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


class Result:
    """BF16 output bits plus the fp64 sum R and magnitude sum S per output."""

    def __init__(self, c, r, s):
        self.c, self.r, self.s = c, r, s


def q2_gemv(A, W, M, N, K) -> Result:
    A = _c(A, np.uint16).reshape(M, K)
    W = _c(W, np.uint8)
    assert W.size == N * (K // 128) * 34
    C = np.zeros((M, N), np.uint16)
    R = np.zeros((M, N), np.float64)
    S = np.zeros((M, N), np.float64)
    _load().oracle_q2_gemv(_p(A), _p(W), M, N, K, _p(C), _p(R), _p(S))
    return Result(C, R, S)


def w4_gemv(A, codes, scales, g, M, N, K) -> Result:
    A = _c(A, np.uint16).reshape(M, K)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    assert codes.size == N * K // 2 and scales.size == N * K // 16
    C = np.zeros((M, N), np.uint16)
    R = np.zeros((M, N), np.float64)
    S = np.zeros((M, N), np.float64)
    _load().oracle_w4_gemv(_p(A), _p(codes), _p(scales), float(g), M, N, K, _p(C), _p(R), _p(S))
    return Result(C, R, S)


def w8_gemm(A, w, bs, M, N, K) -> Result:
    A = _c(A, np.uint16).reshape(M, K)
    w = _c(w, np.uint8)
    bs = _c(bs, np.float32)
    assert w.size == N * K and bs.size == ((N + 127) // 128) * (K // 128)
    C = np.zeros((M, N), np.uint16)
    R = np.zeros((M, N), np.float64)
    S = np.zeros((M, N), np.float64)
    _load().oracle_w8_gemm(_p(A), _p(w), _p(bs), M, N, K, _p(C), _p(R), _p(S))
    return Result(C, R, S)


def q2_dequant(W, N, K) -> np.ndarray:
    W = _c(W, np.uint8)
    out = np.zeros((N, K), np.float32)
    _load().oracle_q2_dequant(_p(W), N, K, _p(out))
    return out


def w4_dequant(codes, scales, g, N, K) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    out = np.zeros((N, K), np.float32)
    _load().oracle_w4_dequant(_p(codes), _p(scales), float(g), N, K, _p(out))
    return out


def w8_dequant(w, bs, N, K) -> np.ndarray:
    w = _c(w, np.uint8)
    bs = _c(bs, np.float32)
    out = np.zeros((N, K), np.float32)
    _load().oracle_w8_dequant(_p(w), _p(bs), N, K, _p(out))
    return out


def bf16_to_f32(b: int) -> float:
    return _load().oracle_bf16_to_f32(int(b))


def f32_to_bf16(x: float) -> int:
    return _load().oracle_f32_to_bf16(float(x))


def f16_to_f32(h: int) -> float:
    return _load().oracle_f16_to_f32(int(h))


def e4m3_to_f32(b: int) -> float:
    return _load().oracle_e4m3_to_f32(int(b))


def e2m1_to_f32(n: int) -> float:
    return _load().oracle_e2m1_to_f32(int(n))
