"""Helpers for the GPU tests: move numpy inputs to the device and call the
CUDA path through the ctypes binding (the C ABI)."""
from __future__ import annotations

import numpy as np
import torch

import weight_only_quantized_packed_gb300 as wqp
from weight_only_quantized_packed_gb300 import synth

DEV = "cuda"


def dev_u8(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint8)).to(DEV)


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).to(DEV).view(torch.bfloat16)


def dev_f32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV)


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def make(fmt: str, M: int, N: int, K: int, seed: int):
    """Seeded inputs of one format; returns a dict with host and device arrays."""
    A = synth.activations(M, K, seed)
    d = {"A": A, "dA": dev_bf16(A), "M": M, "N": N, "K": K, "fmt": fmt}
    if fmt == "q2":
        W, _, _ = synth.q2_weights(N, K, seed + 1)
        d.update(W=W, dW=dev_u8(W))
    elif fmt == "w4":
        W, S, _ = synth.w4_weights(N, K, seed + 1)
        d.update(W=W, S=S, dW=dev_u8(W), dS=dev_u8(S), g=1.0)
    elif fmt == "w8":
        W, S = synth.w8_weights(N, K, seed + 1)
        d.update(W=W, S=S, dW=dev_u8(W), dS=dev_f32(S))
    return d


def run_gpu(d, tc: bool = False, A=None, out=None):
    A = d["dA"] if A is None else A
    N, K = d["N"], d["K"]
    if d["fmt"] == "q2" and tc == "mma":
        C = wqp.q2_gemm_mma(A, d["dW"], N, K, out=out)
    elif d["fmt"] == "q2" and tc:
        C = wqp.q2_gemm_tc(A, d["dW"], N, K, out=out)
    elif d["fmt"] == "q2":
        C = wqp.q2_gemv(A, d["dW"], N, K, out=out)
    elif d["fmt"] == "w4" and tc == "mma":
        C = wqp.w4a16_gemm_mma(A, d["dW"], d["dS"], N, K, d.get("g", 1.0), out=out)
    elif d["fmt"] == "w4" and tc:
        C = wqp.w4a16_gemm_tc(A, d["dW"], d["dS"], N, K, d.get("g", 1.0), out=out)
    elif d["fmt"] == "w4":
        C = wqp.w4a16_gemv(A, d["dW"], d["dS"], N, K, d.get("g", 1.0), out=out)
    elif tc == "mma":
        C = wqp.w8a16_gemm_mma(A, d["dW"], d["dS"], N, K, out=out)
    elif tc:
        C = wqp.w8a16_gemm_tc(A, d["dW"], d["dS"], N, K, out=out)
    else:
        C = wqp.w8a16_gemm(A, d["dW"], d["dS"], N, K, out=out)
    torch.cuda.synchronize()
    return C


def run_oracle(oracle, d, A=None):
    A = d["A"] if A is None else A
    M = A.shape[0]
    N, K = d["N"], d["K"]
    if d["fmt"] == "q2":
        return oracle.q2_gemv(A, d["W"], M, N, K)
    if d["fmt"] == "w4":
        return oracle.w4_gemv(A, d["W"], d["S"], d.get("g", 1.0), M, N, K)
    return oracle.w8_gemm(A, d["W"], d["S"], M, N, K)
