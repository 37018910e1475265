"""Parity of the scalar-FMA CUDA kernels with the CPU oracle (GPU needed).

Scalar tolerance (tests/_tol.py): 1 BF16 ULP, or the FP32 reordering floor
8 * sqrt(K) * 2^-24 * sum|a*w|. Exact-arithmetic inputs and the dequant
entries are compared bit for bit, and so is each batched row against the M=1
call, the invariant of "gemv_q2_vec.rs" (doc of `q2_0_gemv_vec_batchm`) and
"w4a16_gemv_tiers.rs" (doc of `select_tier`).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests import _gpu as G
from tests._tol import assert_scalar_term, bf16_exact_bits, bf16_to_f64
from weight_only_quantized_packed_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__

    __graft_entry__.build()
    import weight_only_quantized_packed_gb300 as wqp

    wqp.set_pdl(False)
    yield
    assert wqp.get_device_error() == 0


FMTS = ["q2", "w4", "w8"]
SHAPES = [  # (N, K): tails, single group, several K tiles, ragged last tile
    (1, 128), (5, 256), (8, 512), (9, 384), (37, 1024), (256, 512), (130, 2048),
    (1000, 1152), (77, 3200), (264, 5120),
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,K", SHAPES)
def test_parity_small(oracle_lib, fmt, N, K):
    for M in (1, 3, 8, 16):
        d = G.make(fmt, M, N, K, seed=1000 + N + K + M)
        C = G.host_bits(G.run_gpu(d))
        ref = G.run_oracle(oracle_lib, d)
        assert_scalar_term(C, ref, K, f"{fmt} M={M} N={N} K={K}")


@pytest.mark.parametrize("fmt", FMTS)
def test_every_m_bit_identical_to_m1(fmt):
    """Each row of an M-row call equals the M=1 call on that row, for M=1..16."""
    N, K = 200, 2048
    d = G.make(fmt, 16, N, K, seed=77)
    rows1 = [G.host_bits(G.run_gpu(d, A=d["dA"][m:m + 1]))[0] for m in range(16)]
    for M in range(1, 17):
        C = G.host_bits(G.run_gpu(d, A=d["dA"][:M]))
        for m in range(M):
            assert np.array_equal(C[m], rows1[m]), (fmt, M, m)


@pytest.mark.parametrize("fmt", FMTS)
def test_m_above_16_is_chunked(oracle_lib, fmt):
    N, K = 40, 512
    for M in (17, 33):
        d = G.make(fmt, M, N, K, seed=5 + M)
        C = G.host_bits(G.run_gpu(d))
        ref = G.run_oracle(oracle_lib, d)
        assert_scalar_term(C, ref, K, f"{fmt} M={M}")
        one = G.host_bits(G.run_gpu(d, A=d["dA"][M - 1:M]))
        assert np.array_equal(C[M - 1], one[0])


@pytest.mark.parametrize("fmt", FMTS)
def test_exact_arithmetic_bit_exact(oracle_lib, fmt):
    """Small-integer activations and power-of-two scales make every order of
    summation exact: GPU == oracle == bf16(exact sum), bit for bit."""
    r = np.random.default_rng(3)
    M, N, K = 5, 300, 2048
    a = r.integers(-4, 5, size=(M, K)).astype(np.float32)
    A = synth.bf16_bits_from_f32(a)
    d = {"A": A, "dA": G.dev_bf16(A), "M": M, "N": N, "K": K, "fmt": fmt}
    if fmt == "q2":
        codes = r.integers(0, 3, size=(N, K), dtype=np.uint8)
        dd = (2.0 ** -r.integers(2, 6, size=(N, K // 128))).astype(np.float16)
        W = synth.pack_q2(codes, dd)
        d.update(W=W, dW=G.dev_u8(W))
    elif fmt == "w4":
        nib = r.integers(0, 16, size=(N, K), dtype=np.uint8)
        S = synth.e4m3_round(2.0 ** r.integers(-3, 2, size=(N, K // 16)))
        W = synth.pack_w4(nib)
        d.update(W=W, S=S, dW=G.dev_u8(W), dS=G.dev_u8(S), g=1.0)
    else:
        W = synth.e4m3_round(r.integers(-16, 17, size=(N, K)) / 8.0)
        S = (2.0 ** r.integers(-2, 3, size=((N + 127) // 128, K // 128))).astype(np.float32)
        d.update(W=W, S=S, dW=G.dev_u8(W), dS=G.dev_f32(S))
    C = G.host_bits(G.run_gpu(d))
    ref = G.run_oracle(oracle_lib, d)
    assert np.array_equal(C, ref.c)
    assert np.array_equal(bf16_to_f64(C), bf16_to_f64(bf16_exact_bits(ref.r)))


def test_q2_code3_and_closed_form(oracle_lib):
    """All-ones A, all codes 2, uniform d -> K*d exactly; code 3 -> +2d."""
    N, K = 24, 5120
    d16 = np.float16(0.0371)
    W = synth.pack_q2(np.full((N, K), 2, np.uint8), np.full((N, K // 128), d16, np.float16))
    A = synth.bf16_bits_from_f32(np.ones((1, K), np.float32))
    C = G.host_bits(G.run_gpu({"dA": G.dev_bf16(A), "dW": G.dev_u8(W), "N": N, "K": K, "fmt": "q2"}))
    assert np.array_equal(C, bf16_exact_bits(np.full((1, N), K * float(d16))))
    W3 = synth.pack_q2(np.full((N, K), 3, np.uint8), np.full((N, K // 128), 0.25, np.float16))
    A1 = np.zeros((1, K), np.float32)
    A1[0, 4097] = 1.0
    C3 = G.host_bits(G.run_gpu({"dA": G.dev_bf16(synth.bf16_bits_from_f32(A1)), "dW": G.dev_u8(W3),
                                "N": N, "K": K, "fmt": "q2"}))
    assert np.array_equal(C3, bf16_exact_bits(np.full((1, N), 0.5)))


@pytest.mark.parametrize("fmt", FMTS)
def test_activation_range(oracle_lib, fmt):
    """Activations scaled by 2^40 and 2^-40: within the Q2_0 kernel's stated
    range (pre-scaled activations finite for |a| < 2^48, products normal for
    |a| >= 2^-57); the other formats take any finite activation."""
    for scale in (2.0 ** 40, 2.0 ** -40):
        M, N, K = 4, 300, 2048
        d = G.make(fmt, M, N, K, seed=91)
        d["A"] = synth.activations(M, K, 92, scale=scale)
        d["dA"] = G.dev_bf16(d["A"])
        C = G.host_bits(G.run_gpu(d))
        assert_scalar_term(C, G.run_oracle(oracle_lib, d), K, f"{fmt} activation scale {scale:g}")


@pytest.mark.parametrize("fmt", FMTS)
def test_strided_rows_and_canary(oracle_lib, fmt):
    """Row pitches lda > K and ldc > N; bytes outside C's rows stay untouched."""
    M, N, K = 6, 70, 1024
    d = G.make(fmt, M, N, K, seed=9)
    lda, ldc = K + 64, N + 13
    Abig = torch.zeros((M, lda), dtype=torch.bfloat16, device="cuda")
    Abig[:, :K] = d["dA"]
    canary = torch.full((M + 2, ldc), -7.0, dtype=torch.bfloat16, device="cuda")
    out = canary[1:M + 1].as_strided((M, N), (ldc, 1))
    G.run_gpu(d, A=Abig[:, :K], out=out)
    host = canary.float().cpu().numpy()
    assert (host[0] == -7.0).all() and (host[M + 1] == -7.0).all()
    assert (host[1:M + 1, N:] == -7.0).all()
    C = G.host_bits(canary[1:M + 1, :N].contiguous())
    ref = G.run_oracle(oracle_lib, d)
    assert_scalar_term(C, ref, K, f"{fmt} strided")


def test_dequant_bit_exact(oracle_lib):
    """GPU dequant == oracle dequant bit for bit, over every Q2 code (with
    code 3), all 16 E2M1 nibbles and all 256 E4M3 bytes."""
    import weight_only_quantized_packed_gb300 as wqp

    N, K = 24, 512
    r = np.random.default_rng(0)
    codes = r.integers(0, 4, size=(N, K), dtype=np.uint8)
    dd = r.uniform(-0.3, 0.3, size=(N, K // 128)).astype(np.float16)
    W = synth.pack_q2(codes, dd)
    got = wqp.q2_dequant(G.dev_u8(W), N, K).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), oracle_lib.q2_dequant(W, N, K).view(np.uint32))

    nib = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    S = np.arange(N * K // 16, dtype=np.uint32).astype(np.uint8).reshape(N, K // 16)
    S[S == 0x7F] = 0x7E
    S[S == 0xFF] = 0xFE
    for g in (1.0, 0.75):
        got = wqp.w4a16_dequant(G.dev_u8(synth.pack_w4(nib)), G.dev_u8(S), N, K, g).cpu().numpy()
        exp = oracle_lib.w4_dequant(synth.pack_w4(nib), S, g, N, K)
        assert np.array_equal(got.view(np.uint32), exp.view(np.uint32)), g

    W8 = np.tile(np.arange(256, dtype=np.uint32).astype(np.uint8), (N, K // 256))
    W8[W8 == 0x7F] = 0x7E
    W8[W8 == 0xFF] = 0xFE
    S8 = r.uniform(0.5, 2.0, size=(1, K // 128)).astype(np.float32)
    got = wqp.w8a16_dequant(G.dev_u8(W8), G.dev_f32(S8), N, K).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), oracle_lib.w8_dequant(W8, S8, N, K).view(np.uint32))


@pytest.mark.parametrize("fmt,N,K,Ms", [
    ("q2", 5120, 5120, (1, 4, 8)),                 # 27B qkv/o projection shape
    ("w4", 5120, 5120, (1, 5, 8)),
    ("w8", 17408, 5120, (1, 16)),                  # dense FFN gate/up
    ("w8", 5120, 17408, (2, 16)),                  # dense FFN down
    ("q2", 5120, 17408, (16,)),
])
def test_full_size_parity(oracle_lib, fmt, N, K, Ms):
    for M in Ms:
        d = G.make(fmt, M, N, K, seed=synth.seed_for(7, M))
        C = G.host_bits(G.run_gpu(d))
        ref = G.run_oracle(oracle_lib, d)
        assert_scalar_term(C, ref, K, f"{fmt} full M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [1, 8])
def test_pdl_launch_same_result(M):
    """Back-to-back launches with programmatic dependent launch give the same
    bits as a launch without it."""
    import weight_only_quantized_packed_gb300 as wqp

    d = G.make("q2", M, 640, 5120, seed=4)
    base = G.host_bits(G.run_gpu(d))
    wqp.set_pdl(True)
    try:
        outs = [G.run_gpu(d) for _ in range(4)]
    finally:
        wqp.set_pdl(False)
    for o in outs:
        assert np.array_equal(G.host_bits(o), base)
