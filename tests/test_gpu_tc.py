"""Parity of the tensor-core GEMMs (tcgen05 for W8A16, Q2_0 and W4A16; the
warp-level MMA for Q2_0) with the CPU oracle (GPU needed).

Terms:
* Q2_0 and W4A16: every product entering the MMA is exact (c * a * 2^-69 for
  Q2_0; e2m1 * e4m3 * a for W4), only the order of the FP32 additions
  differs from the oracle's, so these engines are held to the scalar term:
  1 BF16 ULP, or the FP32 reordering floor 8 * sqrt(K) * 2^-24 * sum|a*w|,
  with the share of outputs that pass only by the floor bounded and logged.
* FP8 (W8A16) tensor core ("w8a16_gemm_m16.rs", module docs: within a few
  BF16 ULP of the reference or under an absolute floor set by the reduction
  depth and the row's RMS): at most 4 BF16 ULP, or
  |gpu - oracle| < 1e-3 * sqrt(K) * rms(a[m,:]) * max_k |w[n,k]|, with w
  including its block scale.
Exact-arithmetic inputs must match bit for bit on every engine.
"""
from __future__ import annotations

import numpy as np
import pytest

from tests import _gpu as G
from tests._tol import assert_scalar_term, bf16_exact_bits, bf16_to_f64, log_parity, parity_report, tc_ok
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


def _check_tc(oracle_lib, d, C, what):
    """Q2_0, W4 and the FP8 warp-level MMA path: the scalar term on every
    output. FP8 on tcgen05: the tensor-core term, and the share within the
    scalar term is returned."""
    ref = G.run_oracle(oracle_lib, d)
    if d["fmt"] in ("q2", "w4") or "mma" in what:
        assert_scalar_term(C, ref, d["K"], what)
        return 1.0
    a = synth.bf16_bits_to_f32(d["A"]).astype(np.float64)
    a_rms = np.sqrt((a ** 2).mean(axis=1))
    w_max = np.abs(oracle_lib.w8_dequant(d["W"], d["S"], d["N"], d["K"])).max(axis=1)
    ok = tc_ok(C, ref, d["K"], a_rms, w_max)
    bad = np.argwhere(~ok)
    assert bad.size == 0, (what, len(bad), bad[:3], bf16_to_f64(C[tuple(bad[0])]),
                           bf16_to_f64(ref.c[tuple(bad[0])]))
    rep = parity_report(C, ref, d["K"])
    log_parity(what + " (fp8 tensor core)", rep)
    return 1.0 - rep["fail"] / rep["n"]


@pytest.mark.parametrize("N,K", [(128, 128), (200, 512), (1000, 1024), (384, 2048), (77, 640)])
def test_tc_parity_small(oracle_lib, N, K):
    for M in (1, 5, 16):
        d = G.make("w8", M, N, K, seed=300 + N + K + M)
        C = G.host_bits(G.run_gpu(d, tc=True))
        _check_tc(oracle_lib, d, C, f"M={M} N={N} K={K}")


def test_tc_exact_arithmetic_bit_exact(oracle_lib):
    r = np.random.default_rng(5)
    M, N, K = 16, 300, 2048
    a = r.integers(-4, 5, size=(M, K)).astype(np.float32)
    A = synth.bf16_bits_from_f32(a)
    W = synth.e4m3_round(r.integers(-16, 17, size=(N, K)) / 8.0)
    S = (2.0 ** r.integers(-2, 3, size=((N + 127) // 128, K // 128))).astype(np.float32)
    d = {"A": A, "dA": G.dev_bf16(A), "M": M, "N": N, "K": K, "fmt": "w8", "W": W, "S": S,
         "dW": G.dev_u8(W), "dS": G.dev_f32(S)}
    C = G.host_bits(G.run_gpu(d, tc=True))
    assert np.array_equal(C, G.run_oracle(oracle_lib, d).c)


def test_tc_split_k_deterministic_and_row_independent():
    """N = 640 splits K over a cluster; repeated calls give identical bits and
    each row does not depend on the other activation rows."""
    d = G.make("w8", 16, 640, 5120, seed=11)
    c1 = G.host_bits(G.run_gpu(d, tc=True))
    c2 = G.host_bits(G.run_gpu(d, tc=True))
    assert np.array_equal(c1, c2)
    one = G.host_bits(G.run_gpu(d, tc=True, A=d["dA"][3:4]))
    assert np.array_equal(one[0], c1[3])


@pytest.mark.parametrize("N,K,Ms", [(17408, 5120, (16, 1)), (5120, 17408, (16, 8))])
def test_tc_full_size(oracle_lib, N, K, Ms):
    for M in Ms:
        d = G.make("w8", M, N, K, seed=synth.seed_for(3, M))
        C = G.host_bits(G.run_gpu(d, tc=True))
        frac = _check_tc(oracle_lib, d, C, f"full M={M} N={N} K={K}")
        assert frac > 0.99   # almost every output is also within the scalar 1-ULP term


# ------------------------------------------------------------------ Q2_0
# Both tensor-core engines: tcgen05 through tensor memory (q2_gemm_tc) and the
# warp-level mma.sync path (q2_gemm_mma).
ENGINES = pytest.mark.parametrize("eng", [True, "mma"], ids=["tcgen05", "mma_sync"])


@pytest.mark.parametrize("N,K", [(128, 1024), (200, 2048), (1000, 1024), (77, 3072), (384, 8192)])
@ENGINES
def test_q2_tc_parity_small(oracle_lib, N, K, eng):
    for M in (1, 4, 16):
        d = G.make("q2", M, N, K, seed=500 + N + K + M)
        C = G.host_bits(G.run_gpu(d, tc=eng))
        _check_tc(oracle_lib, d, C, f"q2 M={M} N={N} K={K} {eng}")


@ENGINES
def test_q2_tc_exact_arithmetic_bit_exact(oracle_lib, eng):
    """Codes 0..3 (weights -1, 0, 1 and, for code 3, +2) times small
    integers, power-of-two d: exact in any order."""
    r = np.random.default_rng(8)
    M, N, K = 16, 260, 3072
    a = r.integers(-4, 5, size=(M, K)).astype(np.float32)
    A = synth.bf16_bits_from_f32(a)
    codes = r.integers(0, 4, size=(N, K), dtype=np.uint8)
    dd = (2.0 ** -r.integers(2, 6, size=(N, K // 128))).astype(np.float16)
    W = synth.pack_q2(codes, dd)
    d = {"A": A, "dA": G.dev_bf16(A), "M": M, "N": N, "K": K, "fmt": "q2", "W": W, "dW": G.dev_u8(W)}
    C = G.host_bits(G.run_gpu(d, tc=eng))
    assert np.array_equal(C, G.run_oracle(oracle_lib, d).c)


@ENGINES
def test_q2_tc_closed_form_and_code3(eng):
    """All-ones A with every code 2 and one d gives K*d exactly (every partial
    sum is exact for K <= 8192); code 3 decodes to +2d (one-hot A)."""
    N, K = 200, 5120
    d16 = np.float16(0.0371)
    W = synth.pack_q2(np.full((N, K), 2, np.uint8), np.full((N, K // 128), d16, np.float16))
    for M in (1, 8, 16):
        A = synth.bf16_bits_from_f32(np.ones((M, K), np.float32))
        C = G.host_bits(G.run_gpu({"dA": G.dev_bf16(A), "dW": G.dev_u8(W), "N": N, "K": K, "fmt": "q2"}, tc=eng))
        assert np.array_equal(C, bf16_exact_bits(np.full((M, N), K * float(d16)))), M
    W3 = synth.pack_q2(np.full((N, K), 3, np.uint8), np.full((N, K // 128), 0.25, np.float16))
    for j in (0, 1, 7, 8, 15, 4097, K - 1):      # every position class of a code in its word
        A1 = np.zeros((2, K), np.float32)
        A1[0, j] = 1.0
        A1[1, j] = -3.0
        C3 = G.host_bits(G.run_gpu({"dA": G.dev_bf16(synth.bf16_bits_from_f32(A1)), "dW": G.dev_u8(W3),
                                    "N": N, "K": K, "fmt": "q2"}, tc=eng))
        exp = np.stack([np.full(N, 0.5), np.full(N, -1.5)])
        assert np.array_equal(C3, bf16_exact_bits(exp)), j


@ENGINES
def test_q2_tc_rows_independent_and_k_rule(eng):
    import weight_only_quantized_packed_gb300 as wqp

    d = G.make("q2", 16, 5120, 5120, seed=21)
    c16 = G.host_bits(G.run_gpu(d, tc=eng))
    for m in (0, 7, 15):
        one = G.host_bits(G.run_gpu(d, tc=eng, A=d["dA"][m:m + 1]))
        assert np.array_equal(one[0], c16[m])
    bad = G.make("q2", 1, 64, 640, seed=2)
    with pytest.raises(wqp.WqpError):
        G.run_gpu(bad, tc=eng)          # K % 1024 != 0


@pytest.mark.parametrize("N,K,Ms", [(5120, 5120, (1, 4, 8, 16)), (7168, 5120, (8,)),
                                    (5120, 17408, (16,)), (34816, 5120, (4, 16))])
@ENGINES
def test_q2_tc_full_size(oracle_lib, N, K, Ms, eng):
    for M in Ms:
        d = G.make("q2", M, N, K, seed=synth.seed_for(1, M))
        C = G.host_bits(G.run_gpu(d, tc=eng))
        _check_tc(oracle_lib, d, C, f"q2 full M={M} N={N} K={K} {eng}")


def test_q2_mma_persistent_rows_independent():
    """The dense-FFN gate+up shape runs on the persistent kernel: a row of a
    16-row call (two column tiles, weights read once) equals the row computed
    alone, and a 12-row call gives the same rows."""
    d = G.make("q2", 16, 34816, 5120, seed=24)
    c16 = G.host_bits(G.run_gpu(d, tc="mma"))
    c12 = G.host_bits(G.run_gpu(d, tc="mma", A=d["dA"][:12]))
    assert np.array_equal(c12, c16[:12])
    for m in (0, 9, 15):
        one = G.host_bits(G.run_gpu(d, tc="mma", A=d["dA"][m:m + 1]))
        assert np.array_equal(one[0], c16[m]), m


@pytest.mark.parametrize("K", [1024, 2048])
def test_q2_mma_persistent_register_fragments(oracle_lib, K):
    """Persistent plans whose ranks own one stage each (B fragments kept in
    registers): N = 20000 (persistent, a ragged last tile) at K = 1024 and
    2048, 5 and 16 rows; parity with the oracle and rows equal to the rows
    computed alone."""
    N = 20000
    for M in (5, 16):
        d = G.make("q2", M, N, K, seed=37 + M + K)
        C = G.host_bits(G.run_gpu(d, tc="mma"))
        _check_tc(oracle_lib, d, C, f"q2 persistent M={M} N={N} K={K} mma")
        for m in (0, M - 1):
            one = G.host_bits(G.run_gpu(d, tc="mma", A=d["dA"][m:m + 1]))
            assert np.array_equal(one[0], C[m]), (M, m)


def test_q2_mma_tall_tiles_ragged(oracle_lib):
    """A shape whose single-stage grid of 64-row CTAs would need a fourth CTA
    slot per SM runs as 96-row CTAs (N = 7000, K = 5120: a partial last
    96-row tile and a partial 16-row tile); parity with the oracle, and rows
    equal to the rows computed alone."""
    N, K = 7000, 5120
    d = G.make("q2", 8, N, K, seed=33)
    c8 = G.host_bits(G.run_gpu(d, tc="mma"))
    _check_tc(oracle_lib, d, c8, f"q2 96-row tiles M=8 N={N} K={K} mma")
    for m in (0, 3, 7):
        one = G.host_bits(G.run_gpu(d, tc="mma", A=d["dA"][m:m + 1]))
        assert np.array_equal(one[0], c8[m]), m


def test_q2_mma_tile_height_keeps_rows():
    """The tile height changes no row's summation order: rows of a call run
    on 96-row CTAs (N = 7000) equal the same rows of the same weights run on
    64-row CTAs (N = 5120, the first 5120 rows), bit for bit."""
    d = G.make("q2", 8, 7000, 5120, seed=35)
    c96 = G.host_bits(G.run_gpu(d, tc="mma"))
    c64 = G.host_bits(G.run_gpu(dict(d, N=5120), tc="mma"))
    assert np.array_equal(c64, c96[:, :5120])


def test_q2_mma_paired_ragged(oracle_lib):
    """A ragged shape on the persistent kernel's paired 16-row plan (no K
    split, B fragments shared by two CTAs): N = 20001 leaves a partial last
    tile; parity with the oracle, and rows equal to the rows computed alone."""
    N, K = 20001, 5120
    d = G.make("q2", 16, N, K, seed=31)
    c16 = G.host_bits(G.run_gpu(d, tc="mma"))
    _check_tc(oracle_lib, d, c16, f"q2 paired M=16 N={N} K={K} mma")
    for m in (0, 7, 8, 15):
        one = G.host_bits(G.run_gpu(d, tc="mma", A=d["dA"][m:m + 1]))
        assert np.array_equal(one[0], c16[m]), m


@ENGINES
def test_q2_tc_activation_range(oracle_lib, eng):
    """The pre-scale 2^(64 - 2j) stays exact for large and small activations
    (|a| up to 2^40 and down to 2^-40), within the stated range."""
    for scale in (2.0 ** 40, 2.0 ** -40):
        M, N, K = 4, 300, 2048
        A = synth.activations(M, K, 77, scale=scale)
        W, _, _ = synth.q2_weights(N, K, 78)
        d = {"A": A, "dA": G.dev_bf16(A), "M": M, "N": N, "K": K, "fmt": "q2", "W": W, "dW": G.dev_u8(W)}
        C = G.host_bits(G.run_gpu(d, tc=eng))
        _check_tc(oracle_lib, d, C, f"q2 activation scale {scale:g}")


@ENGINES
def test_q2_tc_strided_rows_and_canary(oracle_lib, eng):
    """Row pitches lda > K and ldc > N, ragged N; bytes outside C's rows stay
    untouched."""
    import torch

    M, N, K = 6, 200, 2048
    d = G.make("q2", M, N, K, seed=19)
    lda, ldc = K + 64, N + 13
    Abig = torch.zeros((M, lda), dtype=torch.bfloat16, device="cuda")
    Abig[:, :K] = d["dA"]
    canary = torch.full((M + 2, ldc), -7.0, dtype=torch.bfloat16, device="cuda")
    out = canary[1:M + 1].as_strided((M, N), (ldc, 1))
    G.run_gpu(d, tc=eng, A=Abig[:, :K], out=out)
    host = canary.float().cpu().numpy()
    assert (host[0] == -7.0).all() and (host[M + 1] == -7.0).all()
    assert (host[1:M + 1, N:] == -7.0).all()
    C = G.host_bits(canary[1:M + 1, :N].contiguous())
    _check_tc(oracle_lib, d, C, "q2 strided")


@ENGINES
def test_q2_tc_dependent_chain_under_pdl(eng):
    """x_{i+1} = q2(x_i) with N = K: each call reads the previous call's
    output and overwrites the buffer the call before it read. Launched with
    programmatic dependent launch, the chain gives the same bits as without
    it (the grid-dependency wait orders both)."""
    import torch
    import weight_only_quantized_packed_gb300 as wqp

    M, N = 4, 5120
    d = G.make("q2", M, N, N, seed=33)

    f = wqp.q2_gemm_mma if eng == "mma" else wqp.q2_gemm_tc

    def chain():
        bufs = [d["dA"].clone(), torch.empty_like(d["dA"])]
        for i in range(6):
            f(bufs[i % 2], d["dW"], N, N, out=bufs[(i + 1) % 2])
        torch.cuda.synchronize()
        return G.host_bits(bufs[0])

    base = chain()
    wqp.set_pdl(True)
    try:
        runs = [chain() for _ in range(3)]
    finally:
        wqp.set_pdl(False)
    for r in runs:
        assert np.array_equal(r, base)
    assert np.isfinite(bf16_to_f64(base)).all() and (base != 0).any()


# ---------------------------------------------------------------- W4A16
@pytest.mark.parametrize("N,K", [(128, 256), (200, 512), (1000, 1024), (77, 2560), (384, 4096)])
def test_w4_tc_parity_small(oracle_lib, N, K):
    for M in (1, 3, 8, 16):
        d = G.make("w4", M, N, K, seed=700 + N + K + M)
        C = G.host_bits(G.run_gpu(d, tc=True))
        _check_tc(oracle_lib, d, C, f"w4 M={M} N={N} K={K}")


def test_w4_tc_global_scale(oracle_lib):
    d = G.make("w4", 5, 300, 1024, seed=31)
    d["g"] = 0.37109375
    C = G.host_bits(G.run_gpu(d, tc=True))
    _check_tc(oracle_lib, d, C, "w4 global scale")


def test_w4_tc_exact_arithmetic_bit_exact(oracle_lib):
    """Integer activations, power-of-two group scales, g = 1: every partial sum
    is exact, so any summation order gives the oracle's bits."""
    r = np.random.default_rng(9)
    M, N, K = 16, 260, 2048
    A = synth.bf16_bits_from_f32(r.integers(-4, 5, size=(M, K)).astype(np.float32))
    nib = r.integers(0, 16, size=(N, K), dtype=np.uint8)
    W = synth.pack_w4(nib)
    S = synth.e4m3_round(2.0 ** r.integers(-2, 3, size=(N, K // 16)))
    d = {"A": A, "dA": G.dev_bf16(A), "M": M, "N": N, "K": K, "fmt": "w4", "W": W, "S": S,
         "dW": G.dev_u8(W), "dS": G.dev_u8(S), "g": 1.0}
    C = G.host_bits(G.run_gpu(d, tc=True))
    assert np.array_equal(C, G.run_oracle(oracle_lib, d).c)


def test_w4_tc_rows_independent_and_k_rule():
    import weight_only_quantized_packed_gb300 as wqp

    d = G.make("w4", 16, 5120, 5120, seed=22)
    c16 = G.host_bits(G.run_gpu(d, tc=True))
    assert np.array_equal(c16, G.host_bits(G.run_gpu(d, tc=True)))   # deterministic split-K
    for m in (0, 9, 15):
        one = G.host_bits(G.run_gpu(d, tc=True, A=d["dA"][m:m + 1]))
        assert np.array_equal(one[0], c16[m])
    bad = G.make("w4", 1, 64, 384, seed=3)
    with pytest.raises(wqp.WqpError):
        G.run_gpu(bad, tc=True)          # K % 256 != 0


@pytest.mark.parametrize("N,K,Ms", [(5120, 5120, (1, 8, 16)), (17408, 5120, (4,))])
def test_w4_tc_full_size(oracle_lib, N, K, Ms):
    for M in Ms:
        d = G.make("w4", M, N, K, seed=synth.seed_for(2, M))
        C = G.host_bits(G.run_gpu(d, tc=True))
        _check_tc(oracle_lib, d, C, f"w4 full M={M} N={N} K={K}")


# ------------------------------------------------------- strided, M > 16
def _strided_canary(oracle_lib, d, tc, lda, ldc, what):
    """Runs one call with row pitches lda > K and ldc > N inside a canary
    buffer; checks the bytes outside C's rows and returns C's bits."""
    import torch

    M, N, K = d["M"], d["N"], d["K"]
    Abig = torch.zeros((M, lda), dtype=torch.bfloat16, device="cuda")
    Abig[:, :K] = d["dA"]
    canary = torch.full((M + 2, ldc), -7.0, dtype=torch.bfloat16, device="cuda")
    out = canary[1:M + 1].as_strided((M, N), (ldc, 1))
    G.run_gpu(d, tc=tc, A=Abig[:, :K], out=out)
    host = canary.float().cpu().numpy()
    assert (host[0] == -7.0).all() and (host[M + 1] == -7.0).all(), what
    assert (host[1:M + 1, N:] == -7.0).all(), what
    C = G.host_bits(canary[1:M + 1, :N].contiguous())
    _check_tc(oracle_lib, d, C, what)
    return C


@pytest.mark.parametrize("fmt,N,K", [("w8", 200, 2048), ("w8", 1000, 5120), ("w4", 200, 2048), ("w4", 77, 4096)])
def test_w8_w4_tc_strided_rows_and_canary(oracle_lib, fmt, N, K):
    """The FP8 and W4 tensor-core entries with row pitches lda = K + 64 and
    ldc = N + 13 ("w8a16_gemm_m16.rs", doc of `w8a16_gemm_m16_strided`): the
    activation tensor map's row pitch and the epilogues' ldc stores."""
    for M in (5, 16):
        d = G.make(fmt, M, N, K, seed=41 + M + N)
        C = _strided_canary(oracle_lib, d, True, K + 64, N + 13, f"{fmt} tc strided M={M} N={N} K={K}")
        base = G.host_bits(G.run_gpu(d, tc=True))
        assert np.array_equal(C, base)       # the pitches change nothing in the result


TC_ALL = pytest.mark.parametrize("fmt,eng,K", [("w8", True, 2048), ("w4", True, 2048), ("q2", True, 2048),
                                               ("q2", "mma", 2048)],
                                 ids=["w8_tcgen05", "w4_tcgen05", "q2_tcgen05", "q2_mma_sync"])


@TC_ALL
def test_tc_m_above_16(oracle_lib, fmt, eng, K):
    """M = 17 and 32 on the tensor-core entries: row blocks of one launch
    each ("w8a16_gemm_m16.rs", doc of `w8a16_gemm_m16`: more rows than the
    M tile run as further launches on contiguous row blocks). Each row equals
    the same row computed in a call of its own."""
    N = 300
    for M in (17, 32):
        d = G.make(fmt, M, N, K, seed=900 + M)
        C = G.host_bits(G.run_gpu(d, tc=eng))
        _check_tc(oracle_lib, d, C, f"{fmt} {eng} M={M}")
        for m in (0, 16, M - 1):
            one = G.host_bits(G.run_gpu(d, tc=eng, A=d["dA"][m:m + 1]))
            assert np.array_equal(one[0], C[m]), (M, m)


# ------------------------------------------ FP8 and W4 on the warp-level MMA
# w8a16_gemm_mma and w4a16_gemm_mma: FP16 operands, exact weights, activations
# scaled per (row, 128-K block) by a power of two; held to the scalar term.
F16_FMTS = pytest.mark.parametrize("fmt", ["w8", "w4"])


@F16_FMTS
@pytest.mark.parametrize("N,K", [(128, 1024), (200, 2048), (1000, 1024), (77, 3072), (384, 8192)])
def test_f16_mma_parity_small(oracle_lib, fmt, N, K):
    for M in (1, 5, 7, 8, 16):
        d = G.make(fmt, M, N, K, seed=1300 + N + K + M)
        C = G.host_bits(G.run_gpu(d, tc="mma"))
        _check_tc(oracle_lib, d, C, f"{fmt} mma M={M} N={N} K={K}")


@F16_FMTS
def test_f16_mma_exact_arithmetic_bit_exact(oracle_lib, fmt):
    """Small-integer activations and power-of-two scales: every partial sum
    is exact, so the MMA path gives the oracle's bits."""
    r = np.random.default_rng(13)
    M, N, K = 16, 260, 3072
    A = synth.bf16_bits_from_f32(r.integers(-4, 5, size=(M, K)).astype(np.float32))
    d = {"A": A, "dA": G.dev_bf16(A), "M": M, "N": N, "K": K, "fmt": fmt}
    if fmt == "w8":
        W = synth.e4m3_round(r.integers(-16, 17, size=(N, K)) / 8.0)
        S = (2.0 ** r.integers(-2, 3, size=((N + 127) // 128, K // 128))).astype(np.float32)
        d.update(W=W, S=S, dW=G.dev_u8(W), dS=G.dev_f32(S))
    else:
        nib = r.integers(0, 16, size=(N, K), dtype=np.uint8)
        W = synth.pack_w4(nib)
        S = synth.e4m3_round(2.0 ** r.integers(-2, 3, size=(N, K // 16)))
        d.update(W=W, S=S, dW=G.dev_u8(W), dS=G.dev_u8(S), g=1.0)
    C = G.host_bits(G.run_gpu(d, tc="mma"))
    assert np.array_equal(C, G.run_oracle(oracle_lib, d).c)


@F16_FMTS
def test_f16_mma_one_hot_and_order(oracle_lib, fmt):
    """One-hot activations pick single weights: each output is the dequantised
    weight (times the block scale for FP8), bit for bit, at k positions that
    cover every lane and MMA step of a block."""
    N, K = 136, 2048
    d0 = G.make(fmt, 1, N, K, seed=77)
    if fmt == "w8":
        deq = oracle_lib.w8_dequant(d0["W"], d0["S"], N, K)
    else:
        deq = oracle_lib.w4_dequant(d0["W"], d0["S"], 1.0, N, K)
    for j in (0, 1, 2, 3, 4, 17, 31, 32, 63, 100, 127, 128, 1023, 1024, 2047):
        A = np.zeros((2, K), np.float32)
        A[0, j] = 1.0
        A[1, j] = -0.5
        Ab = synth.bf16_bits_from_f32(A)
        d = dict(d0, A=Ab, dA=G.dev_bf16(Ab), M=2)
        C = G.host_bits(G.run_gpu(d, tc="mma"))
        exp = np.stack([deq[:, j], -0.5 * deq[:, j]]).astype(np.float64) + 0.0   # a zero weight gives +0
        assert np.array_equal(C, bf16_exact_bits(exp)), j


@F16_FMTS
def test_f16_mma_activation_range(oracle_lib, fmt):
    """The per-block power-of-two scaling of the activations keeps large,
    small and mixed-magnitude rows within the scalar term."""
    M, N, K = 4, 300, 2048
    for scale in (2.0 ** 40, 2.0 ** -40, 1.0):
        d = G.make(fmt, M, N, K, seed=81)
        A = synth.bf16_bits_to_f32(d["A"]).astype(np.float64) * scale
        if scale == 1.0:                          # one row spanning 2^-30 .. 2^30 within a block
            A[1] *= 2.0 ** np.linspace(-30, 30, K)
        Ab = synth.bf16_bits_from_f32(A.astype(np.float32))
        d = dict(d, A=Ab, dA=G.dev_bf16(Ab))
        C = G.host_bits(G.run_gpu(d, tc="mma"))
        _check_tc(oracle_lib, d, C, f"{fmt} mma activation scale {scale:g}")


def test_w4_mma_global_scale(oracle_lib):
    d = G.make("w4", 5, 300, 1024, seed=31)
    d["g"] = 0.37109375
    C = G.host_bits(G.run_gpu(d, tc="mma"))
    _check_tc(oracle_lib, d, C, "w4 mma global scale")


@F16_FMTS
@pytest.mark.parametrize("N", [5120, 17408])
def test_f16_mma_rows_independent_and_k_rule(fmt, N):
    import weight_only_quantized_packed_gb300 as wqp

    d = G.make(fmt, 16, N, 5120, seed=23)
    c16 = G.host_bits(G.run_gpu(d, tc="mma"))
    assert np.array_equal(c16, G.host_bits(G.run_gpu(d, tc="mma")))   # deterministic
    for m in (0, 8, 15):
        one = G.host_bits(G.run_gpu(d, tc="mma", A=d["dA"][m:m + 1]))
        assert np.array_equal(one[0], c16[m])
    bad = G.make(fmt, 1, 64, 640 if fmt == "w8" else 768, seed=3)
    with pytest.raises(wqp.WqpError):
        G.run_gpu(bad, tc="mma")                 # K % 1024 != 0


@pytest.mark.parametrize("fmt,N,K,Ms", [("w8", 17408, 5120, (1, 8, 16)), ("w8", 5120, 17408, (2, 16)),
                                        ("w8", 17000, 5120, (16,)), ("w4", 5120, 5120, (1, 8, 16)),
                                        ("w4", 17408, 5120, (4, 16)), ("w4", 20000, 5120, (3, 16))])
def test_f16_mma_full_size(oracle_lib, fmt, N, K, Ms):
    for M in Ms:
        d = G.make(fmt, M, N, K, seed=synth.seed_for(3 if fmt == "w8" else 2, M))
        C = G.host_bits(G.run_gpu(d, tc="mma"))
        _check_tc(oracle_lib, d, C, f"{fmt} mma full M={M} N={N} K={K}")


@pytest.mark.parametrize("fmt,N,K", [("w8", 200, 2048), ("w8", 1000, 5120), ("w4", 200, 2048), ("w4", 77, 4096)])
def test_f16_mma_strided_rows_and_canary(oracle_lib, fmt, N, K):
    for M in (5, 16):
        d = G.make(fmt, M, N, K, seed=51 + M + N)
        C = _strided_canary(oracle_lib, d, "mma", K + 64, N + 13, f"{fmt} mma strided M={M} N={N} K={K}")
        assert np.array_equal(C, G.host_bits(G.run_gpu(d, tc="mma")))


@F16_FMTS
def test_f16_mma_m_above_16(oracle_lib, fmt):
    N, K = 300, 2048
    for M in (17, 32):
        d = G.make(fmt, M, N, K, seed=950 + M)
        C = G.host_bits(G.run_gpu(d, tc="mma"))
        _check_tc(oracle_lib, d, C, f"{fmt} mma M={M}")
        for m in (0, 16, M - 1):
            one = G.host_bits(G.run_gpu(d, tc="mma", A=d["dA"][m:m + 1]))
            assert np.array_equal(one[0], C[m]), (M, m)


# -------------------------------------------------------------------- long K
# The persistent kernels keep each rank's B-fragment sets in shared memory
# beside a ring of two stages; at 8 K splits those fit up to K = 57344 for
# Q2_0 and FP8 and K = 43008 for W4. Past that, Q2_0 runs on the short-CTA
# kernel and FP8 / W4 rebuild each item's fragments. The weights are a seeded
# block of R rows repeated down N, and the oracle runs on the block.
def _tiled(fmt, M, N, K, R, seed):
    base = G.make(fmt, M, R, K, seed=seed)
    reps = -(-N // R)
    W = np.tile(base["W"], (reps, 1))[:N]
    d = dict(base, N=N, W=W, dW=G.dev_u8(W))
    if fmt == "w4":
        S = np.tile(base["S"], (reps, 1))[:N]
        d.update(S=S, dS=G.dev_u8(S))
    elif fmt == "w8":
        assert R % 128 == 0                      # whole 128-row scale groups
        S = np.tile(base["S"], (reps, 1))[:-(-N // 128)]
        d.update(S=S, dS=G.dev_f32(S))
    return base, d


def _tiled_ref(ref, N):
    reps = -(-N // ref.c.shape[1])
    return type(ref)(np.tile(ref.c, (1, reps))[:, :N], np.tile(ref.r, (1, reps))[:, :N],
                     np.tile(ref.s, (1, reps))[:, :N])


@pytest.mark.parametrize("fmt", ["q2", "w8", "w4"])
def test_mma_long_k(oracle_lib, fmt):
    """K = 65536 on the warp-level MMA engines, past the fragment-set limit.
    Q2_0 at N = 128 x SMs + 37, a shape the persistent kernel takes at a
    shorter K; FP8 and W4 at a ragged N = 4133. 16 rows against the oracle
    on every output, and the first 3 rows equal to a 3-row call's."""
    import torch

    K, R = 65536, 256
    N = 128 * torch.cuda.get_device_properties(0).multi_processor_count + 37 if fmt == "q2" else 4133
    base, d = _tiled(fmt, 16, N, K, R, seed=970)
    ref = _tiled_ref(G.run_oracle(oracle_lib, base), N)
    C16 = G.host_bits(G.run_gpu(d, tc="mma"))
    assert_scalar_term(C16, ref, K, f"{fmt} mma long K M=16 N={N} K={K}")
    C3 = G.host_bits(G.run_gpu(d, tc="mma", A=d["dA"][:3]))
    assert np.array_equal(C3, C16[:3])


@pytest.mark.parametrize("fmt", ["q2", "w8", "w4"])
def test_largest_k_every_engine(oracle_lib, fmt):
    """K = 2^20, the largest K the C ABI accepts, on the scalar, tcgen05 and
    warp-level MMA engines of each format (N = 40, M = 3): the scalar term
    (the FP8 tensor-core term on tcgen05) against the oracle."""
    K, N, M = 1 << 20, 40, 3
    d = G.make(fmt, M, N, K, seed=980)
    ref = G.run_oracle(oracle_lib, d)
    C = G.host_bits(G.run_gpu(d))
    assert_scalar_term(C, ref, K, f"{fmt} scalar K={K}")
    for eng in (True, "mma"):
        C = G.host_bits(G.run_gpu(d, tc=eng))
        _check_tc(oracle_lib, d, C, f"{fmt} {eng} K={K}")


# ------------------------------------------------- fewer rows than one tile
@pytest.mark.parametrize("fmt,eng,K", [("q2", True, 1024), ("q2", "mma", 1024), ("w4", True, 256), ("w4", "mma", 1024),
                                       ("w8", True, 1024), ("w8", "mma", 1024)])
def test_tc_fewer_rows_than_a_tile(oracle_lib, fmt, eng, K):
    """N = 1, 15 and 17 (less than one 16-row MMA tile, and just over) at
    the smallest K each engine accepts, M = 1 and 16: the rows past N of the
    engine's tile are never stored, and every stored output meets its term."""
    for N in (1, 15, 17):
        for M in (1, 16):
            d = G.make(fmt, M, N, K, seed=990 + N + M)
            C = G.host_bits(G.run_gpu(d, tc=eng))
            assert C.shape == (M, N)
            _check_tc(oracle_lib, d, C, f"{fmt} {eng} N={N} M={M} K={K}")
