"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test fixes part of the oracle against a format definition, a library
routine, a closed form, an exact-arithmetic sum, or an invariant that the
source pages state. The tests are chosen so that a plausible slip fails one
of them: a wrong code bit position or nibble order, a dropped -1 offset, a
wrong group or block index, a transposed operand, or a scale folded in the
wrong place.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from tests._tol import bf16_bits, bf16_exact_bits, bf16_to_f64, scalar_ok
from weight_only_quantized_packed_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------- decoders
def test_e4m3_decoder_matches_torch_all_codes(oracle_lib):
    """Every E4M3 encoding decodes as torch.float8_e4m3fn does (library)."""
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle_lib.e4m3_to_f32(i) for i in range(256)], np.float32)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin].view(np.uint32), got[fin].view(np.uint32))


def test_e4m3_decoder_spec_points(oracle_lib):
    """OCP FP8 E4M3 fixed points: max normal, min normal, min/max subnormal, 1."""
    pts = {0x7E: 448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 0.875 * 2.0 ** -6,
           0x38: 1.0, 0xB8: -1.0, 0x00: 0.0, 0x3F: 1.875, 0x40: 2.0}
    for code, v in pts.items():
        assert oracle_lib.e4m3_to_f32(code) == v, hex(code)
    assert math.isnan(oracle_lib.e4m3_to_f32(0x7F))
    assert math.isnan(oracle_lib.e4m3_to_f32(0xFF))


def test_e2m1_decoder_table(oracle_lib):
    """OCP MX E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}; bit 3 is the sign."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for i in range(16):
        v = oracle_lib.e2m1_to_f32(i)
        assert abs(v) == mags[i & 7]
        assert math.copysign(1.0, v) == (-1.0 if i & 8 else 1.0)
    ml = pytest.importorskip("ml_dtypes")
    lib = np.arange(16, dtype=np.uint8).view(ml.float4_e2m1fn).astype(np.float32)
    got = np.array([oracle_lib.e2m1_to_f32(i) for i in range(16)], np.float32)
    assert np.array_equal(lib.view(np.uint32), got.view(np.uint32))


def test_f16_decoder_matches_numpy_all_codes(oracle_lib):
    h = np.arange(65536, dtype=np.uint16)
    ref = h.view(np.float16).astype(np.float32)
    got = np.array([oracle_lib.f16_to_f32(int(x)) for x in h], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan].view(np.uint32), got[~nan].view(np.uint32))


def test_bf16_round_matches_torch(oracle_lib):
    r = np.random.default_rng(1)
    x = np.concatenate([
        r.standard_normal(2000).astype(np.float32),
        # exact ties: low 16 bits 0x8000, both parities of bit 16
        (np.arange(64, dtype=np.uint32) * 0x10000 + 0x3F808000).view(np.float32),
        np.array([0.0, -0.0, 3.0e38, -3.0e38, 1e-40], np.float32),
    ])
    got = np.array([oracle_lib.f32_to_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, bf16_bits(x))


# ----------------------------------------------------------------- Q2_0
def _onehot_rows(M, K, cols):
    A = np.zeros((M, K), np.float32)
    for m, j in enumerate(cols):
        A[m, j] = 1.0
    return synth.bf16_bits_from_f32(A)


def test_q2_closed_form_all_ones_all_twos(oracle_lib):
    """All-ones A with every code 2 and one uniform d gives K*d. Partial sums
    k*d need at most 11 + 13 bits, so the f32 sum is exact for K <= 8192."""
    N = 3
    for K in (128, 512, 5120, 8192):
        d = np.float16(0.0371)
        W = synth.pack_q2(np.full((N, K), 2, np.uint8), np.full((N, K // 128), d, np.float16))
        A = synth.bf16_bits_from_f32(np.ones((1, K), np.float32))
        r = oracle_lib.q2_gemv(A, W, 1, N, K)
        expect = bf16_exact_bits(np.full((1, N), K * float(d)))
        assert np.array_equal(r.c, expect), K
        assert np.allclose(r.r, K * float(d), rtol=0, atol=0)


def test_q2_one_hot_pins_code_order_and_group(oracle_lib):
    """A = e_j returns column j of the dequantised weights. Expected values come
    from the unpacked codes and scales, not from the oracle's own unpacking.
    This pins the bit position, the byte index, the -1 offset, the group
    index and the byte order of d."""
    N, K = 9, 384
    r = np.random.default_rng(7)
    codes = r.integers(0, 3, size=(N, K), dtype=np.uint8)
    d = r.uniform(0.01, 0.05, size=(N, K // 128)).astype(np.float16)
    W = synth.pack_q2(codes, d)
    cols = [0, 1, 2, 3, 4, 5, 126, 127, 128, 131, 200, 255, 256, 383, 302, 77]
    A = _onehot_rows(len(cols), K, cols)
    res = oracle_lib.q2_gemv(A, W, len(cols), N, K)
    for m, j in enumerate(cols):
        w = (codes[:, j].astype(np.float64) - 1.0) * d[:, j // 128].astype(np.float64)
        assert np.array_equal(res.c[m], bf16_exact_bits(w)), j


def test_q2_code3_literal_reading(oracle_lib):
    """Code 3 is never generated; the literal formula ((c & 3) - 1) * d gives +2d."""
    N, K = 2, 128
    codes = np.full((N, K), 3, np.uint8)
    d = np.full((N, 1), 0.25, np.float16)
    A = _onehot_rows(1, K, [5])
    res = oracle_lib.q2_gemv(A, synth.pack_q2(codes, d), 1, N, K)
    assert np.array_equal(res.c[0], bf16_exact_bits([0.5, 0.5]))


def test_q2_exact_arithmetic_random(oracle_lib):
    """Small-integer A and power-of-two d make every partial sum exact in f32,
    so the oracle must equal bf16 of the exact sum (computed in fp64 from the
    unpacked values, which is exact here)."""
    r = np.random.default_rng(11)
    for (M, N, K) in [(1, 5, 256), (4, 13, 1024), (3, 8, 640)]:
        codes = r.integers(0, 3, size=(N, K), dtype=np.uint8)
        d = (2.0 ** -r.integers(2, 7, size=(N, K // 128))).astype(np.float16)
        a = r.integers(-8, 9, size=(M, K)).astype(np.float32)
        res = oracle_lib.q2_gemv(synth.bf16_bits_from_f32(a), synth.pack_q2(codes, d), M, N, K)
        w = (codes.astype(np.float64) - 1.0) * np.repeat(d.astype(np.float64), 128, axis=1)
        exact = a.astype(np.float64) @ w.T
        assert np.array_equal(res.c, bf16_exact_bits(exact))
        assert np.array_equal(res.r, exact)


def test_q2_transpose_pin(oracle_lib):
    """Rows of A map to rows of C, weight rows to columns of C (N != K != M)."""
    N, K = 7, 256
    codes = np.zeros((N, K), np.uint8) + 1
    codes[3, 100] = 2       # only weight (n=3, k=100) is non-zero
    d = np.full((N, 2), 1.0, np.float16)
    A = _onehot_rows(3, K, [0, 100, 255])
    res = oracle_lib.q2_gemv(A, synth.pack_q2(codes, d), 3, N, K)
    expect = np.zeros((3, N))
    expect[1, 3] = 1.0
    assert np.array_equal(res.c, bf16_exact_bits(expect))


def test_q2_sign_flip_and_linearity(oracle_lib):
    """c -> 2 - c negates every output exactly; A * 2^p scales it by 2^p."""
    M, N, K = 3, 11, 512
    W, codes, d = synth.q2_weights(N, K, seed=5)
    A = synth.activations(M, K, seed=6)
    base = oracle_lib.q2_gemv(A, W, M, N, K)
    flip = oracle_lib.q2_gemv(A, synth.pack_q2(2 - codes, d), M, N, K)
    assert np.array_equal(bf16_to_f64(flip.c), -bf16_to_f64(base.c))
    A4 = synth.bf16_bits_from_f32(synth.bf16_bits_to_f32(A) * 4.0)
    scaled = oracle_lib.q2_gemv(A4, W, M, N, K)
    assert np.array_equal(bf16_to_f64(scaled.c), 4.0 * bf16_to_f64(base.c))


def test_q2_brute_force_tiny_within_one_ulp_of_exact(oracle_lib):
    """Against bf16 of the fp64 sum: the f32 sequential sum is within 1 ULP
    (or the reordering floor)."""
    for K in (128, 256):
        for N in (1, 5, 8, 9):
            W, codes, d = synth.q2_weights(N, K, seed=100 + K + N)
            M = 2
            A = synth.activations(M, K, seed=200 + K + N)
            res = oracle_lib.q2_gemv(A, W, M, N, K)
            w = (codes.astype(np.float64) - 1.0) * np.repeat(d.astype(np.float64), 128, axis=1)
            exact = synth.bf16_bits_to_f32(A).astype(np.float64) @ w.T
            assert np.allclose(res.r, exact, rtol=1e-12, atol=1e-12)
            ok, _ = scalar_ok(res.c, type(res)(bf16_bits(exact), exact, res.s), K)
            assert ok.all()


def _pages_gen_inputs(m, n, k):
    """The deterministic generator of the Q2_0 unit tests ("gemv_q2_vec.rs",
    test helper `gen_inputs`), restated: a = sin(0.09131 i) * 1.3, code =
    ((i * 2654435761) >> 6) % 3, scale = 0.015 + 0.01 * (i % 5)."""
    i = np.arange(m * k, dtype=np.float32)
    act = (np.sin(i * np.float32(0.09131)) * np.float32(1.3)).astype(np.float32).reshape(m, k)
    ci = np.arange(n * k, dtype=np.uint64)
    codes = (((ci * np.uint64(2654435761)) >> np.uint64(6)) % np.uint64(3)).astype(np.uint8).reshape(n, k)
    si = np.arange(n * (k // 128))
    scales = (np.float32(0.015) + np.float32(0.01) * (si % 5).astype(np.float32)).reshape(n, k // 128)
    return act, codes, scales


def test_q2_pages_fixed_vector_batched_equals_rows(oracle_lib):
    """The pages' fixed vector (n=5, k=256, m up to 16): a batched oracle call
    equals one M=1 call per row, bit for bit ("gemv_q2_vec.rs", test
    `chunked_batchm_equals_per_row_gemv`). The result is also within
    tolerance of the fp64 sum."""
    n, k = 5, 256
    for m in (1, 2, 3, 8, 9, 16):
        act, codes, scales = _pages_gen_inputs(m, n, k)
        A = synth.bf16_bits_from_f32(act)
        W = synth.pack_q2(codes, scales.astype(np.float16))
        full = oracle_lib.q2_gemv(A, W, m, n, k)
        for row in range(m):
            one = oracle_lib.q2_gemv(A[row:row + 1], W, 1, n, k)
            assert np.array_equal(one.c[0], full.c[row])
        w = (codes.astype(np.float64) - 1) * np.repeat(scales.astype(np.float16).astype(np.float64), 128, axis=1)
        exact = synth.bf16_bits_to_f32(A).astype(np.float64) @ w.T
        ok, _ = scalar_ok(full.c, type(full)(bf16_bits(exact), exact, full.s), k)
        assert ok.all()


def test_q2_dequant_matches_unpacked(oracle_lib):
    N, K = 6, 384
    W, codes, d = synth.q2_weights(N, K, seed=3)
    got = oracle_lib.q2_dequant(W, N, K)
    exp = (codes.astype(np.float64) - 1) * np.repeat(d.astype(np.float64), 128, axis=1)
    assert np.array_equal(got.astype(np.float64), exp)


# ----------------------------------------------------------------- W4
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                 -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def _e4m3_value(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_w4_one_hot_pins_nibble_order_and_group(oracle_lib):
    N, K = 16, 256
    r = np.random.default_rng(3)
    nib = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    nib = (nib + np.arange(N, dtype=np.uint8)[:, None]) & 15     # row n shifted by n
    scales = synth.e4m3_round(r.uniform(0.01, 3.0, size=(N, K // 16)))
    codes = synth.pack_w4(nib)
    cols = [0, 1, 2, 15, 16, 17, 31, 32, 100, 101, 254, 255]
    A = _onehot_rows(len(cols), K, cols)
    res = oracle_lib.w4_gemv(A, codes, scales, 1.0, len(cols), N, K)
    for m, j in enumerate(cols):
        w = E2M1[nib[:, j]] * _e4m3_value(scales[:, j // 16])
        # a sum that starts at +0 turns a -0 weight into +0: compare values
        assert np.array_equal(bf16_to_f64(res.c[m]), bf16_to_f64(bf16_exact_bits(w))), j


def test_w4_exact_arithmetic_random(oracle_lib):
    r = np.random.default_rng(21)
    pow2 = synth.e4m3_round(2.0 ** np.arange(-3, 3))
    for (M, N, K) in [(1, 7, 256), (5, 16, 512), (8, 9, 128)]:
        nib = r.integers(0, 16, size=(N, K), dtype=np.uint8)
        scales = pow2[r.integers(0, len(pow2), size=(N, K // 16))]
        a = r.integers(-8, 9, size=(M, K)).astype(np.float32)
        for g in (1.0, 0.5, 4.0):
            res = oracle_lib.w4_gemv(synth.bf16_bits_from_f32(a), synth.pack_w4(nib), scales, g, M, N, K)
            w = E2M1[nib] * np.repeat(_e4m3_value(scales), 16, axis=1) * g
            exact = a.astype(np.float64) @ w.T
            assert np.array_equal(res.c, bf16_exact_bits(exact)), (M, N, K, g)


def test_w4_sign_flip(oracle_lib):
    M, N, K = 2, 9, 256
    codes, scales, nib = synth.w4_weights(N, K, seed=9)
    A = synth.activations(M, K, seed=10)
    base = oracle_lib.w4_gemv(A, codes, scales, 1.0, M, N, K)
    flip = oracle_lib.w4_gemv(A, synth.pack_w4(nib ^ 8), scales, 1.0, M, N, K)
    assert np.array_equal(bf16_to_f64(flip.c), -bf16_to_f64(base.c))


def test_w4_dequant_and_brute_force(oracle_lib):
    N, K = 9, 256
    codes, scales, nib = synth.w4_weights(N, K, seed=12)
    deq = oracle_lib.w4_dequant(codes, scales, 1.0, N, K)
    exp = E2M1[nib] * np.repeat(_e4m3_value(scales), 16, axis=1)
    assert np.array_equal(deq.astype(np.float64), exp)
    A = synth.activations(3, K, seed=13)
    res = oracle_lib.w4_gemv(A, codes, scales, 1.0, 3, N, K)
    exact = synth.bf16_bits_to_f32(A).astype(np.float64) @ exp.T
    assert np.allclose(res.r, exact, rtol=1e-12, atol=1e-12)
    ok, _ = scalar_ok(res.c, type(res)(bf16_bits(exact), exact, res.s), K)
    assert ok.all()


# ----------------------------------------------------------------- W8
def test_w8_one_hot_pins_block_scale_index(oracle_lib):
    """A = e_j gives bf16(e4m3(w[n, j]) * s[n/128, j/128]), with N = 300 so
    that a partial third scale row exists."""
    N, K = 300, 384
    w, bs = synth.w8_weights(N, K, seed=4)
    cols = [0, 127, 128, 255, 256, 383]
    A = _onehot_rows(len(cols), K, cols)
    res = oracle_lib.w8_gemm(A, w, bs, len(cols), N, K)
    q = _e4m3_value(w).astype(np.float32)
    for m, j in enumerate(cols):
        v = q[:, j] * bs[np.arange(N) // 128, j // 128]          # one f32 multiply
        assert np.array_equal(res.c[m], bf16_bits(v)), j


def test_w8_exact_arithmetic_random(oracle_lib):
    """Weights are multiples of 2^-3 with |w| <= 2 (all E4M3-exact), block
    scales are powers of two and A holds small integers. Every partial sum is then exact, so the
    result is bf16 of the exact sum."""
    r = np.random.default_rng(31)
    for (M, N, K) in [(1, 130, 256), (16, 64, 384), (5, 257, 128)]:
        wv = r.integers(-16, 17, size=(N, K)) / 8.0
        w = synth.e4m3_round(wv)
        assert np.array_equal(_e4m3_value(w), wv)
        nb = (N + 127) // 128
        bs = (2.0 ** r.integers(-2, 3, size=(nb, K // 128))).astype(np.float32)
        a = r.integers(-4, 5, size=(M, K)).astype(np.float32)
        res = oracle_lib.w8_gemm(synth.bf16_bits_from_f32(a), w, bs, M, N, K)
        full = wv * np.repeat(np.repeat(bs.astype(np.float64), 128, axis=0)[:N], 128, axis=1)
        exact = a.astype(np.float64) @ full.T
        assert np.array_equal(res.c, bf16_exact_bits(exact)), (M, N, K)


def test_w8_block_scale_folded_once_per_block(oracle_lib):
    """With a scale that is not a power of two, folding once per block,
    bf16(f32(I * s)) with I the exact inner sum, differs from scaling each
    element. The oracle must give the per-block value ("w8a16_gemm_m16.rs",
    module docs)."""
    K, N = 128, 1
    w = synth.e4m3_round(np.full((N, K), 1.0))
    a = np.zeros((1, K), np.float32)
    a[0, :7] = 1.0                                  # I = 7
    s = np.float32(0.1)
    bs = np.full((1, 1), s, np.float32)
    res = oracle_lib.w8_gemm(synth.bf16_bits_from_f32(a), w, bs, 1, N, K)
    per_block = np.float32(7.0) * s
    per_elem = np.float32(0.0)
    for _ in range(7):
        per_elem = np.float32(per_elem + np.float32(np.float32(1.0) * s))
    assert per_block != per_elem                    # the test discriminates
    assert res.c[0, 0] == bf16_bits(per_block)[()]
    # Two blocks with different scales: f32(f32(I1*s1) + f32(I2*s2)).
    K = 256
    w = synth.e4m3_round(np.full((N, K), 1.0))
    a = np.zeros((1, K), np.float32)
    a[0, :7] = 1.0
    a[0, 128:131] = 1.0                             # I2 = 3
    bs = np.array([[0.1, 0.3]], np.float32)
    res = oracle_lib.w8_gemm(synth.bf16_bits_from_f32(a), w, bs, 1, N, K)
    exp = np.float32(np.float32(7.0) * bs[0, 0]) + np.float32(np.float32(3.0) * bs[0, 1])
    assert res.c[0, 0] == bf16_bits(np.float32(exp))[()]


def test_w8_sign_flip_and_dequant(oracle_lib):
    M, N, K = 2, 200, 256
    w, bs = synth.w8_weights(N, K, seed=8)
    A = synth.activations(M, K, seed=9)
    base = oracle_lib.w8_gemm(A, w, bs, M, N, K)
    flip = oracle_lib.w8_gemm(A, w ^ np.uint8(0x80), bs, M, N, K)
    assert np.array_equal(bf16_to_f64(flip.c), -bf16_to_f64(base.c))
    deq = oracle_lib.w8_dequant(w, bs, N, K)
    exp = (_e4m3_value(w).astype(np.float32) *
           np.repeat(np.repeat(bs, 128, axis=0)[:N], 128, axis=1))
    assert np.array_equal(deq, exp)
    full = _e4m3_value(w) * np.repeat(np.repeat(bs.astype(np.float64), 128, axis=0)[:N], 128, axis=1)
    exact = synth.bf16_bits_to_f32(A).astype(np.float64) @ full.T
    assert np.allclose(base.r, exact, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- sizes
def test_weight_bytes_match_pages_table():
    """The pages' W4 table counts packed codes plus E4M3 group scales:
    14,745,600 B at N=K=5120, and 14.7456 MB / 70.5 us = 209.2 GB/s."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "w4a16_tier_table.json")))
    b = synth.w4_weight_bytes(g["n"], g["k"])
    assert b == 14_745_600
    for row in g["rows"]:
        # times are printed to 0.1 us: the GB/s column must fall inside the
        # range that rounding allows (plus its own 0.05 print rounding)
        lo = b / ((row["us"] + 0.05) * 1e-6) / 1e9
        hi = b / ((row["us"] - 0.05) * 1e-6) / 1e9
        assert lo - 0.05 <= row["gbs"] <= hi + 0.05
        assert abs(row["gbs"] / g["peak_gbs"] * 100 - row["pct"]) < 0.06
    assert synth.q2_weight_bytes(5120, 5120) == 6_963_200
    assert synth.w8_weight_bytes(17408, 5120) == 89_128_960 + 21_760
