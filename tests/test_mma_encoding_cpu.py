"""The arithmetic of the warp-level Q2_0 kernel (q2_gemm_mma), emulated on the
CPU for one 16-row x 128-K block and one 8-row activation tile, and checked
exactly against the Q2_0 formula of "spark_model/layers/ops/gemv_q2_vec.rs"
(module docs; test helper `gemv_row`): sum_k (c - 1) * a * d.

The emulation follows the kernel's data flow lane by lane:
  * lane (g, t) takes code words 2t and 2t + 1 of rows g and g + 8 and masks
    them in place: (w & 0x00030003 << 2x) and ((w >> 8) & ...);
  * it pairs its 32 activations (k = 32 t .. 32 t + 31 of row g) with byte
    permutes and multiplies them by 2^(64 - 2x);
  * the chain starts from the block's offset -2^-69 * sum_k a: four MMAs with
    the lane's raw activations as the A operand (rows g and g + 8 each hold
    half of activation row g) against -2^-69 in every B element, the two
    halves added, and the sums of activation rows 2t and 2t + 1 taken from
    lanes 8t and 8t + 4 (the shuffle) as the chain's C input;
and places every register into the m16n8k16 matrices by the fragment layout
the PTX ISA gives for .bf16 operands. The products are exact, so the float64
sums must equal the formula bit for bit: a wrong lane assignment, permute
selector, mask, pre-scale or fragment position fails. No GPU is needed.
"""
from __future__ import annotations

import numpy as np
import pytest

from weight_only_quantized_packed_gb300 import synth


def bf16_bits_to_f64(bits):
    """BF16 bit patterns (subnormals included) to float64."""
    b = np.asarray(bits, dtype=np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def byte_perm(x, y, sel):
    """The 32-bit byte permute of CUDA's __byte_perm for selectors 0x5410 and
    0x7632 (no sign replication)."""
    src = [(x >> (8 * i)) & 0xFF for i in range(4)] + [(y >> (8 * i)) & 0xFF for i in range(4)]
    out = 0
    for i in range(4):
        out |= src[(sel >> (4 * i)) & 7] << (8 * i)
    return out


def mul_pow2_bf16x2(v, e):
    """Both BF16 halves of v times 2^e (exact for the values used here)."""
    out = 0
    for h in range(2):
        bits = (v >> (16 * h)) & 0xFFFF
        x = float(bf16_bits_to_f64([bits])[0]) * 2.0 ** e
        nb = int(np.array([x], dtype=np.float32).view(np.uint32)[0]) >> 16
        assert bf16_bits_to_f64([nb])[0] == x
        out |= nb << (16 * h)
    return out


def mma_fragments_to_matrices(a_regs, b_regs):
    """m16n8k16 .bf16: per lane, A registers {a0..a3} and B registers {b0, b1}
    to the 16x16 A and 16x8 B matrices (PTX ISA fragment layout: group
    g = lane / 4, thread-in-group t = lane % 4)."""
    A = np.zeros((16, 16))
    B = np.zeros((16, 8))
    for lane in range(32):
        g, t = lane // 4, lane % 4
        for j, (row, col) in enumerate([(g, 2 * t), (g + 8, 2 * t), (g, 2 * t + 8), (g + 8, 2 * t + 8)]):
            lo, hi = bf16_bits_to_f64([a_regs[lane][j] & 0xFFFF, a_regs[lane][j] >> 16])
            A[row, col], A[row, col + 1] = lo, hi
        for j, krow in enumerate([2 * t, 2 * t + 8]):
            lo, hi = bf16_bits_to_f64([b_regs[lane][j] & 0xFFFF, b_regs[lane][j] >> 16])
            B[krow, g], B[krow + 1, g] = lo, hi
    return A, B


NEG_UNIT = 0x9D009D00      # -2^-69 in both BF16 halves


def emulate_block(codes, act_bits, scale_exp=lambda x: 64 - 2 * x, swap_a_halves=False, offset=True,
                  offset_src=lambda t: (8 * t, 8 * t + 4)):
    """One warp, one block, one row tile: D[row, m] = 2^-69 sum_k (c - 1) a.
    The keyword arguments plant mistakes for the tests that must catch them."""
    # Code words: word i of row r holds codes 16 i .. 16 i + 15, code q at bits 2q.
    words = np.zeros((16, 8), dtype=np.uint64)
    for q in range(16):
        words |= codes[:, q::16].astype(np.uint64) << np.uint64(2 * q)
    words = words.astype(np.uint32)
    D = np.zeros((16, 8))
    # B fragments (built once per block).
    bregs = []
    for st in range(8):
        x, o = st & 3, 8 * (st >> 2) + ((st & 3) >> 1)
        sel = 0x7632 if x & 1 else 0x5410
        per_lane = []
        for lane in range(32):
            g, t = lane // 4, lane % 4
            r = [int(act_bits[g, 32 * t + 2 * i]) | (int(act_bits[g, 32 * t + 2 * i + 1]) << 16) for i in range(16)]
            b0 = mul_pow2_bf16x2(byte_perm(r[o], r[o + 4], sel), scale_exp(x))
            b1 = mul_pow2_bf16x2(byte_perm(r[o + 2], r[o + 6], sel), scale_exp(x))
            per_lane.append((b0, b1))
        bregs.append(per_lane)
    if offset:
        # Four MMAs: lane (g, t) passes its raw activation registers 4j .. 4j + 3.
        O = np.zeros((16, 8))
        for j in range(4):
            a_regs = []
            for lane in range(32):
                g, t = lane // 4, lane % 4
                r = [int(act_bits[g, 32 * t + 2 * i]) | (int(act_bits[g, 32 * t + 2 * i + 1]) << 16) for i in range(16)]
                a_regs.append(r[4 * j:4 * j + 4])
            A, B = mma_fragments_to_matrices(a_regs, [[NEG_UNIT, NEG_UNIT]] * 32)
            O += A @ B
        # Lane (g, t) holds D[g, 2t] and D[g + 8, 2t]; their sum is its s.
        s = [O[lane // 4, 2 * (lane % 4)] + O[lane // 4 + 8, 2 * (lane % 4)] for lane in range(32)]
        # The chain's C input of lane (g, t): columns 2t and 2t + 1 of rows g and g + 8.
        for lane in range(32):
            g, t = lane // 4, lane % 4
            src0, src1 = offset_src(t)
            for row in (g, g + 8):
                D[row, 2 * t] += s[src0]
                D[row, 2 * t + 1] += s[src1]
    # The codes' chain.
    for st in range(8):
        m = 0x00030003 << (2 * (st & 3))
        w = st >> 2
        a_regs = []
        for lane in range(32):
            g, t = lane // 4, lane % 4
            wg, wh = int(words[g, 2 * t + w]), int(words[g + 8, 2 * t + w])
            regs = [wg & m, wh & m, (wg >> 8) & m, (wh >> 8) & m]
            a_regs.append([regs[2], regs[3], regs[0], regs[1]] if swap_a_halves else regs)
        A, B = mma_fragments_to_matrices(a_regs, bregs[st])
        D += A @ B
    return D


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_mma_encoding_is_exact(seed):
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 4, size=(16, 128), dtype=np.uint8)     # code 3 included (+2)
    act = synth.activations(8, 128, seed)                          # BF16 bits, N(0,1)
    D = emulate_block(codes, act)
    a = bf16_bits_to_f64(act)
    want = (codes.astype(np.float64) - 1.0) @ a.T                  # [16 rows, 8 activation rows]
    assert np.array_equal(D * 2.0 ** 69, want)


def test_mma_encoding_large_and_small_activations():
    """The pre-scale stays exact across the documented activation range."""
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 3, size=(16, 128), dtype=np.uint8)
    for scale in (2.0 ** 40, 2.0 ** -40):
        act = synth.activations(8, 128, 9, scale=scale)
        D = emulate_block(codes, act)
        want = (codes.astype(np.float64) - 1.0) @ bf16_bits_to_f64(act).T
        assert np.array_equal(D * 2.0 ** 69, want)


def test_a_wrong_permute_is_caught():
    """Swapping the permute selectors (a plausible slip) breaks the identity."""
    global byte_perm
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 3, size=(16, 128), dtype=np.uint8)
    act = synth.activations(8, 128, 12)
    good = byte_perm
    try:
        byte_perm = lambda x, y, sel: good(x, y, 0x5410 if sel == 0x7632 else 0x7632)  # noqa: E731
        D = emulate_block(codes, act)
    finally:
        byte_perm = good
    want = (codes.astype(np.float64) - 1.0) @ bf16_bits_to_f64(act).T
    assert not np.array_equal(D * 2.0 ** 69, want)


@pytest.mark.parametrize("mistake", [
    dict(scale_exp=lambda x: 64 - x),        # pre-scale exponent per position off
    dict(swap_a_halves=True),                # codes (x, 8+x) and (4+x, 12+x) swapped
    dict(offset=False),                      # the "- 1" (the offset) dropped
    dict(offset_src=lambda t: (4 * t, 4 * t + 1)),   # offsets fetched from the wrong lanes
])
def test_planted_mistakes_are_caught(mistake):
    rng = np.random.default_rng(13)
    codes = rng.integers(0, 3, size=(16, 128), dtype=np.uint8)
    act = synth.activations(8, 128, 14)
    D = emulate_block(codes, act, **mistake)
    want = (codes.astype(np.float64) - 1.0) @ bf16_bits_to_f64(act).T
    assert not np.array_equal(D * 2.0 ** 69, want)
