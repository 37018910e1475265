"""Seeded synthetic inputs for the packed weight-only-quantized GEMV/GEMM.

This module only draws random numbers and lays them out in the packed byte
formats. It holds none of the GEMV arithmetic (no dequantisation, no dot
products): both the CUDA path's tests/bench and the CPU oracle take their
inputs from here, and nothing here is derived from either of them.

Formats (all little-endian, row-major per output row n):

* ``A`` / ``C``: BF16 bit patterns, ``uint16[M, K]`` / ``uint16[M, N]``.
* Q2_0 ternary ("gemv_q2_vec.rs", module docs and the ``block_q2_0`` weight
  handle): per (row n, 128-wide K group) one 34-byte block: bytes 0..31 hold
  the 128 two-bit codes, code ``i`` in bits ``2*(i%4)`` of byte ``i//4``;
  bytes 32..33 hold the fp16 scale ``d``. Blocks are stored ``[N][K/128]``
  with no padding, so a row is ``34*K/128`` bytes.
* W4 (NVFP4-style, "w4a16_gemv_tiers.rs"): E2M1 codes ``uint8[N, K/2]``,
  element ``2j`` in the low nibble and ``2j+1`` in the high nibble of byte
  ``j``; one E4M3 scale per 16-element K group, ``uint8[N, K/16]``; one FP32
  per-tensor scale.
* W8 (FP8 E4M3, "w8a16_gemm_m16.rs"): ``uint8[N, K]`` E4M3 codes and FP32
  block scales ``float32[ceil(N/128), K/128]``.
"""
from __future__ import annotations

import numpy as np

Q2_GROUP = 128
Q2_BLOCK_BYTES = 34
W4_GROUP = 16
W8_BLOCK = 128

SEED_BASE = 20261202


def seed_for(workload: int, m: int) -> int:
    """Seed recipe: base + 1000 * workload index + M."""
    return SEED_BASE + 1000 * int(workload) + int(m)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


# ---------------------------------------------------------------- BF16 inputs
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (round-to-nearest-even); returns uint16."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(m: int, k: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """A ~ N(0, 1) * scale rounded to BF16, as uint16[m, k]."""
    x = rng(seed).standard_normal((m, k), dtype=np.float32) * np.float32(scale)
    return bf16_bits_from_f32(x)


# ---------------------------------------------------------------- E4M3 encoder
def _e4m3_table() -> np.ndarray:
    """Non-negative finite E4M3 values for codes 0..126 (OCP FP8, bias 7)."""
    c = np.arange(127)
    e = c >> 3
    m = c & 7
    sub = m.astype(np.float64) * 2.0 ** -9
    nrm = (1.0 + m / 8.0) * 2.0 ** (e.astype(np.float64) - 7)
    return np.where(e == 0, sub, nrm)


_E4M3_POS = _e4m3_table()


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Quantise float values to E4M3 codes: nearest, ties to even, saturating
    at +-448; returns uint8 codes. Input-generation helper only."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.minimum(np.abs(x), _E4M3_POS[-1])
    hi = np.clip(np.searchsorted(_E4M3_POS, ax, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    dlo = ax - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - ax
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    sign = (np.signbit(x) & (code != 0)).astype(np.uint8) << 7
    return code | sign


# ---------------------------------------------------------------- Q2_0 packing
def pack_q2(codes: np.ndarray, d_f16: np.ndarray) -> np.ndarray:
    """Lay out 2-bit codes ``uint8[N, K]`` (values 0..3) and fp16 scales
    ``float16[N, K/128]`` as Q2_0 blocks; returns ``uint8[N, 34*K/128]``."""
    codes = np.asarray(codes, dtype=np.uint8)
    n, k = codes.shape
    assert k % Q2_GROUP == 0
    g = k // Q2_GROUP
    d_f16 = np.asarray(d_f16, dtype=np.float16).reshape(n, g)
    c = (codes & 3).reshape(n, g, 32, 4).astype(np.uint8)
    code_bytes = c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)
    d_bytes = d_f16.astype("<f2").view(np.uint8).reshape(n, g, 2)
    blocks = np.concatenate([code_bytes, d_bytes], axis=2)  # [n, g, 34]
    return np.ascontiguousarray(blocks.reshape(n, g * Q2_BLOCK_BYTES))


def q2_weights(n: int, k: int, seed: int, d_low: float = 0.01, d_high: float = 0.05):
    """Codes uniform in {0,1,2}; d uniform [d_low, d_high] rounded to fp16.
    Returns (packed uint8[N, 34*K/128], codes uint8[N,K], d float16[N,K/128])."""
    r = rng(seed)
    codes = r.integers(0, 3, size=(n, k), dtype=np.uint8)
    d = r.uniform(d_low, d_high, size=(n, k // Q2_GROUP)).astype(np.float16)
    return pack_q2(codes, d), codes, d


# ---------------------------------------------------------------- W4 packing
def pack_w4(nibbles: np.ndarray) -> np.ndarray:
    """``uint8[N, K]`` nibbles (0..15) -> ``uint8[N, K/2]``, element 2j low."""
    x = np.asarray(nibbles, dtype=np.uint8) & 0xF
    return np.ascontiguousarray(x[:, 0::2] | (x[:, 1::2] << 4))


def w4_weights(n: int, k: int, seed: int, scale_sigma: float = 0.05):
    """E2M1 codes uniform over the 16 encodings; E4M3 group scales from
    |N(0,1)|*scale_sigma. Returns (codes uint8[N,K/2], scales uint8[N,K/16],
    nibbles uint8[N,K])."""
    r = rng(seed)
    nib = r.integers(0, 16, size=(n, k), dtype=np.uint8)
    s = np.abs(r.standard_normal((n, k // W4_GROUP))) * scale_sigma
    return pack_w4(nib), e4m3_round(s), nib


# ---------------------------------------------------------------- W8 packing
def w8_weights(n: int, k: int, seed: int, sigma: float = 0.05,
               s_low: float = 0.5, s_high: float = 2.0):
    """E4M3 weights from N(0,1)*sigma; FP32 block scales uniform
    [s_low, s_high] of shape [ceil(N/128), K/128]."""
    r = rng(seed)
    w = e4m3_round(r.standard_normal((n, k)) * sigma)
    nb = (n + W8_BLOCK - 1) // W8_BLOCK
    s = r.uniform(s_low, s_high, size=(nb, k // W8_BLOCK)).astype(np.float32)
    return w, s


# ---------------------------------------------------------------- sizes
def q2_weight_bytes(n: int, k: int) -> int:
    return n * (k // Q2_GROUP) * Q2_BLOCK_BYTES


def w4_weight_bytes(n: int, k: int) -> int:
    """Packed codes + E4M3 group scales (the per-tensor scale is not counted)."""
    return n * k // 2 + n * k // W4_GROUP


def w8_weight_bytes(n: int, k: int) -> int:
    return n * k + ((n + W8_BLOCK - 1) // W8_BLOCK) * (k // W8_BLOCK) * 4
