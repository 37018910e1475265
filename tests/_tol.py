"""Comparison helpers shared by the oracle pins and the GPU parity tests.

Tolerances (stated once, used everywhere):

* Integer/byte work (dequant, row identity across M): bit-exact.
* Scalar-FMA GEMVs vs the oracle: a BF16 ULP distance of at most 1, or
  ``|gpu - oracle| <= 8 * sqrt(K) * 2**-24 * S``, where ``S = sum_k |a*w|``
  (fp64, from the oracle). Both sides accumulate in FP32 but in different
  orders. The second term is a probabilistic bound on FP32 reordering error,
  ``lambda * sqrt(K) * u * S`` with ``u = 2**-24`` and ``lambda = 8``
  (Higham & Mary, 2019). It matters only for outputs near zero, where one
  BF16 ULP is smaller than the reordering noise.
* Tensor-core path: at most 4 BF16 ULP, or
  ``|gpu - oracle| < 1e-3 * sqrt(K) * rms(a[m,:]) * max_k |w[n,k]|``
  (w including its block scale, max taken per weight row n).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch


def bf16_bits(x) -> np.ndarray:
    """Round float values to BF16 via torch (RNE); returns uint16 bits."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_exact_bits(x64) -> np.ndarray:
    """BF16 of values that are exactly representable in float32."""
    x64 = np.asarray(x64, dtype=np.float64)
    x32 = x64.astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x64), "value not exact in f32"
    return bf16_bits(x32)


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_ulp_dist(a_bits, b_bits) -> np.ndarray:
    """Distance in BF16 units in the last place (+0 and -0 coincide)."""
    def order(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)

    return np.abs(order(a_bits) - order(b_bits))


def scalar_ok(gpu_bits, ref, K: int):
    """Mask of outputs within the scalar-FMA tolerance, and the count that
    pass only by the reordering floor."""
    d = bf16_ulp_dist(gpu_bits, ref.c)
    err = np.abs(bf16_to_f64(gpu_bits) - bf16_to_f64(ref.c))
    floor = 8.0 * np.sqrt(K) * 2.0 ** -24 * ref.s
    ok = (d <= 1) | (err <= floor)
    only_floor = int(np.count_nonzero((d > 1) & (err <= floor)))
    return ok, only_floor


def tc_ok(gpu_bits, ref, K: int, a_rms, w_absmax):
    """Tensor-core tolerance mask; a_rms is [M], w_absmax is [N]."""
    d = bf16_ulp_dist(gpu_bits, ref.c)
    err = np.abs(bf16_to_f64(gpu_bits) - bf16_to_f64(ref.c))
    floor = 1e-3 * np.sqrt(K) * np.outer(a_rms, w_absmax)
    return (d <= 4) | (err < floor)


def assert_scalar_parity(gpu_bits, ref, K: int, what: str = ""):
    ok, only_floor = scalar_ok(gpu_bits, ref, K)
    bad = np.argwhere(~ok)
    if bad.size:
        m, n = bad[0]
        raise AssertionError(
            f"{what}: {len(bad)} outputs outside 1 ULP / floor; first at (m={m}, n={n}): "
            f"gpu={bf16_to_f64(gpu_bits[m, n])!r} oracle={bf16_to_f64(ref.c[m, n])!r} "
            f"ulp={bf16_ulp_dist(gpu_bits[m, n], ref.c[m, n])} S={ref.s[m, n]!r}")
    return only_floor


def parity_report(gpu_bits, ref, K: int) -> dict:
    """Counts behind the scalar term: outputs within 1 ULP, outputs that pass
    only by the reordering floor, and the largest ULP distance."""
    d = bf16_ulp_dist(gpu_bits, ref.c)
    ok, only_floor = scalar_ok(gpu_bits, ref, K)
    return {"n": int(d.size), "exact": int(np.count_nonzero(d == 0)), "le1ulp": int(np.count_nonzero(d <= 1)),
            "floor_only": only_floor, "fail": int(np.count_nonzero(~ok)), "max_ulp": int(d.max()) if d.size else 0}


# Outputs allowed to pass the scalar term only through the reordering floor
# (the rest must be within 1 BF16 ULP): at most 2, or 0.2 % of the outputs.
# Measured on GB300 over every parity case of the GPU tests: at most 1 in
# 1040 outputs of a case, 0.025 % or less on cases of 100,000 outputs or more.
FLOOR_ONLY_MAX_FRAC = 0.002
FLOOR_ONLY_MIN_ALLOWED = 2


def log_parity(what: str, rep: dict) -> None:
    """Append one parity report as a JSON line to $WQP_PARITY_LOG, if set."""
    path = os.environ.get("WQP_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": what, **rep}) + "\n")


def assert_scalar_term(gpu_bits, ref, K: int, what: str = "") -> dict:
    """Every output within the scalar term, the floor-only share bounded;
    returns (and logs) the counts."""
    rep = parity_report(gpu_bits, ref, K)
    log_parity(what, rep)
    assert_scalar_parity(gpu_bits, ref, K, what)
    assert rep["floor_only"] <= max(FLOOR_ONLY_MIN_ALLOWED, FLOOR_ONLY_MAX_FRAC * rep["n"]), (what, rep)
    return rep
