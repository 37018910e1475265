"""The library's host-side state under concurrent and many-buffer use (GPU
needed).

The library keeps process-wide state that the first call of a shape or a
weight buffer fills in: launch plans, encoded tensor maps (keyed by address,
shape, pitch and box), occupancy queries and the shared-memory attributes of
each kernel.
* Several host threads, each with its own CUDA stream, inputs and outputs,
  start together on shapes no other test uses, so they race to fill those
  entries; every result must equal the same call made alone, bit for bit.
* More weight buffers than a model's layers would give, called in turn, and
  a buffer freed and replaced at the same address by one of another shape:
  every result against the oracle.
"""
from __future__ import annotations

import threading

import numpy as np
import pytest
import torch

from tests import _gpu as G

pytestmark = pytest.mark.gpu

THREADS = 6
REPEATS = 4
# (format, engine, N, K): one shape per engine, unused elsewhere in the tests.
CASES = [(fmt, eng, n, 3072) for fmt, base in (("q2", 1111), ("w4", 1237), ("w8", 1361))
         for eng, n in ((False, base), (True, base + 16), ("mma", base + 32))]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__

    __graft_entry__.build()
    import weight_only_quantized_packed_gb300 as wqp

    yield
    assert wqp.get_device_error() == 0


def test_threads_race_on_first_calls():
    inputs = [[G.make(fmt, 5, N, K, seed=1000 + 31 * i + j) for j, (fmt, eng, N, K) in enumerate(CASES)]
              for i in range(THREADS)]
    results = [[None] * len(CASES) for _ in range(THREADS)]
    errors = []
    start = threading.Barrier(THREADS)

    def worker(i):
        try:
            stream = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(stream):
                for _ in range(REPEATS):
                    outs = [G.run_gpu(d, tc=eng) for d, (_, eng, _, _) in zip(inputs[i], CASES)]
                    stream.synchronize()
                    for j, c in enumerate(outs):
                        bits = G.host_bits(c)
                        if results[i][j] is None:
                            results[i][j] = bits
                        elif not np.array_equal(results[i][j], bits):
                            errors.append((i, CASES[j], "repeat differs"))
        except Exception as e:   # noqa: BLE001 - reported below with its thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(THREADS)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, errors[:4]
    for i in range(THREADS):
        for j, (fmt, eng, N, K) in enumerate(CASES):
            alone = G.host_bits(G.run_gpu(inputs[i][j], tc=eng))
            assert np.array_equal(alone, results[i][j]), (i, fmt, eng, N)


# Engines held to the scalar term whose weight maps come from each cache path:
# the scalar kernel's row map, a 2-D map (Q2_0 warp-level MMA; W4 tcgen05 with
# its scale map) and a 3-D map (FP8 warp-level MMA).
@pytest.mark.parametrize("fmt,eng", [("q2", False), ("q2", "mma"), ("w4", True), ("w8", "mma")])
def test_many_weight_buffers_and_reused_addresses(oracle_lib, fmt, eng):
    from tests._tol import assert_scalar_term

    N, K, M, count = 96, 1024, 3, 300
    base = G.make(fmt, M, N, K, seed=1100)
    ref = G.run_oracle(oracle_lib, base)
    bufs = [dict(base, dW=G.dev_u8(base["W"])) for _ in range(count)]   # 300 distinct addresses
    first = None
    for rnd in range(2):
        for d in bufs:
            C = G.host_bits(G.run_gpu(d, tc=eng))
            if first is None:
                first = C
                assert_scalar_term(C, ref, K, f"{fmt} {eng} many buffers")
            assert np.array_equal(C, first), (fmt, eng, rnd)
    del bufs, d
    torch.cuda.synchronize()
    # Freed blocks come back at the same addresses; a different shape there
    # must not reuse the earlier maps.
    other = G.make(fmt, M, N + 32, K, seed=1101)
    ref2 = G.run_oracle(oracle_lib, other)
    for _ in range(4):
        d = dict(other, dW=G.dev_u8(other["W"]))
        C = G.host_bits(G.run_gpu(d, tc=eng))
        assert_scalar_term(C, ref2, K, f"{fmt} {eng} reused address")
