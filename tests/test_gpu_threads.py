"""Calls from several host threads at once (GPU needed).

The C ABI states that every entry point may be called from several host
threads. The library keeps process-wide state that the first call of a
shape fills in: launch plans, encoded tensor maps, occupancy queries and the
shared-memory attributes of each kernel. Here several threads, each with its
own CUDA stream, inputs and outputs, start together on shapes no other test
uses, so they race to fill those entries; every result must equal the same
call made alone afterwards, bit for bit.
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
