"""Failure path on the GPU without a fault: a bounded wait that nothing
completes must give up, report WQP_ERR_DEVICE_TIMEOUT through the device error
word, and leave the context usable (GPU needed)."""
from __future__ import annotations

import time

import pytest

from tests import _gpu as G
from tests._tol import assert_scalar_term

pytestmark = pytest.mark.gpu

WQP_ERR_DEVICE_TIMEOUT = 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__

    __graft_entry__.build()
    import weight_only_quantized_packed_gb300 as wqp

    wqp.set_pdl(False)
    assert wqp.get_device_error() == 0
    yield
    assert wqp.get_device_error() == 0


def test_bounded_wait_timeout_is_reported_and_context_stays_usable(oracle_lib):
    import weight_only_quantized_packed_gb300 as wqp

    t0 = time.perf_counter()
    wqp.selftest_wait_timeout(2000)        # 2 ms
    status = wqp.get_device_error()          # synchronises: the kernel has returned
    elapsed = time.perf_counter() - t0
    assert status == WQP_ERR_DEVICE_TIMEOUT, wqp.status_string(status)
    assert elapsed < 5.0
    assert wqp.get_device_error() == 0       # reading cleared the word
    # The context still computes: a small GEMV against the oracle.
    d = G.make("q2", 3, 64, 1024, seed=9)
    C = G.host_bits(G.run_gpu(d))
    ref = G.run_oracle(oracle_lib, d)
    assert_scalar_term(C, ref, 1024, "q2 after the timeout self-test")


def test_selftest_rejects_bad_limits():
    import weight_only_quantized_packed_gb300 as wqp

    for limit_us in (0, -1, 1000001):
        with pytest.raises(wqp.WqpError):
            wqp.selftest_wait_timeout(limit_us)
