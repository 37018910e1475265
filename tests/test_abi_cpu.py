"""C-ABI checks that need no GPU: libwqp.so loads, exports every symbol that
include/wqp.h declares, rejects bad arguments before any CUDA call, and the
host row-chunking reproduces the source page's worked example."""
from __future__ import annotations

import ctypes
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from weight_only_quantized_packed_gb300 import build

    build.build()
    from weight_only_quantized_packed_gb300 import binding

    return binding.lib()


def _header_functions():
    src = open(os.path.join(ROOT, "include", "wqp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M))


def test_library_exports_every_declared_symbol(L):
    from weight_only_quantized_packed_gb300 import binding

    decl = _header_functions()
    assert decl, "no declarations parsed"
    assert decl == set(binding.EXPORTS), decl ^ set(binding.EXPORTS)
    for name in decl:
        assert hasattr(L, name), name
    assert L.wqp_abi_version() == 1


def test_status_strings(L):
    from weight_only_quantized_packed_gb300 import binding

    assert binding.status_string(0) == "WQP_OK"
    assert binding.status_string(1) == "WQP_ERR_INVALID_ARG"
    assert binding.status_string(4) == "WQP_ERR_DEVICE_TIMEOUT"
    assert binding.status_string(99) == "WQP_ERR_UNKNOWN"


def test_row_chunks_pages_worked_example(L):
    """"gemv_q2_vec.rs", tests `launch_chunks_advance_...` and
    `batchm_row_chunks_cover_all_rows_exactly`."""
    from weight_only_quantized_packed_gb300 import binding

    g = json.load(open(os.path.join(ROOT, "tests", "golden", "chunk_example.json")))
    ex = g["worked_example"]
    got = binding.row_chunks(ex["m"], ex["k"], ex["n"], g["max_rows"])
    assert [list(c) for c in got] == ex["chunks"]
    for m in g["coverage_m"]:
        ch = binding.row_chunks(m, 256, 5, g["max_rows"])
        r0 = 0
        for a_off, c_off, rows in ch:
            assert a_off == r0 * 256 * 2 and c_off == r0 * 5 * 2
            assert 1 <= rows <= g["max_rows"]
            r0 += rows
        assert r0 == m
        assert (len(ch) == 0) == (m == 0)


def test_row_chunks_rejects_small_cap(L):
    buf = (ctypes.c_longlong * 3)()
    assert L.wqp_row_chunks(17, 256, 5, 8, buf, 1) == -1
    assert L.wqp_row_chunks(0, 256, 5, 8, buf, 0) == 0


def test_selftest_limit_is_validated_before_any_cuda_call(L):
    for limit_us in (0, -3, 1000001):
        assert L.wqp_selftest_wait_timeout(limit_us, None) == 1
        assert b"limit_us" in L.wqp_last_error()


def test_pdl_policy_roundtrip(L):
    old = L.wqp_set_pdl(1)
    assert L.wqp_set_pdl(old) == 1


# Aligned fake device addresses: validation must reject before any CUDA call.
P16 = ctypes.c_void_p(0x10000)
P16b = ctypes.c_void_p(0x20000)
P16c = ctypes.c_void_p(0x30000)
NUL = ctypes.c_void_p(0)
ODD = ctypes.c_void_p(0x10008)
S = ctypes.c_void_p(0)


@pytest.mark.parametrize("args,why", [
    ((P16, P16b, NUL, P16c, -1, 8, 128, S), "M<0"),
    ((P16, P16b, NUL, P16c, 1, 0, 128, S), "N<1"),
    ((P16, P16b, NUL, P16c, 1, 8, 100, S), "K%128"),
    ((P16, P16b, NUL, P16c, 1, 8, 0, S), "K=0"),
    ((P16, P16b, NUL, P16c, 1, 8, (1 << 20) + 128, S), "K>2^20"),
    ((P16, P16b, NUL, P16c, 1, (1 << 24) + 1, 128, S), "N>2^24"),
    ((NUL, P16b, NUL, P16c, 1, 8, 128, S), "A NULL"),
    ((P16, NUL, NUL, P16c, 1, 8, 128, S), "W NULL"),
    ((P16, P16b, NUL, NUL, 1, 8, 128, S), "C NULL"),
    ((ODD, P16b, NUL, P16c, 1, 8, 128, S), "A misaligned"),
    ((P16, ODD, NUL, P16c, 1, 8, 128, S), "W misaligned"),
    ((P16, P16b, P16, P16c, 1, 8, 128, S), "Q2 scales must be NULL"),
    ((P16, P16b, NUL, ctypes.c_void_p(0x30001), 1, 8, 128, S), "C odd"),
])
def test_q2_validation(L, args, why):
    assert L.q2_gemv(*args) == 1, why
    assert L.wqp_last_error().decode(), why


@pytest.mark.parametrize("name", ["q2_gemm_tc", "q2_gemm_mma"])
def test_largest_shapes_accepted_and_one_past_rejected(L, name):
    """The limits K <= 2^20 and N <= 2^24 on the tensor-core entries: one
    past each is rejected before any CUDA call (the largest K itself runs on
    the GPU in the long-K parity tests)."""
    f = getattr(L, name)
    assert f(P16, P16b, P16c, 1, 8, (1 << 20) + 1024, S) == 1
    assert b"2^20" in L.wqp_last_error()
    assert f(P16, P16b, P16c, 1, (1 << 24) + 1, 1024, S) == 1
    assert b"2^24" in L.wqp_last_error()


def test_validation_other_formats(L):
    # W4/W8 need a scale pointer; M < 0 is invalid for every entry.
    assert L.w4a16_gemv(P16, P16b, NUL, P16c, 1, 8, 128, S) == 1
    assert L.w4a16_gemv(P16, P16b, ctypes.c_void_p(0x40008), P16c, 1, 8, 128, S) == 1  # 16-B scales
    assert L.w8a16_gemm(P16, P16b, NUL, P16c, 1, 8, 128, S) == 1
    assert L.w8a16_gemm(P16, P16b, ctypes.c_void_p(0x40002), P16c, 1, 8, 128, S) == 1
    assert L.w8a16_gemm_tc(P16, P16b, P16, P16c, -1, 8, 128, S) == 1
    assert L.w4a16_gemm_tc(P16, P16b, P16, P16c, -1, 8, 256, S) == 1
    # strided: lda < K, lda % 8, ldc < N
    assert L.q2_gemv_strided(P16, 120, P16b, P16c, 8, 1, 8, 128, S) == 1
    assert L.q2_gemv_strided(P16, 132, P16b, P16c, 8, 1, 8, 128, S) == 1
    assert L.q2_gemv_strided(P16, 128, P16b, P16c, 7, 1, 8, 128, S) == 1
    assert L.w4a16_gemv_ex(P16, 128, P16b, P16, ctypes.c_float(float("nan")), P16c, 8, 1, 8, 128, S) == 1
    # dequant
    assert L.q2_dequant(P16, NUL, 8, 128, S) == 1
    assert L.q2_dequant(P16, P16b, 8, 100, S) == 1
    assert L.w8a16_dequant(P16, NUL, P16b, 8, 128, S) == 1


@pytest.mark.parametrize("name", ["q2_gemm_tc", "q2_gemm_mma"])
def test_q2_tensor_core_validation(L, name):
    """Both Q2_0 tensor-core entries: M >= 0, K % 1024 == 0, 16-byte
    aligned A and W, row pitches; rejected before any CUDA call."""
    f = getattr(L, name)
    fs = getattr(L, name + "_strided")
    assert f(P16, P16b, P16c, -1, 8, 1024, S) == 1
    for k in (640, 1152, 128):
        assert f(P16, P16b, P16c, 1, 8, k, S) == 1, k
        assert b"1024" in L.wqp_last_error(), k
    assert f(ODD, P16b, P16c, 1, 8, 1024, S) == 1
    assert f(P16, ODD, P16c, 1, 8, 1024, S) == 1
    assert f(NUL, P16b, P16c, 1, 8, 1024, S) == 1
    assert f(P16, P16b, P16c, 1, 0, 1024, S) == 1
    # strided: lda < K, lda % 8, ldc < N
    assert fs(P16, 1000, P16b, P16c, 8, 1, 8, 1024, S) == 1
    assert fs(P16, 1028, P16b, P16c, 8, 1, 8, 1024, S) == 1
    assert fs(P16, 1024, P16b, P16c, 7, 1, 8, 1024, S) == 1
    assert name.encode() in L.wqp_last_error()


def test_m_zero_is_a_noop(L):
    """M == 0 returns OK without touching CUDA (the page's empty chunk list)."""
    assert L.q2_gemv(P16, P16b, NUL, P16c, 0, 8, 128, S) == 0
    assert L.w8a16_gemm(P16, P16b, P16, P16c, 0, 8, 128, S) == 0
    assert L.w4a16_gemv(P16, P16b, P16, P16c, 0, 8, 128, S) == 0
    # The tensor-core entries too (any M >= 0 is accepted; M > 16 runs in
    # 16-row launches).
    assert L.w8a16_gemm_tc(P16, P16b, P16, P16c, 0, 8, 128, S) == 0
    assert L.w4a16_gemm_tc(P16, P16b, P16, P16c, 0, 8, 256, S) == 0
    assert L.q2_gemm_tc(P16, P16b, P16c, 0, 8, 1024, S) == 0
    assert L.q2_gemm_mma(P16, P16b, P16c, 0, 8, 1024, S) == 0


def test_product_package_does_not_import_oracle():
    """The product path must never reach the oracle."""
    pkg = os.path.join(ROOT, "weight_only_quantized_packed_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f
                assert "liboracle" not in txt, f


def test_missing_library_and_host_tensors_fail_loudly():
    """No fallback: without libwqp.so every entry raises ImportError, and
    host (CPU) tensors are refused before any call. Run in a child process
    so that this process keeps its loaded library."""
    import subprocess
    import sys
    import textwrap

    code = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {ROOT!r})
        import torch
        from weight_only_quantized_packed_gb300 import binding as B
        A = torch.zeros((1, 1024), dtype=torch.bfloat16)
        W = torch.zeros((16, 272), dtype=torch.uint8)
        for f in (lambda: B.q2_gemm_mma(A, W, 16, 1024), lambda: B.q2_gemv(A, W, 16, 1024)):
            try:
                f()
                print("computed")
            except ValueError as e:
                print("refused" if "no CPU fallback" in str(e) else "other: " + str(e))
        B.lib_path = {os.path.join(ROOT, "no_such_dir", "libwqp.so")!r}
        B._lib = None
        for f in (B.lib, lambda: B.set_pdl(True), B.get_device_error):
            try:
                f()
                print("loaded")
            except ImportError:
                print("importerror")
    """)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == ["refused", "refused", "importerror", "importerror", "importerror"], r.stdout
