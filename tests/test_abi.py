"""The C-ABI library builds, loads and exports every declared symbol (CPU only).

Also checks the host-side argument validation: these calls return an error
code before anything touches a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cdll():
    from fp8_fine_grained_24_b300 import build
    path = build.build()
    return ctypes.CDLL(path)


def _declared():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names += re.findall(r"FP8FG_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return names


def test_every_declared_symbol_is_exported(cdll):
    names = _declared()
    for required in ("fp8_quant_1x128", "fp8_quant_128x128", "fp8_requant_128x1", "fp8_gemm_dense",
                     "fp8_gemm_grouped_contig", "fp8_gemm_grouped_masked"):
        assert required in names
    for n in names:
        assert hasattr(cdll, n), n


def test_binding_loads_and_names_match():
    import fp8_fine_grained_24_b300 as fg
    for n in _declared():
        assert hasattr(fg.lib, n)
    assert fg.version().startswith("fp8fg")
    assert fg.scale_ld(1) == 4 and fg.scale_ld(4096) == 4096 and fg.scale_ld(4097) == 4100


def _err(fg):
    return fg.lib.fp8fg_last_error_string().decode()


def test_host_validation_without_gpu():
    import fp8_fine_grained_24_b300 as fg
    L = fg.lib
    P = ctypes.c_void_p
    good = P(0x10000)
    odd = P(0x10008)
    # quant: K not a multiple of 128
    assert L.fp8_quant_1x128(good, fg.BF16, 4, 100, 100, good, good, 0, None) == fg.ERR_UNSUPPORTED_SHAPE
    assert "multiple of 128" in _err(fg)
    # bad dtype, null pointers, misalignment, negative size
    assert L.fp8_quant_1x128(good, 7, 4, 128, 128, good, good, 0, None) == fg.ERR_INVALID_ARG
    assert L.fp8_quant_1x128(None, fg.BF16, 4, 128, 128, good, good, 0, None) == fg.ERR_INVALID_ARG
    assert L.fp8_quant_1x128(odd, fg.BF16, 4, 128, 128, good, good, 0, None) == fg.ERR_MISALIGNED
    assert L.fp8_quant_1x128(good, fg.BF16, -1, 128, 128, good, good, 0, None) == fg.ERR_INVALID_ARG
    assert L.fp8_quant_1x128(good, fg.BF16, 4, 128, 64, good, good, 0, None) == fg.ERR_INVALID_ARG
    # empty is a no-op
    assert L.fp8_quant_1x128(None, fg.BF16, 0, 128, 128, None, None, 0, None) == fg.OK
    assert L.fp8_quant_128x128(good, fg.FP32, 1, 10, 130, good, good, 0, None) == fg.ERR_UNSUPPORTED_SHAPE
    assert L.fp8_requant_128x1(good, fg.E4M3, None, 1, 128, 128, None, good, good, 0, None) == fg.ERR_INVALID_ARG
    assert L.fp8_requant_128x1(good, fg.BF16, None, 1, 100, 128, None, good, good, 0, None) == \
        fg.ERR_UNSUPPORTED_SHAPE
    # GEMMs
    args = (good, good, good, good)
    assert L.fp8_gemm_dense(*args, 0, good, fg.BF16, 0, 128, 128, 100, None, 0, None) == fg.ERR_UNSUPPORTED_SHAPE
    assert L.fp8_gemm_dense(*args, 0, good, fg.BF16, 0, 128, 100, 128, None, 0, None) == fg.ERR_UNSUPPORTED_SHAPE
    assert L.fp8_gemm_dense(*args, 0, good, fg.BF16, 1, 128, 128, 128, None, 0, None) == fg.ERR_INVALID_ARG
    assert L.fp8_gemm_dense(*args, 5, good, fg.BF16, 0, 128, 128, 128, None, 0, None) == fg.ERR_INVALID_ARG
    assert L.fp8_gemm_dense(good, good, odd, good, 0, good, fg.BF16, 0, 128, 128, 128, None, 0, None) == \
        fg.ERR_MISALIGNED
    assert L.fp8_gemm_dense(*args, 0, good, fg.BF16, 0, 0, 128, 128, None, 0, None) == fg.OK
    assert L.fp8_gemm_grouped_contig(*args, good, good, fg.BF16, 100, 128, 128, 2, None) == \
        fg.ERR_UNSUPPORTED_SHAPE
    assert L.fp8_gemm_grouped_contig(*args, None, good, fg.BF16, 128, 128, 128, 2, None) == fg.ERR_INVALID_ARG
    assert L.fp8_gemm_grouped_masked(*args, 0, good, 3, good, fg.BF16, 0, 2, 128, 128, 128, 0, None) == \
        fg.ERR_INVALID_ARG
    assert L.fp8_gemm_grouped_masked(*args, 0, None, 0, good, fg.BF16, 0, 2, 128, 128, 128, 0, None) == \
        fg.ERR_INVALID_ARG
    assert L.fp8fg_debug_set(99, 0) == fg.ERR_INVALID_ARG
    # split policy (key 4): 0 automatic, 1 Stream-K, 2 cluster split; others rejected
    for bad in (-1, 3):
        assert L.fp8fg_debug_set(4, bad) == fg.ERR_INVALID_ARG
    for v in (fg.SPLIT_STREAM, fg.SPLIT_CLUSTER, fg.SPLIT_AUTO):
        assert L.fp8fg_debug_set(4, v) == fg.OK
