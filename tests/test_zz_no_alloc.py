"""fp8_gemm_dense_noalloc: the dense GEMM for callers that cannot allocate.

Some callers only hold device pointers handed to them (no allocator), so they
cannot pass the split-K workspace that fp8_gemm_dense asks for on
decode-sized shapes. The no-allocation entry point uses a scratch array the
library reserves when it is loaded instead. This test calls it through the C
ABI and checks its output against the existing fp8_gemm_dense entry point
(given a caller workspace) on the same inputs, on two calls in a row (the
shared scratch must be left usable), within the GEMM tolerance the other GPU
tests use. The file sorts last so that a run stopping at the first failure
has already run every other test.
"""
import ctypes

import pytest
import torch

import workloads as wl
from parity import compare_gemm

pytestmark = pytest.mark.gpu


def _entry(fg):
    f = fg.lib.fp8_gemm_dense_noalloc
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.restype = ci
    f.argtypes = [vp, vp, vp, vp, ci, vp, ci, ci, i64, i64, i64, vp]
    return f


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("M,N,K,out_dtype", [
    (64, 4096, 7168, torch.bfloat16),    # splits K: uses the static scratch
    (128, 7168, 2048, torch.bfloat16),   # splits K
    (64, 520, 2048, torch.float32),      # splits K, FP32 output
    (512, 1024, 1024, torch.bfloat16),   # enough tiles: no split, no scratch
])
def test_noalloc_matches_dense_entry(lib, M, N, K, out_dtype):
    fg = lib
    f = _entry(fg)
    x = wl.activations(M, K, 9100 + M, device="cuda")
    w = wl.weights((N, K), 9200 + N, device="cuda")
    qa, sa = fg.fp8_quant_1x128(x)
    qb, sb = fg.fp8_quant_128x128(w)
    ref = fg.fp8_gemm_dense(qa, sa, qb, sb, out_dtype=out_dtype)  # existing entry point, caller workspace
    torch.cuda.synchronize()
    ref_np = ref.double().cpu().numpy()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = fg.FP32 if out_dtype == torch.float32 else fg.BF16
    for _ in range(2):
        c = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
        rc = f(_p(qa), _p(sa), _p(qb), _p(sb), fg.SCALE_BLOCK128, _p(c), code, 0, M, N, K, stream)
        assert rc == 0, fg.lib.fp8fg_last_error_string().decode()
        fg.check()
        compare_gemm(c, ref_np, out_dtype == torch.bfloat16)


def test_noalloc_rejects_bad_arguments_without_enqueueing(lib):
    fg = lib
    f = _entry(fg)
    good = torch.zeros(16, dtype=torch.uint8, device="cuda")
    rc = f(_p(good), _p(good), _p(good), _p(good), 0, _p(good), fg.BF16, 0, 64, 100, 128, None)
    assert rc == fg.ERR_UNSUPPORTED_SHAPE
    rc = f(_p(good), _p(good), _p(good), _p(good), 0, _p(good), fg.BF16, 1, 64, 128, 128, None)
    assert rc == fg.ERR_INVALID_ARG
    fg.check()
