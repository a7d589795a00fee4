"""fp8_gemm_dense_noalloc: the dense GEMM for callers that cannot allocate.

Some callers only hold device pointers handed to them (no allocator), so they
cannot pass the split-K workspace that fp8_gemm_dense asks for on
decode-sized shapes. The no-allocation entry point uses a fixed scratch array
inside the library instead. These tests call it through the C ABI and check
its output against the oracle's FP64 product of the same (oracle-quantized)
operands, within the GEMM tolerance the other GPU tests use, on two calls in
a row (the shared scratch must be left usable by the first call). Shapes that
split K are asserted to need scratch and run under both split policies:
Stream-K, which sums its partials in the static array, and the cluster
split, which needs none.
The file sorts last so that a run stopping at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import gemm, quant
from parity import compare_gemm, dev, pad_rows_scale, to_np32

pytestmark = pytest.mark.gpu


def _entry(fg):
    f = fg.lib.fp8_gemm_dense_noalloc
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.restype = ci
    f.argtypes = [vp, vp, vp, vp, ci, vp, ci, ci, i64, i64, i64, vp]
    return f


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _operands(M, N, K, seed, col_blocks):
    """Oracle-quantized A (all rows) and B (all rows), plus the oracle's
    FP64 product restricted to the given 128-column blocks of C."""
    x = wl.activations(M, K, seed, device="cpu")
    w = wl.weights((N, K), seed + 1, device="cpu")
    qa, sa = quant.quant_1x128(to_np32(x))
    qb, sb = quant.quant_128x128(to_np32(w))
    refs = {}
    for nb in col_blocks:
        cols = slice(nb * 128, min(N, nb * 128 + 128))
        refs[nb] = gemm.gemm_dense(qa, sa, qb[cols], sb[nb:nb + 1])
    return dev(qa), dev(pad_rows_scale(sa, M)), dev(qb), dev(sb), refs


@pytest.fixture(params=["stream", "cluster"])
def policy(request, lib):
    lib.set_split_policy(lib.SPLIT_STREAM if request.param == "stream" else lib.SPLIT_CLUSTER)
    yield request.param
    lib.set_split_policy(lib.SPLIT_AUTO)


@pytest.mark.parametrize("M,N,K,out_dtype,splits", [
    (64, 4096, 7168, torch.bfloat16, True),    # splits K: Stream-K uses the static scratch
    (128, 7168, 2048, torch.bfloat16, True),   # splits K
    (64, 520, 2048, torch.float32, True),      # splits K, FP32 output
    (1024, 4096, 512, torch.bfloat16, False),  # 128 tiles fill the GPU: no split, no scratch
])
def test_noalloc_matches_oracle(lib, M, N, K, out_dtype, splits, policy):
    fg = lib
    f = _entry(fg)
    need = fg.gemm_workspace_size(M, N, K)
    assert (need > 0) == splits, f"scratch need {need} bytes for {M}x{N}x{K}"
    nbl = (N + 127) // 128
    blocks = sorted({0, nbl // 2, nbl - 1})
    qa, sa, qb, sb, refs = _operands(M, N, K, 9100 + M + N, blocks)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = fg.FP32 if out_dtype == torch.float32 else fg.BF16
    for _ in range(2):
        c = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
        rc = f(_p(qa), _p(sa), _p(qb), _p(sb), fg.SCALE_BLOCK128, _p(c), code, 0, M, N, K, stream)
        assert rc == 0, fg.lib.fp8fg_last_error_string().decode()
        fg.check()
        for nb, ref in refs.items():
            compare_gemm(c[:, nb * 128:min(N, nb * 128 + 128)], ref, out_dtype == torch.bfloat16)


def test_noalloc_fp32_accumulate_matches_oracle(lib, policy):
    # C += A B^T into a nonzero FP32 C: with K split, the partials' sum is
    # added into C once (by the last Stream-K piece of each tile, or by the
    # cluster's reduction)
    fg = lib
    f = _entry(fg)
    M, N, K = 64, 1792, 6912
    assert fg.gemm_workspace_size(M, N, K) > 0
    blocks = [0, 7, 13]
    qa, sa, qb, sb, refs = _operands(M, N, K, 9301, blocks)
    c0 = wl.normal((M, N), 9302, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        c = c0.clone()
        rc = f(_p(qa), _p(sa), _p(qb), _p(sb), fg.SCALE_BLOCK128, _p(c), fg.FP32, 1, M, N, K, stream)
        assert rc == 0, fg.lib.fp8fg_last_error_string().decode()
        fg.check()
        for nb, ref in refs.items():
            cols = slice(nb * 128, nb * 128 + 128)
            compare_gemm(c[:, cols], ref + c0[:, cols].double().cpu().numpy(), False)


def test_noalloc_rejects_bad_arguments_without_enqueueing(lib):
    fg = lib
    f = _entry(fg)
    good = torch.zeros(16, dtype=torch.uint8, device="cuda")
    rc = f(_p(good), _p(good), _p(good), _p(good), 0, _p(good), fg.BF16, 0, 64, 100, 128, None)
    assert rc == fg.ERR_UNSUPPORTED_SHAPE
    rc = f(_p(good), _p(good), _p(good), _p(good), 0, _p(good), fg.BF16, 1, 64, 128, 128, None)
    assert rc == fg.ERR_INVALID_ARG
    assert f(None, None, None, None, 0, None, fg.BF16, 0, 0, 128, 128, None) == fg.OK
    fg.check()
