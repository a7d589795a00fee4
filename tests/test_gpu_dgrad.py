"""Data gradient dX = dY W on the GPU (fp8_gemm_dgrad) against the oracle.

The weight is the forward pass's E4M3 bytes and 128x128 block scales, read
by the kernel as its own transpose (MN-major operand); dY is quantized per
1x128 tile along N. Operands come from the oracle's quantizers; the
reference is the oracle's FP64 product (DeepSeek-V3 report excerpt, page 1,
paragraph 3: Dgrad in FP8; page 2, paragraph 3: transposed GEMMs).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import gemm, quant
from parity import compare_gemm, dev, pad_rows_scale, to_np32

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    dy = wl.normal((M, N), seed, device="cpu", dtype=torch.bfloat16)
    w = wl.weights((N, K), seed + 1, device="cpu")
    qdy, sdy = quant.quant_1x128(to_np32(dy))
    qw, sw = quant.quant_128x128(to_np32(w))
    return qdy, sdy, qw, sw, dev(qdy), dev(pad_rows_scale(sdy, M)), dev(qw), dev(sw)


@pytest.mark.parametrize("M,N,K,out_dtype", [
    (256, 512, 384, torch.bfloat16),
    (200, 384, 1024, torch.bfloat16),   # ragged rows
    (130, 1024, 640, torch.float32),    # two row tiles, partial last one
    (64, 2048, 1024, torch.bfloat16),   # decode-sized: K split over the SMs
    (1024, 1024, 2048, torch.bfloat16), # several tiles per CTA
])
def test_dgrad_matches_oracle(lib, M, N, K, out_dtype):
    qdy, sdy, qw, sw, qdy_d, sdy_d, qw_d, sw_d = _operands(M, N, K, 6000 + M + K)
    dx = lib.fp8_gemm_dgrad(qdy_d, sdy_d, qw_d, sw_d, out_dtype=out_dtype)
    lib.check()
    compare_gemm(dx, gemm.dgrad(qdy, sdy, qw, sw), out_dtype == torch.bfloat16)


@pytest.mark.parametrize("policy", [1, 2])  # Stream-K, cluster split
@pytest.mark.parametrize("M,N,K,out_dtype", [(64, 2048, 1024, torch.bfloat16), (96, 4096, 1152, torch.float32)])
def test_dgrad_decode_split(lib, M, N, K, out_dtype, policy):
    # W read MN-major with the reduction dimension split over the SMs
    qdy, sdy, qw, sw, qdy_d, sdy_d, qw_d, sw_d = _operands(M, N, K, 6200 + M + K)
    lib.set_split_policy(policy)
    try:
        outs = [lib.fp8_gemm_dgrad(qdy_d, sdy_d, qw_d, sw_d, out_dtype=out_dtype) for _ in range(2)]
        lib.check()
    finally:
        lib.set_split_policy(lib.SPLIT_AUTO)
    compare_gemm(outs[0], gemm.dgrad(qdy, sdy, qw, sw), out_dtype == torch.bfloat16)
    assert torch.equal(outs[0], outs[1])


def test_dgrad_fp32_accumulate(lib):
    M, N, K = 192, 512, 768
    qdy, sdy, qw, sw, qdy_d, sdy_d, qw_d, sw_d = _operands(M, N, K, 6101)
    base = wl.normal((M, K), 6102, device="cuda")
    dx = base.clone()
    lib.fp8_gemm_dgrad_out(qdy_d, sdy_d, qw_d, sw_d, dx, accumulate=True, workspace=lib.gemm_workspace(M, K, N))
    lib.check()
    compare_gemm(dx, gemm.dgrad(qdy, sdy, qw, sw) + base.double().cpu().numpy(), False)


def test_dgrad_rejects_bad_shapes(lib):
    t = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    f = torch.zeros(4096, dtype=torch.float32, device="cuda")
    c = torch.zeros(64 * 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.Fp8fgError) as ei:   # N (the reduction) not a multiple of 128
        lib.fp8_gemm_dgrad_out(t[:64 * 200].view(64, 200), f, t[:200 * 128].view(200, 128), f, c[:64 * 128].view(64, 128))
    assert ei.value.code == lib.ERR_UNSUPPORTED_SHAPE


@pytest.mark.slow
@pytest.mark.parametrize("N", [7168, 4096])
def test_dgrad_prefill_sampled(lib, N):
    # the prefill layers' data gradient: dX[4096, 7168] = dY[4096, N] W[N, 7168]
    M, K = wl.PREFILL_M, wl.PREFILL_K
    dy = wl.normal((M, N), 1031 + N, device="cuda", dtype=torch.bfloat16)
    w = wl.weights((N, K), 2000 + N, device="cuda")
    qdy_d, sdy_d = lib.fp8_quant_1x128(dy)
    qw_d, sw_d = lib.fp8_quant_128x128(w)
    dx = lib.fp8_gemm_dgrad(qdy_d, sdy_d, qw_d, sw_d)
    lib.check()
    rng = np.random.default_rng(N)
    rows = np.sort(rng.choice(M, 40, replace=False))
    qdy, sdy = quant.quant_1x128(to_np32(dy[rows]))
    qw, sw = quant.quant_128x128(to_np32(w))
    for kb in (0, 23, K // 128 - 1):
        cols = np.arange(kb * 128, kb * 128 + 128)
        compare_gemm(dx[rows][:, kb * 128:kb * 128 + 128], gemm.dgrad(qdy, sdy, qw, sw, cols=cols), True)
