"""Block-scaled MMA path (FP8FG_SCALE_ROW_POW2) against the oracle.

When both operands carry power-of-two scales per row and 128-wide K block
(the backward pass's 128x1 tiles with power-of-2 scaling factors,
DeepSeek-V3 report excerpt, page 2, paragraph 1), the dense FP32 GEMM
applies the scales inside the tensor core (tcgen05 block-scaled MMA, UE8M0)
and accumulates over all of K in TMEM. The result is the same product as the
promotion path's up to the order of FP32 additions, checked here against
the oracle's FP64 reference at the GEMM tolerance.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import gemm, quant
from parity import compare_gemm, dev, pad_rows_scale, to_np32

pytestmark = pytest.mark.gpu


def _operands(T, N, C, seed):
    """G [T, N] bf16 and X [T, C] -> oracle 128x1 pow2 operands (transposed)."""
    g = wl.normal((T, N), seed, device="cpu", dtype=torch.bfloat16)
    x = wl.activations(T, C, seed + 1, device="cpu")
    qgT, sgT = quant.requant_128x1(to_np32(g), None, None, True)
    qxT, sxT = quant.requant_128x1(to_np32(x), None, None, True)
    return qgT, sgT, qxT, sxT


@pytest.mark.parametrize("T,N,C,accumulate", [
    (384, 136, 264, False),    # ragged rows and columns: one 224-column tile and a partial one
    (512, 1024, 2240, True),   # 80 tiles, C +=
    (2048, 256, 448, False),   # long K: 16 K blocks chained in TMEM
])
def test_block_scaled_wgrad_matches_oracle(lib, T, N, C, accumulate):
    qgT, sgT, qxT, sxT = _operands(T, N, C, 7000 + T + N)
    base = wl.normal((N, C), 7001, device="cuda") if accumulate else None
    out = base.clone() if accumulate else torch.full((N, C), float("nan"), dtype=torch.float32, device="cuda")
    lib.fp8_gemm_dense_out(dev(qgT), dev(pad_rows_scale(sgT, N)), dev(qxT), dev(pad_rows_scale(sxT, C)), out,
                           b_scale_kind=lib.SCALE_ROW_POW2, accumulate=accumulate)
    lib.check()
    ref = gemm.wgrad(qgT, sgT, qxT, sxT)
    if accumulate:
        ref = ref + base.double().cpu().numpy()
    compare_gemm(out, ref, False)


def test_block_scaled_and_promoted_paths_agree(lib):
    T, N, C = 1024, 512, 896
    qgT, sgT, qxT, sxT = _operands(T, N, C, 7101)
    args = (dev(qgT), dev(pad_rows_scale(sgT, N)), dev(qxT), dev(pad_rows_scale(sxT, C)))
    o1 = lib.fp8_gemm_dense(*args, out_dtype=torch.float32, b_scale_kind=lib.SCALE_ROW_POW2)
    o2 = lib.fp8_gemm_dense(*args, out_dtype=torch.float32, b_scale_kind=lib.SCALE_ROW)
    lib.check()
    compare_gemm(o1, o2.double().cpu().numpy(), False)


def test_block_scaled_rejects_a_scale_that_is_not_a_power_of_two(lib):
    T, N, C = 256, 256, 224
    g = wl.normal((T, N), 7201, device="cpu", dtype=torch.bfloat16)
    x = wl.activations(T, C, 7202, device="cpu")
    qgT, sgT = quant.requant_128x1(to_np32(g), None, None, False)   # amax/448 scales
    qxT, sxT = quant.requant_128x1(to_np32(x), None, None, True)
    assert np.any(np.frexp(sgT)[0] != 0.5), "the test needs scales that are not powers of two"
    out = torch.empty((N, C), dtype=torch.float32, device="cuda")
    lib.fp8_gemm_dense_out(dev(qgT), dev(pad_rows_scale(sgT, N)), dev(qxT), dev(pad_rows_scale(sxT, C)), out,
                           b_scale_kind=lib.SCALE_ROW_POW2)
    with pytest.raises(lib.Fp8fgError) as ei:
        lib.check()
    assert ei.value.code == lib.ERR_INVALID_ARG
    lib.check()  # the status word is clear again


def test_block_scaled_timeout_reports_error_and_context_survives(lib):
    T, N, C = 512, 512, 448
    qgT, sgT, qxT, sxT = _operands(T, N, C, 7301)
    args = (dev(qgT), dev(pad_rows_scale(sgT, N)), dev(qxT), dev(pad_rows_scale(sxT, C)))
    lib.check()
    try:
        lib.debug_set(1, 50_000_000)
        lib.debug_set(2, 1)
        lib.fp8_gemm_dense(*args, out_dtype=torch.float32, b_scale_kind=lib.SCALE_ROW_POW2)
        with pytest.raises(lib.Fp8fgError) as ei:
            lib.check()
        assert ei.value.code == lib.ERR_TIMEOUT
    finally:
        lib.debug_set(2, -1)
        lib.debug_set(1, 0)
    out = lib.fp8_gemm_dense(*args, out_dtype=torch.float32, b_scale_kind=lib.SCALE_ROW_POW2)
    lib.check()
    compare_gemm(out, gemm.wgrad(qgT, sgT, qxT, sxT), False)


@pytest.mark.slow
def test_block_scaled_dense_wgrad_prefill_tokens_sampled(lib):
    # dW[4096, 7168] += G^T X over the 4096 prefill tokens on the block-scaled path
    T, N, C = 4096, 4096, 7168
    g = wl.normal((T, N), 1021, device="cuda", dtype=torch.bfloat16)
    x = wl.activations(T, C, 1022, device="cuda")
    qx, sx = lib.fp8_quant_1x128(x)
    qxT, sxT = lib.fp8_requant_128x1(qx.view(torch.float8_e4m3fn), sx, pow2=True)
    qgT, sgT = lib.fp8_requant_128x1(g, pow2=True)
    base = wl.normal((N, C), 1023, device="cuda")
    out = base.clone()
    lib.fp8_gemm_dense_out(qgT, sgT, qxT, sxT, out, b_scale_kind=lib.SCALE_ROW_POW2, accumulate=True)
    lib.check()
    rng = np.random.default_rng(13)
    for nb, cb in [(0, 0), (N // 128 - 1, C // 128 - 1), tuple(rng.integers(0, (N // 128, C // 128)))]:
        rows = slice(nb * 128, nb * 128 + 128)
        cols = slice(cb * 128, cb * 128 + 128)
        q_o, s_o = quant.quant_1x128(to_np32(x[:, cols]))
        qxT_o, sxT_o = quant.requant_128x1(q_o, s_o, None, True)
        qgT_o, sgT_o = quant.requant_128x1(to_np32(g[:, rows]), None, None, True)
        ref = gemm.wgrad(qgT_o, sgT_o, qxT_o, sxT_o) + base[rows, cols].double().cpu().numpy()
        compare_gemm(out[rows, cols], ref, False)
