"""GPU parity of the FP8 GEMMs against the oracle's FP64 product (tolerance in parity.py).

Operands are quantized by the oracle (never by the CUDA path) and uploaded;
the library multiplies them; the oracle multiplies the same dequantized
operands in FP64.
"""
import contextlib

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import gemm, quant
from parity import compare_gemm, dev, ld4, pad_rows_scale, to_np32

pytestmark = pytest.mark.gpu


def _quant_a(x, pow2=False):
    q, s = quant.quant_1x128(to_np32(x), pow2)
    M = q.shape[0]
    return q, s, dev(q), dev(pad_rows_scale(s, M))


def _quant_b(w, pow2=False):
    q, s = quant.quant_128x128(to_np32(w), pow2)
    return q, s, dev(q), dev(s)


def _dense_case(fg, M, N, K, seed, out_dtype=torch.bfloat16, a_dtype=torch.bfloat16):
    x = wl.activations(M, K, seed, device="cpu", dtype=a_dtype)
    w = wl.weights((N, K), seed + 1, device="cpu")
    qa, sa, qa_d, sa_d = _quant_a(x)
    qb, sb, qb_d, sb_d = _quant_b(w)
    c = fg.fp8_gemm_dense(qa_d, sa_d, qb_d, sb_d, out_dtype=out_dtype)
    torch.cuda.synchronize()
    cref = gemm.gemm_dense(qa, sa, qb, sb)
    return compare_gemm(c, cref, out_dtype == torch.bfloat16)


def test_dense_tiny_config(lib):
    a, b = wl.tiny_inputs(1000, device="cpu")
    qa, sa, qa_d, sa_d = _quant_a(a)
    qb, sb, qb_d, sb_d = _quant_b(b)
    c = lib.fp8_gemm_dense(qa_d, sa_d, qb_d, sb_d)
    torch.cuda.synchronize()
    compare_gemm(c, gemm.gemm_dense(qa, sa, qb, sb), True)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (200, 264, 384), (1, 8, 128), (64, 2112, 1024),
                                   (300, 520, 640), (513, 768, 256), (128, 7168, 2048),
                                   # one K block per tile on 256-wide tiles (each stage is a
                                   # tile's first and last), ragged N past the last scale block
                                   (300, 520, 128), (1500, 1288, 128)])
def test_dense_shapes(lib, M, N, K):
    _dense_case(lib, M, N, K, seed=M * 7 + N)


def test_dense_fp32_out_and_accumulate(lib):
    M, N, K = 192, 320, 512
    x = wl.activations(M, K, 11, device="cpu")
    w = wl.weights((N, K), 12, device="cpu")
    qa, sa, qa_d, sa_d = _quant_a(x)
    qb, sb, qb_d, sb_d = _quant_b(w)
    cref = gemm.gemm_dense(qa, sa, qb, sb)
    c = lib.fp8_gemm_dense(qa_d, sa_d, qb_d, sb_d, out_dtype=torch.float32)
    compare_gemm(c, cref, False)
    base = torch.randn((M, N), dtype=torch.float32, device="cuda")
    c2 = base.clone()
    lib.fp8_gemm_dense_out(qa_d, sa_d, qb_d, sb_d, c2, accumulate=True)
    compare_gemm(c2, cref + base.double().cpu().numpy(), False)


def _wgrad_operands(T, N, C, seed, valid=None):
    """G [T, N] bf16 and X [T, C] bf16 -> oracle 128x1 pow2 operands (transposed)."""
    g = wl.normal((T, N), seed, device="cpu", dtype=torch.bfloat16)
    x = wl.activations(T, C, seed + 1, device="cpu")
    qgT, sgT = quant.requant_128x1(to_np32(g), None, valid, True)
    qxT, sxT = quant.requant_128x1(to_np32(x), None, valid, True)
    return qgT, sgT, qxT, sxT


def test_dense_row_scaled_b_wgrad(lib):
    T, N, C = 384, 136, 264
    qgT, sgT, qxT, sxT = _wgrad_operands(T, N, C, 21)
    c = lib.fp8_gemm_dense(dev(qgT), dev(pad_rows_scale(sgT, N)), dev(qxT), dev(pad_rows_scale(sxT, C)),
                           out_dtype=torch.float32, b_scale_kind=lib.SCALE_ROW)
    compare_gemm(c, gemm.wgrad(qgT, sgT, qxT, sxT), False)


def test_dense_outputs_stay_in_bounds(lib):
    # canaries around C: nothing outside [M, N] is written
    M, N, K = 130, 72, 256
    x = wl.activations(M, K, 31, device="cpu")
    w = wl.weights((N, K), 32, device="cpu")
    qa, sa, qa_d, sa_d = _quant_a(x)
    qb, sb, qb_d, sb_d = _quant_b(w)
    buf = torch.full((M + 2, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    c = buf[1:M + 1]
    lib.fp8_gemm_dense_out(qa_d, sa_d, qb_d, sb_d, c)
    torch.cuda.synchronize()
    assert torch.isnan(buf[0]).all() and torch.isnan(buf[M + 1]).all()
    compare_gemm(c, gemm.gemm_dense(qa, sa, qb, sb), True)


@pytest.mark.slow
@pytest.mark.parametrize("N,pair", [(n, 0) for n in wl.PREFILL_NS] + [(7168, 1)])
def test_dense_prefill_sampled(lib, N, pair):
    M, K = wl.PREFILL_M, wl.PREFILL_K
    x = wl.activations(M, K, 1001, device="cuda")
    w = wl.weights((N, K), 2000 + N, device="cuda")
    qa_d, sa_d = lib.fp8_quant_1x128(x)
    qb_d, sb_d = lib.fp8_quant_128x128(w)
    try:
        lib.debug_set(3, pair)   # 1: the CTA-pair kernel
        c = lib.fp8_gemm_dense(qa_d, sa_d, qb_d, sb_d)
        torch.cuda.synchronize()
    finally:
        lib.debug_set(3, 0)
    rng = np.random.default_rng(N)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, 62, replace=False)]))
    nblocks = np.unique(np.concatenate([[0, (N - 1) // 128], rng.choice((N + 127) // 128, 2, replace=False)]))
    # oracle operands from the generator's values only
    qa, sa = quant.quant_1x128(to_np32(x[rows]))
    for nb in nblocks:
        cols = slice(nb * 128, min(N, nb * 128 + 128))
        qb, sb = quant.quant_128x128(to_np32(w[cols]))
        cref = gemm.gemm_dense(qa, sa, qb, sb)
        compare_gemm(c[rows][:, cols], cref, True)


# ---------------------------------------------------------------- grouped contiguous
def _contig_case(fg, counts, N, K, seed, sentinel=True):
    lay = wl.contig_layout(counts)
    E = len(counts)
    x = wl.activations(lay.m_total, K, seed, device="cpu")
    wl.zero_rows_beyond(x.view(1, lay.m_total, K), [lay.m_total], lay.m_total)
    x[torch.from_numpy(lay.m_indices < 0)] = 0  # padding rows are zero
    w = wl.weights((E, N, K), seed + 1, device="cpu")
    qa, sa, qa_d, sa_d = _quant_a(x)
    qb, sb, qb_d, sb_d = _quant_b(w)
    mi = dev(lay.m_indices)
    c = torch.full((lay.m_total, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fg.fp8_gemm_grouped_contig_out(qa_d, sa_d, qb_d, sb_d, mi, c)
    torch.cuda.synchronize()
    cref = gemm.gemm_grouped_contig(qa, sa, qb, sb, lay.m_indices)
    real = lay.m_indices >= 0
    compare_gemm(c[torch.from_numpy(real).cuda()], cref[real], True)
    if sentinel:
        assert torch.isnan(c[torch.from_numpy(~real).cuda()]).all(), "padding rows were written"


def test_contig_small(lib):
    _contig_case(lib, np.array([130, 0, 61, 256, 1]), 264, 384, 41)


def test_contig_zipf_counts(lib):
    counts = wl.zipf_counts(2000, 8, 1.1, seed=42)
    _contig_case(lib, counts, 256, 512, 43)


@pytest.mark.slow
@pytest.mark.parametrize("case", range(len(wl.CONTIG_CASES)))
def test_contig_full_sampled(lib, case):
    E, tokens, N, K = wl.CONTIG_CASES[case]
    counts = wl.zipf_counts(tokens, E, 1.1, seed=1004)
    lay = wl.contig_layout(counts)
    x = wl.activations(lay.m_total, K, 1005 + 10 * case, device="cuda")
    x[torch.from_numpy(lay.m_indices < 0).cuda()] = 0
    w = wl.weights((E, N, K), 1006 + 10 * case, device="cuda")
    qa_d, sa_d = lib.fp8_quant_1x128(x)
    qb_d, sb_d = lib.fp8_quant_128x128(w)
    c = torch.full((lay.m_total, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lib.fp8_gemm_grouped_contig_out(qa_d, sa_d, qb_d, sb_d, dev(lay.m_indices), c)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5 + case)
    real_rows = np.flatnonzero(lay.m_indices >= 0)
    rows = np.sort(rng.choice(real_rows, 48, replace=False))
    qa, sa = quant.quant_1x128(to_np32(x[rows]))
    for nb in (0, 17, N // 128 - 1):
        cols = slice(nb * 128, nb * 128 + 128)
        for e in np.unique(lay.m_indices[rows]):
            sel = lay.m_indices[rows] == e
            qb, sb = quant.quant_128x128(to_np32(w[e, cols]))
            cref = gemm.gemm_dense(qa[sel], sa[:, sel], qb, sb)
            compare_gemm(c[rows[sel]][:, cols], cref, True)
    pad = np.flatnonzero(lay.m_indices < 0)
    assert torch.isnan(c[torch.from_numpy(pad).cuda()]).all()


# ---------------------------------------------------------------- grouped masked
def _masked_case(fg, E, Mmax, N, K, masked, seed):
    x = wl.activations(E * Mmax, K, seed, device="cpu").view(E, Mmax, K)
    wl.zero_rows_beyond(x, masked, Mmax)
    w = wl.weights((E, N, K), seed + 1, device="cpu")
    qas, sas = zip(*[quant.quant_1x128(to_np32(x[e])) for e in range(E)])
    qa = np.stack(qas)
    sa = np.stack(sas)
    sa_pad = np.stack([pad_rows_scale(s, Mmax) for s in sas])
    qb, sb = quant.quant_128x128(to_np32(w))
    c = torch.full((E, Mmax, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fg.fp8_gemm_grouped_masked_out(dev(qa), dev(sa_pad), dev(qb), dev(sb),
                                   torch.tensor(masked, dtype=torch.int32, device="cuda"), c)
    torch.cuda.synchronize()
    cref = gemm.gemm_grouped_masked(qa, sa, qb, sb, masked)
    for e in range(E):
        m = int(masked[e])
        if m:
            compare_gemm(c[e, :m], cref[e, :m], True)
        assert torch.isnan(c[e, m:]).all(), f"expert {e}: rows beyond masked_m written"


def test_masked_small(lib):
    _masked_case(lib, 4, 256, 264, 384, np.array([0, 256, 17, 129], np.int32), 51)


def test_masked_sparse_experts(lib):
    # the active tiles are enumerated on the device across all experts: most
    # experts empty, one row, a partial and a full expert, the last one last
    masked = np.zeros(40, np.int32)
    masked[3], masked[17], masked[39] = 1, 200, 256
    _masked_case(lib, 40, 256, 264, 256, masked, 57)


def test_masked_decode_like(lib):
    masked = wl.masked_counts(6, 256, seed=52)
    _masked_case(lib, 6, 256, 512, 1024, masked, 53)


@pytest.mark.parametrize("E,T,N,C,masked", [
    (3, 384, 136, 264, (0, 100, 384)),
    # 256 tiles: CTAs run an empty expert's tile and then a real one, so an
    # empty tile's epilogue overlaps the next tile's operand loads
    (4, 256, 1024, 2048, (0, 256, 100, 0)),
])
def test_masked_k_wgrad(lib, E, T, N, C, masked):
    # per expert dW_e[N, C] = G_e^T X_e over the expert's tokens (K = tokens)
    masked = np.array(masked, np.int32)
    qg, sg, qx, sx = [], [], [], []
    for e in range(E):
        a, b, c_, d = _wgrad_operands(T, N, C, 60 + e, valid=masked[e])
        qg.append(a); sg.append(pad_rows_scale(b, N)); qx.append(c_); sx.append(pad_rows_scale(d, C))
    out = torch.randn((E, N, C), dtype=torch.float32, device="cuda")
    lib.fp8_gemm_grouped_masked_out(dev(np.stack(qg)), dev(np.stack(sg)), dev(np.stack(qx)), dev(np.stack(sx)),
                                    torch.tensor(masked, device="cuda"), out, b_scale_kind=lib.SCALE_ROW,
                                    mask_dim=lib.MASK_K)
    torch.cuda.synchronize()
    for e in range(E):
        ref = gemm.wgrad(qg[e], sg[e][:, :N], qx[e], sx[e][:, :C])
        if masked[e] == 0:
            assert torch.count_nonzero(out[e]) == 0
        else:
            compare_gemm(out[e], ref, False)


@pytest.mark.slow
def test_masked_full_decode_sampled(lib):
    E, Mmax, N, K = wl.MASKED_CASE
    masked = wl.masked_counts(E, Mmax, seed=1007)
    masked[0] = 0
    masked[1] = Mmax
    x = wl.activations(E * Mmax, K, 1008, device="cuda").view(E, Mmax, K)
    wl.zero_rows_beyond(x, masked, Mmax)
    w = wl.weights((E, N, K), 1009, device="cuda")
    qa_d = torch.empty((E, Mmax, K), dtype=torch.uint8, device="cuda")
    sa_d = torch.empty((E, K // 128, ld4(Mmax)), dtype=torch.float32, device="cuda")
    for e in range(E):
        lib.fp8_quant_1x128_out(x[e], qa_d[e], sa_d[e])
    qb_d, sb_d = lib.fp8_quant_128x128(w)
    c = torch.full((E, Mmax, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    mm = torch.tensor(masked, dtype=torch.int32, device="cuda")
    lib.fp8_gemm_grouped_masked_out(qa_d, sa_d, qb_d, sb_d, mm, c, expected_m=128)
    torch.cuda.synchronize()
    for e in (1, 5, 15):
        m = int(masked[e])
        qa, sa = quant.quant_1x128(to_np32(x[e, :m]))
        for nb in (0, 31):
            cols = slice(nb * 128, nb * 128 + 128)
            qb, sb = quant.quant_128x128(to_np32(w[e, cols]))
            compare_gemm(c[e, :m, cols], gemm.gemm_dense(qa, sa, qb, sb), True)
    for e in range(E):
        assert torch.isnan(c[e, int(masked[e]):]).all()


# ---------------------------------------------------------------- weight gradients at full size
@pytest.mark.slow
def test_wgrad_masked_moe_full_config(lib):
    # The MoE weight gradient end to end at its full size: 16 experts of at
    # most 256 tokens, dW_e[4096, 7168] = G_e^T X_e in FP32. X is cached as
    # 1x128 E4M3 and retiled to 128x1 with power-of-2 scales; the activation
    # gradient G (BF16) goes straight to 128x1 pow2 tiles. One expert has no
    # tokens and one a full 256.
    E, Tmax, N, C = wl.MASKED_CASE
    counts = wl.masked_counts(E, Tmax, seed=1011)
    counts[2], counts[7] = 0, Tmax
    g = wl.normal((E, Tmax, N), 1012, device="cuda", dtype=torch.bfloat16)
    x = wl.activations(E * Tmax, C, 1013, device="cuda").view(E, Tmax, C)
    wl.zero_rows_beyond(g, counts, Tmax)
    wl.zero_rows_beyond(x, counts, Tmax)
    vr = torch.as_tensor(counts, device="cuda")
    qx = torch.empty((E, Tmax, C), dtype=torch.uint8, device="cuda")
    sx = torch.empty((E, C // 128, ld4(Tmax)), dtype=torch.float32, device="cuda")
    for e in range(E):
        lib.fp8_quant_1x128_out(x[e], qx[e], sx[e])
    qxT, sxT = lib.fp8_requant_128x1(qx.view(torch.float8_e4m3fn), sx, vr, pow2=True)
    qgT, sgT = lib.fp8_requant_128x1(g, None, vr, pow2=True)
    dw = torch.full((E, N, C), float("nan"), dtype=torch.float32, device="cuda")
    lib.fp8_gemm_grouped_masked_out(qgT, sgT, qxT, sxT, vr, dw, b_scale_kind=lib.SCALE_ROW,
                                    mask_dim=lib.MASK_K, expected_m=Tmax)
    lib.check()
    assert torch.count_nonzero(dw[2]) == 0, "an expert without tokens must get dW = 0"
    rng = np.random.default_rng(11)
    for e in (1, 7, 13):
        m = int(counts[e])
        # oracle operands from the generator's values only
        q_o, s_o = quant.quant_1x128(to_np32(x[e]))
        qxT_o, sxT_o = quant.requant_128x1(q_o, s_o, m, True)
        qgT_o, sgT_o = quant.requant_128x1(to_np32(g[e]), None, m, True)
        assert np.array_equal(qxT[e].cpu().numpy(), qxT_o), f"expert {e}: requantized X differs"
        assert np.array_equal(qgT[e].cpu().numpy(), qgT_o), f"expert {e}: requantized G differs"
        for nb, cb in [(0, 0), (N // 128 - 1, C // 128 - 1)] + [tuple(rng.integers(0, (N // 128, C // 128)))
                                                                  for _ in range(3)]:
            rows = np.arange(nb * 128, nb * 128 + 128)
            cols = np.arange(cb * 128, cb * 128 + 128)
            ref = gemm.wgrad(qgT_o, sgT_o, qxT_o, sxT_o, rows=rows, cols=cols)
            compare_gemm(dw[e, nb * 128:nb * 128 + 128, cb * 128:cb * 128 + 128], ref, False)


@pytest.mark.parametrize("T", [512])
def test_dense_wgrad_many_tiles_accumulate(lib, T):
    # Row-scaled B with FP32 output added into a nonzero C: 32 x 28 output
    # tiles on the SMs, so every CTA runs several tiles (TMEM buffer and
    # ring phases flip across tiles, TMA reduce-add epilogue under load).
    N, C = 4096, 7168
    qgT, sgT, qxT, sxT = _wgrad_operands(T, N, C, 85)
    base = wl.normal((N, C), 86, device="cuda")
    out = base.clone()
    lib.fp8_gemm_dense_out(dev(qgT), dev(pad_rows_scale(sgT, N)), dev(qxT), dev(pad_rows_scale(sxT, C)), out,
                           b_scale_kind=lib.SCALE_ROW, accumulate=True)
    lib.check()
    ref = gemm.wgrad(qgT, sgT, qxT, sxT) + base.double().cpu().numpy()
    compare_gemm(out, ref, False)


@pytest.mark.slow
def test_dense_wgrad_prefill_tokens_accumulate_sampled(lib):
    # Dense weight gradient over the 4096 prefill tokens, added into FP32
    # dW (gradient accumulation): dW[4096, 7168] += G^T X, sampled blocks.
    T, N, C = 4096, 4096, 7168
    g = wl.normal((T, N), 1021, device="cuda", dtype=torch.bfloat16)
    x = wl.activations(T, C, 1022, device="cuda")
    qx, sx = lib.fp8_quant_1x128(x)
    qxT, sxT = lib.fp8_requant_128x1(qx.view(torch.float8_e4m3fn), sx, pow2=True)
    qgT, sgT = lib.fp8_requant_128x1(g, pow2=True)
    base = wl.normal((N, C), 1023, device="cuda")
    out = base.clone()
    lib.fp8_gemm_dense_out(qgT, sgT, qxT, sxT, out, b_scale_kind=lib.SCALE_ROW, accumulate=True)
    lib.check()
    rng = np.random.default_rng(12)
    for nb, cb in [(0, 0), (N // 128 - 1, C // 128 - 1), tuple(rng.integers(0, (N // 128, C // 128)))]:
        rows = slice(nb * 128, nb * 128 + 128)
        cols = slice(cb * 128, cb * 128 + 128)
        # a 128x128 block of dW needs only its 128 channels of G and of X
        # (one 1x128 group of X, 128x1 tiles down the tokens)
        q_o, s_o = quant.quant_1x128(to_np32(x[:, cols]))
        qxT_o, sxT_o = quant.requant_128x1(q_o, s_o, None, True)
        qgT_o, sgT_o = quant.requant_128x1(to_np32(g[:, rows]), None, None, True)
        ref = gemm.wgrad(qgT_o, sgT_o, qxT_o, sxT_o) + base[rows, cols].double().cpu().numpy()
        compare_gemm(out[rows, cols], ref, False)


# ---------------------------------------------------------------- bounded waits
def test_timeout_reports_error_and_context_survives(lib):
    M, N, K = 128, 256, 512
    x = wl.activations(M, K, 71, device="cpu")
    w = wl.weights((N, K), 72, device="cpu")
    qa, sa, qa_d, sa_d = _quant_a(x)
    qb, sb, qb_d, sb_d = _quant_b(w)
    lib.check()
    try:
        lib.debug_set(1, 50_000_000)   # 50 ms wait limit
        lib.debug_set(2, 1)            # the second pipeline fill is never issued
        lib.fp8_gemm_dense(qa_d, sa_d, qb_d, sb_d)
        with pytest.raises(lib.Fp8fgError) as ei:
            lib.check()
        assert ei.value.code == lib.ERR_TIMEOUT
    finally:
        lib.debug_set(2, -1)
        lib.debug_set(1, 0)
    c = lib.fp8_gemm_dense(qa_d, sa_d, qb_d, sb_d)
    lib.check()
    compare_gemm(c, gemm.gemm_dense(qa, sa, qb, sb), True)


# ---------------------------------------------------------------- CTA pairs (large dense problems)
# Debug key 3 sends dense problems whose 128 x 256 tiles outnumber half the
# SMs to the CTA-pair kernel (tcgen05 cta_group::2, 256 x 256 tiles); it is
# off by default. Both kernels are checked on the same shapes.
PAIR_SHAPES = [
    (1000, 2600, 1024, torch.bfloat16),   # ragged: the last pair tile's peer rows and B half partly out of range
    (2048, 2560, 2048, torch.float32),
    (512, 7168, 512, torch.bfloat16),
]


@pytest.mark.parametrize("pair", [1, 0])
@pytest.mark.parametrize("M,N,K,out_dtype", PAIR_SHAPES)
def test_pair_and_single_cta_kernels_match_oracle(lib, M, N, K, out_dtype, pair):
    assert -(-M // 128) * -(-N // 256) * 2 > 148  # large enough for the pair kernel on 148 SMs
    try:
        lib.debug_set(3, pair)
        _dense_case(lib, M, N, K, seed=M + N + K, out_dtype=out_dtype)
    finally:
        lib.debug_set(3, 0)


def test_pair_kernel_row_scaled_accumulate(lib):
    # the weight-gradient form on CTA pairs: per-row B scales, FP32 C +=
    T, N, C = 384, 1024, 2560
    qgT, sgT, qxT, sxT = _wgrad_operands(T, N, C, 87)
    base = wl.normal((N, C), 88, device="cuda")
    out = base.clone()
    try:
        lib.debug_set(3, 1)
        lib.fp8_gemm_dense_out(dev(qgT), dev(pad_rows_scale(sgT, N)), dev(qxT), dev(pad_rows_scale(sxT, C)), out,
                               b_scale_kind=lib.SCALE_ROW, accumulate=True)
        lib.check()
    finally:
        lib.debug_set(3, 0)
    compare_gemm(out, gemm.wgrad(qgT, sgT, qxT, sxT) + base.double().cpu().numpy(), False)


def test_pair_kernel_timeout_reports_error_and_context_survives(lib):
    M, N, K = 1024, 4096, 512
    x = wl.activations(M, K, 73, device="cpu")
    w = wl.weights((N, K), 74, device="cpu")
    qa, sa, qa_d, sa_d = _quant_a(x)
    qb, sb, qb_d, sb_d = _quant_b(w)
    lib.check()
    try:
        lib.debug_set(3, 1)
        lib.debug_set(1, 50_000_000)   # 50 ms wait limit
        lib.debug_set(2, 1)            # every CTA's second pipeline fill is never issued
        lib.fp8_gemm_dense(qa_d, sa_d, qb_d, sb_d)
        with pytest.raises(lib.Fp8fgError) as ei:
            lib.check()
        assert ei.value.code == lib.ERR_TIMEOUT
        lib.debug_set(2, -1)
        lib.debug_set(1, 0)
        c = lib.fp8_gemm_dense(qa_d, sa_d, qb_d, sb_d)
        lib.check()
    finally:
        lib.debug_set(2, -1)
        lib.debug_set(1, 0)
        lib.debug_set(3, 0)
    compare_gemm(c, gemm.gemm_dense(qa, sa, qb, sb), True)


# ---------------------------------------------------------------- split-K (decode-sized M)
# Decode-sized problems (128 x 128 tiles at most half the SMs) split K in
# one of two ways, chosen by the split policy: Stream-K over the caller's
# workspace, or the cluster split (the CTAs of a cluster share a tile and
# sum their partials through distributed shared memory). Each split test
# runs under both.
SPLITS = pytest.mark.parametrize("policy", ["stream", "cluster"])


@contextlib.contextmanager
def split_policy(fg, policy):
    fg.set_split_policy({"auto": fg.SPLIT_AUTO, "stream": fg.SPLIT_STREAM, "cluster": fg.SPLIT_CLUSTER}[policy])
    try:
        yield
    finally:
        fg.set_split_policy(fg.SPLIT_AUTO)


def _split_case(fg, M, N, K, seed, out_dtype=torch.bfloat16, accumulate=False, policy="auto"):
    x = wl.activations(M, K, seed, device="cpu")
    w = wl.weights((N, K), seed + 1, device="cpu")
    qa, sa, qa_d, sa_d = _quant_a(x)
    qb, sb, qb_d, sb_d = _quant_b(w)
    ws = fg.gemm_workspace(M, N, K)
    assert ws is not None, "expected a K-split for this shape"
    cref = gemm.gemm_dense(qa, sa, qb, sb)
    base = torch.randn((M, N), dtype=torch.float32, device="cuda") if accumulate else None
    outs = []
    with split_policy(fg, policy):
        for _ in range(2):  # the workspace counters must come back to zero
            c = base.clone() if accumulate else torch.empty((M, N), dtype=out_dtype, device="cuda")
            fg.fp8_gemm_dense_out(qa_d, sa_d, qb_d, sb_d, c, accumulate=accumulate, workspace=ws)
            torch.cuda.synchronize()
            ref = cref + base.double().cpu().numpy() if accumulate else cref
            compare_gemm(c, ref, out_dtype == torch.bfloat16)
            outs.append(c)
    # partial sums are added in a fixed order whichever CTA finishes first
    assert torch.equal(outs[0], outs[1]), "split result is not deterministic"
    return ws


@SPLITS
@pytest.mark.parametrize("M,N,K", [(1, 256, 2048), (64, 512, 4096), (130, 264, 2048), (128, 1024, 7168)])
def test_split_k_matches_oracle(lib, M, N, K, policy):
    _split_case(lib, M, N, K, seed=M + N, policy=policy)


@SPLITS
def test_split_k_fp32_accumulate(lib, policy):
    _split_case(lib, 64, 520, 2048, seed=81, out_dtype=torch.float32, accumulate=True, policy=policy)


# Cluster split sizes: S = min(8, SMs // tiles, K blocks // 4), lowered
# until every tile's cluster is resident at once. On 148 SMs these shapes
# ask for S = 8 (one tile), 4, 3, 5, 6 and 7, then 2 with a ragged last
# column tile (N = 3144 and 6344: the last tile has 72 columns), once with
# a second row tile of 2 rows (M = 130). S that does not divide the 16
# column chunks of a tile gives CTAs unequal shares (S = 3: 5, 5, 6).
@pytest.mark.parametrize("M,N,K", [(64, 128, 4096), (64, 3072, 2048), (64, 5760, 2048), (32, 3712, 2560),
                                   (64, 3072, 3072), (16, 2688, 3584), (130, 3144, 1024), (64, 6344, 1024)])
def test_cluster_split_sizes(lib, M, N, K):
    _split_case(lib, M, N, K, seed=M + N + K, policy="cluster")


def test_cluster_split_fp32_accumulate_ragged(lib):
    _split_case(lib, 130, 264, 4096, seed=85, out_dtype=torch.float32, accumulate=True, policy="cluster")


@SPLITS
def test_split_k_small_workspace_falls_back(lib, policy):
    # a workspace too small for Stream-K: the GEMM runs unsplit (Stream-K
    # policy) or on the cluster split, and the workspace is never written
    M, N, K = 64, 512, 2048
    x = wl.activations(M, K, 82, device="cpu")
    w = wl.weights((N, K), 83, device="cpu")
    qa, sa, qa_d, sa_d = _quant_a(x)
    qb, sb, qb_d, sb_d = _quant_b(w)
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with split_policy(lib, policy):
        lib.fp8_gemm_dense_out(qa_d, sa_d, qb_d, sb_d, c, workspace=small)
    compare_gemm(c, gemm.gemm_dense(qa, sa, qb, sb), True)
    assert torch.count_nonzero(small) == 0


@SPLITS
def test_split_k_wgrad_row_scales(lib, policy):
    # weight gradient with many tokens and a small output: K (tokens) is split
    T, N, C = 2048, 136, 264
    qgT, sgT, qxT, sxT = _wgrad_operands(T, N, C, 84)
    ws = lib.gemm_workspace(N, C, T)
    assert ws is not None
    outs = []
    with split_policy(lib, policy):
        for _ in range(2):
            out = torch.empty((N, C), dtype=torch.float32, device="cuda")
            lib.fp8_gemm_dense_out(dev(qgT), dev(pad_rows_scale(sgT, N)), dev(qxT), dev(pad_rows_scale(sxT, C)), out,
                                   b_scale_kind=lib.SCALE_ROW, workspace=ws)
            compare_gemm(out, gemm.wgrad(qgT, sgT, qxT, sxT), False)
            outs.append(out)
    assert torch.equal(outs[0], outs[1])


@pytest.mark.slow
@SPLITS
@pytest.mark.parametrize("M,N,K", wl.DECODE_CASES)
def test_decode_full_sampled(lib, M, N, K, policy):
    x = wl.activations(M, K, 1003, device="cuda")
    w = wl.weights((N, K), 1004 + N, device="cuda")
    qa_d, sa_d = lib.fp8_quant_1x128(x)
    qb_d, sb_d = lib.fp8_quant_128x128(w)
    with split_policy(lib, policy):
        c = lib.fp8_gemm_dense(qa_d, sa_d, qb_d, sb_d)
        torch.cuda.synchronize()
    qa, sa = quant.quant_1x128(to_np32(x))
    for nb in (0, 13, N // 128 - 1):
        cols = slice(nb * 128, nb * 128 + 128)
        qb, sb = quant.quant_128x128(to_np32(w[cols]))
        compare_gemm(c[:, cols], gemm.gemm_dense(qa, sa, qb, sb), True)


# ---------------------------------------------------------------- Stream-K segments
# Decode-sized problems split every tile along K over the SMs: CTA c takes
# K blocks [c*U, (c+1)*U) of the tile-major sequence, so when U does not
# divide the tile's K blocks a CTA's range straddles two tiles and a tile's
# pieces come from several CTAs; the last piece to arrive sums them in
# order. On 148 SMs, M=64, N=1792, K=6912 gives 7 tiles of 54 K blocks,
# U = 5.
def _sk_case(fg, M, N, K, seed, out_dtype=torch.bfloat16, accumulate=False, rows=None, policy="stream"):
    x = wl.activations(M, K, seed, device="cpu")
    w = wl.weights((N, K), seed + 1, device="cpu")
    qa, sa, qa_d, sa_d = _quant_a(x)
    qb, sb, qb_d, sb_d = _quant_b(w)
    ws = fg.gemm_workspace(M, N, K)
    if ws is None:
        pytest.skip("this GPU's SM count fills the last wave: no Stream-K split")
    sel = np.arange(M) if rows is None else np.asarray(rows)
    cref = gemm.gemm_dense(qa, sa, qb, sb, rows=sel)
    base = torch.randn((M, N), dtype=torch.float32, device="cuda") if accumulate else None
    outs = []
    with split_policy(fg, policy):
        for _ in range(2):  # the arrival counters must come back to zero
            c = base.clone() if accumulate else torch.empty((M, N), dtype=out_dtype, device="cuda")
            fg.fp8_gemm_dense_out(qa_d, sa_d, qb_d, sb_d, c, accumulate=accumulate, workspace=ws)
            torch.cuda.synchronize()
            ref = cref + base.double().cpu().numpy()[sel] if accumulate else cref
            compare_gemm(c[torch.as_tensor(sel, device="cuda")], ref, out_dtype == torch.bfloat16)
            outs.append(c)
    assert torch.equal(outs[0], outs[1]), "split result is not deterministic"
    # the unsplit product (Stream-K policy, no workspace) agrees within the same tolerance
    c = base.clone() if accumulate else torch.empty((M, N), dtype=out_dtype, device="cuda")
    with split_policy(fg, "stream"):
        fg.fp8_gemm_dense_out(qa_d, sa_d, qb_d, sb_d, c, accumulate=accumulate, workspace=None)
    torch.cuda.synchronize()
    compare_gemm(c[torch.as_tensor(sel, device="cuda")], ref, out_dtype == torch.bfloat16)


def test_stream_k_segments_straddle_tiles(lib):
    _sk_case(lib, 64, 1792, 6912, seed=91)


def test_stream_k_straddle_fp32_accumulate(lib):
    _sk_case(lib, 64, 1792, 6912, seed=93, out_dtype=torch.float32, accumulate=True)
