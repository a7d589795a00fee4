"""Pins for the oracle's FP64 GEMM references (CPU only).

Brute force with exact rationals on tiny inputs, an exact integer special
case against numpy's integer matmul, an identity special case, and the
grouped layouts against per-expert dense products.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import e4m3, gemm, quant


def _codes(rng, shape, lo=0, hi=0x7F):
    c = rng.integers(lo, hi, size=shape).astype(np.uint8)
    c |= (rng.random(shape) < 0.5).astype(np.uint8) << 7
    return c


def _pow2_scales(rng, shape, lo=-6, hi=6):
    return np.exp2(rng.integers(lo, hi, size=shape)).astype(np.float32)


def _rand_scales(rng, shape):
    return (rng.random(shape) * 3 + 0.01).astype(np.float32)


def _exact(qa, sa, qb, sb, m, n, b_kind):
    tot = Fraction(0)
    K = qa.shape[1]
    for k in range(K):
        a = Fraction(float(e4m3.decode(qa[m, k]))) * Fraction(float(sa[k // 128, m]))
        if b_kind == "block":
            sbv = sb[n // 128, k // 128]
        else:
            sbv = sb[k // 128, n]
        b = Fraction(float(e4m3.decode(qb[n, k]))) * Fraction(float(sbv))
        tot += a * b
    return tot


@pytest.mark.parametrize("b_kind", ["block", "row"])
def test_dense_matches_exact_rationals(b_kind):
    rng = np.random.default_rng(21)
    M, N, K = 5, 260, 384
    qa = _codes(rng, (M, K))
    qb = _codes(rng, (N, K))
    sa = _rand_scales(rng, (K // 128, M))
    sb = _rand_scales(rng, (3, K // 128)) if b_kind == "block" else _rand_scales(rng, (K // 128, N))
    c = gemm.gemm_dense(qa, sa, qb, sb, b_kind)
    for m, n in [(0, 0), (4, 259), (2, 130), (3, 127), (1, 128), (0, 255)]:
        ex = _exact(qa, sa, qb, sb, m, n, b_kind)
        assert abs(Fraction(c[m, n]) - ex) <= abs(ex) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 80)


def test_dense_integer_case_is_exact_integer_matmul():
    rng = np.random.default_rng(22)
    # E4M3 represents every integer in [-16, 16] exactly
    ints_a = rng.integers(-16, 17, size=(64, 256))
    ints_b = rng.integers(-16, 17, size=(96, 256))
    qa = e4m3.encode(ints_a.astype(np.float32))
    qb = e4m3.encode(ints_b.astype(np.float32))
    assert np.array_equal(e4m3.decode(qa), ints_a)
    c = gemm.gemm_dense(qa, np.ones((2, 64), np.float32), qb, np.ones((1, 2), np.float32))
    assert np.array_equal(c, (ints_a @ ints_b.T).astype(np.float64))


def test_dense_identity_b_returns_dequantized_a():
    rng = np.random.default_rng(23)
    K = 256
    qa = _codes(rng, (7, K))
    sa = _rand_scales(rng, (2, 7))
    qb = np.zeros((K, K), np.uint8)
    np.fill_diagonal(qb, 0x38)  # 1.0
    c = gemm.gemm_dense(qa, sa, qb, np.ones((2, 2), np.float32))
    ahat = e4m3.decode(qa) * np.repeat(sa.T.astype(np.float64), 128, axis=1)
    assert np.array_equal(np.nan_to_num(c), np.nan_to_num(ahat))


def test_block_scale_indexing_with_distinct_powers():
    # sB[nb, kb] = 2^(nb + 4 kb): a swapped index changes every entry
    rng = np.random.default_rng(24)
    qa = _codes(rng, (3, 256), 0x30, 0x48)
    qb = _codes(rng, (256, 256), 0x30, 0x48)
    sa = np.ones((2, 3), np.float32)
    sb = np.array([[1, 16], [2, 32]], np.float32)
    c = gemm.gemm_dense(qa, sa, qb, sb)
    a = e4m3.decode(qa)
    b = e4m3.decode(qb)
    for n in (0, 200):
        nb = n // 128
        ref = a[:, :128] @ b[n, :128] * sb[nb, 0] + a[:, 128:] @ b[n, 128:] * sb[nb, 1]
        assert np.array_equal(c[:, n], ref)


def test_sampled_rows_cols_equal_full():
    rng = np.random.default_rng(25)
    qa, qb = _codes(rng, (40, 256)), _codes(rng, (300, 256))
    sa, sb = _rand_scales(rng, (2, 40)), _rand_scales(rng, (3, 2))
    full = gemm.gemm_dense(qa, sa, qb, sb)
    rows, cols = np.array([3, 39, 0]), np.array([299, 5, 128])
    part = gemm.gemm_dense(qa, sa, qb, sb, rows=rows, cols=cols)
    assert np.allclose(part, full[np.ix_(rows, cols)], rtol=1e-12, atol=0)


def test_grouped_contig_equals_per_expert_dense():
    rng = np.random.default_rng(26)
    E, N, K = 3, 136, 256
    counts = [130, 0, 61]
    padded = [256, 0, 128]
    m_idx = np.concatenate([np.r_[np.zeros(130), -np.ones(126)], np.r_[np.full(61, 2), -np.ones(67)]]).astype(np.int32)
    Mt = sum(padded)
    qa = _codes(rng, (Mt, K))
    sa = _rand_scales(rng, (2, Mt))
    qb = _codes(rng, (E, N, K))
    sb = _rand_scales(rng, (E, 2, 2))
    c = gemm.gemm_grouped_contig(qa, sa, qb, sb, m_idx)
    assert np.all(np.isnan(c[m_idx < 0]))
    ref0 = gemm.gemm_dense(qa[:130], sa[:, :130], qb[0], sb[0])
    ref2 = gemm.gemm_dense(qa[256:317], sa[:, 256:317], qb[2], sb[2])
    assert np.array_equal(c[:130], ref0)
    assert np.array_equal(c[256:317], ref2)
    assert counts[1] == 0


def test_grouped_masked_equals_per_expert_dense():
    rng = np.random.default_rng(27)
    E, Mmax, N, K = 3, 256, 64, 128
    masked = np.array([0, 256, 17], np.int32)
    qa = _codes(rng, (E, Mmax, K))
    sa = _rand_scales(rng, (E, 1, Mmax))
    qb = _codes(rng, (E, N, K))
    sb = _rand_scales(rng, (E, 1, 1))
    c = gemm.gemm_grouped_masked(qa, sa, qb, sb, masked)
    assert np.all(np.isnan(c[0])) and np.all(np.isnan(c[2, 17:]))
    assert np.array_equal(c[1], gemm.gemm_dense(qa[1], sa[1], qb[1], sb[1]))
    assert np.array_equal(c[2, :17], gemm.gemm_dense(qa[2, :17], sa[2][:, :17], qb[2], sb[2]))


def test_wgrad_is_gt_x_of_dequantized_activations():
    rng = np.random.default_rng(28)
    T, N, C = 256, 8, 130
    g = rng.standard_normal((T, N)).astype(np.float32)
    x = rng.standard_normal((T, C)).astype(np.float32)
    qgT, sgT = quant.requant_128x1(g, None, None, True)
    qxT, sxT = quant.requant_128x1(x, None, None, True)
    dw = gemm.wgrad(qgT, sgT, qxT, sxT)
    assert dw.shape == (N, C)
    for n, cc in [(0, 0), (7, 129), (3, 64)]:
        ex = _exact(qgT, sgT, qxT, sxT, n, cc, "row")
        assert abs(Fraction(dw[n, cc]) - ex) <= abs(ex) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 80)
    # and it approximates G^T X itself (quantization error only)
    rel = np.linalg.norm(dw - g.T.astype(np.float64) @ x) / np.linalg.norm(g.T.astype(np.float64) @ x)
    assert rel < 0.1


def test_tolerance_helpers():
    ref = np.array([1.0, -2.0, 0.0, 4.0])
    assert gemm.frobenius_rel(ref, ref) == 0.0
    ok = gemm.elementwise_ok(ref + np.array([0.0, 0.02, 0.02, 0.0]), ref)
    assert ok.tolist() == [True, True, True, True]
    ok = gemm.elementwise_ok(ref + np.array([0.1, 0.0, 0.0, 0.0]), ref)
    assert ok.tolist() == [False, True, True, True]


# ---------------------------------------------------------------- Dgrad
def test_dgrad_matches_exact_rationals():
    # dX[m, k] = sum_n dYhat[m, n] What[n, k] with W's block scales indexed
    # [n // 128, k // 128] (the forward weight read as it is)
    rng = np.random.default_rng(31)
    M, N, K = 4, 384, 260
    qdy = _codes(rng, (M, N))
    qw = _codes(rng, (N, K))
    sdy = _rand_scales(rng, (N // 128, M))
    sw = _rand_scales(rng, (N // 128, 3))
    dx = gemm.dgrad(qdy, sdy, qw, sw)
    for m, k in [(0, 0), (3, 259), (1, 130), (2, 127), (0, 128)]:
        ex = Fraction(0)
        for n in range(N):
            a = Fraction(float(e4m3.decode(qdy[m, n]))) * Fraction(float(sdy[n // 128, m]))
            b = Fraction(float(e4m3.decode(qw[n, k]))) * Fraction(float(sw[n // 128, k // 128]))
            ex += a * b
        assert abs(Fraction(dx[m, k]) - ex) <= abs(ex) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 80)


def test_block_quantization_is_transpose_invariant_and_dgrad_is_dense_on_wt():
    # A 128x128 block has one amax whichever way it is read, so quantizing
    # W^T gives the transposed codes and scales; dgrad on W then equals the
    # dense product with B = W^T quantized on its own.
    rng = np.random.default_rng(32)
    N, K, M = 256, 384, 6
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qw, sw = quant.quant_128x128(w)
    qwT, swT = quant.quant_128x128(np.ascontiguousarray(w.T))
    assert np.array_equal(qwT, qw.T) and np.array_equal(swT, sw.T)
    dy = rng.standard_normal((M, N)).astype(np.float32)
    qdy, sdy = quant.quant_1x128(dy)
    np.testing.assert_allclose(gemm.dgrad(qdy, sdy, qw, sw), gemm.gemm_dense(qdy, sdy, qwT, swT), rtol=1e-12,
                               atol=1e-12)


def test_dgrad_block_scale_indexing_with_distinct_powers():
    # unit codes everywhere and a distinct power of two per weight block:
    # dX[m, k] = 128 * sum_j sw[j, k // 128], which a transposed or shifted
    # scale index would change
    N, K, M = 384, 256, 2
    one = e4m3.encode(np.ones(1))[0]
    qdy = np.full((M, N), one, np.uint8)
    qw = np.full((N, K), one, np.uint8)
    sdy = np.ones((N // 128, M), np.float32)
    sw = np.exp2(np.arange(6).reshape(3, 2) * 3).astype(np.float32)   # [N/128, K/128]
    dx = gemm.dgrad(qdy, sdy, qw, sw)
    for k in (0, 127, 128, 255):
        assert dx[0, k] == 128.0 * sw[:, k // 128].sum()
