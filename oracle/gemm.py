"""FP64 reference GEMMs on dequantized operands (test infrastructure).

The FP8 GEMMs take FP8 tensors with their fine-grained scales and produce
BF16 or FP32 (DeepSeek-V3 report excerpt, page 1, third paragraph); the
DeepGEMM article (page 4, key features) lists a dense layout and two MoE
layouts. The plain definition of what every variant computes is

    C[m, n] = sum_k  Ahat[m, k] * Bhat[n, k],
    Ahat[m, k] = decode(qA[m, k]) * sA[k // 128, m]
    Bhat[n, k] = decode(qB[n, k]) * sB[n // 128, k // 128]      (128x128 blocks)
              or decode(qB[n, k]) * sB[k // 128, n]             (128x1 / per-row)

i.e. the product of the dequantized operands. Per-block scaling, FP32
promotion and accumulation order are implementation choices with the same
exact result; the oracle evaluates it in float64 (each dequantized value is
exact in float64: a 4-bit significand times a 24-bit one).

Layouts:

* dense:              A[M,K], B[N,K]  -> C[M,N]
* grouped contiguous: A[Mt,K] rows sorted by expert, ``m_indices[row]`` the
  expert of each row or -1 for padding; B[E,N,K] -> C[Mt,N] (padding rows
  have no defined value)
* grouped masked:     A[E,Mmax,K], ``masked_m[e]`` valid rows per expert,
  B[E,N,K] -> C[E,Mmax,N] (rows >= masked_m[e] have no defined value)
* Wgrad:              dW[N,C] = sum_t G[t,n] X[t,c]; with both operands
  128x1-requantized and transposed it is the dense form with per-row scales
  on both sides.
* Dgrad:              dX[M,K] = dY[M,N] W[N,K], W the forward pass's
  128x128-quantized weight read as it is (no transposed copy).
"""
from __future__ import annotations

import numpy as np

from . import e4m3

TILE = 128


def dequant_rows(q, s) -> np.ndarray:
    """Per-row 1x128 (or 128x1 transposed) scales s[K/128, R] -> float64 [R, K]."""
    q = np.asarray(q)
    R, K = q.shape
    s = np.asarray(s, dtype=np.float64)[:, :R]            # [K/128, R]
    return e4m3.decode(q) * np.repeat(s.T, TILE, axis=1)


def dequant_blocks(q, s) -> np.ndarray:
    """128x128 block scales s[ceil(N/128), K/128] -> float64 [N, K]."""
    q = np.asarray(q)
    N, K = q.shape
    s = np.asarray(s, dtype=np.float64)
    full = np.repeat(np.repeat(s, TILE, axis=0), TILE, axis=1)[:N, :K]
    return e4m3.decode(q) * full


def dequant_b(q, s, b_kind: str) -> np.ndarray:
    if b_kind == "block":
        return dequant_blocks(q, s)
    if b_kind == "row":
        return dequant_rows(q, s)
    raise ValueError(b_kind)


def gemm_dense(qa, sa, qb, sb, b_kind: str = "block", rows=None, cols=None) -> np.ndarray:
    """C = Ahat @ Bhat^T in float64; optionally only for selected rows/cols."""
    qa = np.asarray(qa)
    qb = np.asarray(qb)
    a = dequant_rows(qa, sa)
    b = dequant_b(qb, sb, b_kind)
    if rows is not None:
        a = a[np.asarray(rows)]
    if cols is not None:
        b = b[np.asarray(cols)]
    return a @ b.T


def gemm_grouped_contig(qa, sa, qb, sb, m_indices, rows=None) -> np.ndarray:
    """Grouped contiguous layout; padding rows (m_indices == -1) come back as NaN."""
    qa = np.asarray(qa)
    m_idx = np.asarray(m_indices)
    Mt = qa.shape[0]
    E, N, _ = np.asarray(qb).shape
    rows = np.arange(Mt) if rows is None else np.asarray(rows)
    a = dequant_rows(qa, sa)[rows]
    out = np.full((len(rows), N), np.nan)
    for e in range(E):
        sel = m_idx[rows] == e
        if sel.any():
            b = dequant_blocks(qb[e], sb[e])
            out[sel] = a[sel] @ b.T
    return out


def gemm_grouped_masked(qa, sa, qb, sb, masked_m) -> np.ndarray:
    """Grouped masked layout; rows >= masked_m[e] come back as NaN.

    qa [E, Mmax, K], sa [E, K/128, Mmax], qb [E, N, K], sb [E, ceil(N/128), K/128].
    """
    qa = np.asarray(qa)
    E, Mmax, _ = qa.shape
    N = np.asarray(qb).shape[1]
    out = np.full((E, Mmax, N), np.nan)
    for e in range(E):
        m = int(masked_m[e])
        if m == 0:
            continue
        a = dequant_rows(qa[e], sa[e])[:m]
        b = dequant_blocks(qb[e], sb[e])
        out[e, :m] = a @ b.T
    return out


def wgrad(qgT, sgT, qxT, sxT, rows=None, cols=None) -> np.ndarray:
    """dW[N, C] = Ghat^T Xhat from 128x1-requantized, transposed operands.

    qgT [N, T] with sgT [T/128, N]; qxT [C, T] with sxT [T/128, C].
    """
    return gemm_dense(qgT, sgT, qxT, sxT, "row", rows=rows, cols=cols)


def dgrad(qdy, sdy, qw, sw, rows=None, cols=None) -> np.ndarray:
    """dX[M, K] = dYhat @ What: the data gradient of Y = X W^T.

    qdy [M, N] with 1x128 scales sdy [N/128, M] (quantized along N, the
    reduction); qw [N, K] with its 128x128 block scales sw [N/128, K/128],
    the forward pass's quantized weight, used as is (DeepSeek-V3 report
    excerpt, page 1, paragraph 3: Dgrad is one of the FP8 GEMMs).
    """
    a = dequant_rows(np.asarray(qdy), sdy)
    b = dequant_blocks(np.asarray(qw), sw)
    if rows is not None:
        a = a[np.asarray(rows)]
    if cols is not None:
        b = b[:, np.asarray(cols)]
    return a @ b


def frobenius_rel(c, ref) -> float:
    c = np.asarray(c, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(c - ref) / den) if den > 0 else float(np.linalg.norm(c))


def elementwise_ok(c, ref, rel: float = 1e-2, abs_rms: float = 1e-2) -> np.ndarray:
    """Per-element bound |C - Cref| <= rel*|Cref| + abs_rms*rms(Cref)."""
    c = np.asarray(c, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    return np.abs(c - ref) <= rel * np.abs(ref) + abs_rms * rms
