"""Shared helpers for the GPU parity tests.

Inputs come from the seeded generators in ``workloads``; expected values come
from ``oracle`` only (never from the CUDA path). Scale arrays are moved
between the oracle's logical layout and the library's padded row stride.

GEMM tolerance: against the
oracle's FP64 product Cref of the same dequantized operands,
  * relative Frobenius error <= 1e-3, measured against Cref rounded to the
    output type (BF16 output is compared with the oracle's own RNE rounding
    of Cref, FP32 output with Cref);
  * per element |C - Cref| <= 1e-2 |Cref| + 1e-2 rms(Cref).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import bf16, gemm, quant

FROB_TOL = 1e-3


def ld4(r: int) -> int:
    return (r + 3) // 4 * 4


def to_np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def pad_rows_scale(s_logical: np.ndarray, rows: int) -> np.ndarray:
    """[KB, rows] -> [KB, ld4(rows)] (padding zero)."""
    out = np.zeros((s_logical.shape[0], ld4(rows)), np.float32)
    out[:, :rows] = s_logical
    return out


def oracle_quant_rows(x: torch.Tensor, pow2=False):
    """Oracle 1x128 quantization of a [M, K] tensor -> (q np, s [KB, M] np)."""
    return quant.quant_1x128(to_np32(x), pow2)


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def compare_gemm(c_gpu: torch.Tensor, cref: np.ndarray, out_bf16: bool, tol=FROB_TOL):
    """Raise AssertionError with a message unless C matches the oracle's Cref."""
    c = c_gpu.detach().double().cpu().numpy() if isinstance(c_gpu, torch.Tensor) else np.asarray(c_gpu)
    assert c.shape == cref.shape, (c.shape, cref.shape)
    assert np.all(np.isfinite(c)), "non-finite output"
    rounded = bf16.round_bf16(cref) if out_bf16 else cref
    frob = gemm.frobenius_rel(c, rounded)
    ok = gemm.elementwise_ok(c, cref)
    bad = int((~ok).sum())
    assert frob <= tol and bad == 0, f"rel-Frobenius {frob:.3e} (tol {tol}), {bad} elements out of bound"
    return frob
