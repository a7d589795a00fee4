"""Emulator of limited-precision tensor-core accumulation (test infrastructure).

What the pages say (DeepSeek-V3 report excerpt):

* page 2, first paragraph: on Hopper, FP8 GEMM accumulates in fixed point;
  the mantissa products are aligned by right-shifting to the largest
  exponent before they are added, only the highest 14 bits of each product
  survive the sign-fill right shift, and the bits below are truncated;
* page 1, first paragraph: with K=4096 this limited accumulation gives a
  maximum relative error of almost 2% in a preliminary test;
* page 1, third paragraph: the fix is to copy the partial results to FP32
  registers on the CUDA cores at a fixed interval along K and accumulate
  there in full FP32 precision.

Model (the pages leave the group size and the exact alignment set open; the
reading fixed here):

* the tensor core adds ``chunk`` products at a time (one MMA instruction's
  K extent, 32 for FP8) into its FP32 accumulator register;
* for each addition, the largest exponent ``E`` among the accumulator and
  the ``chunk`` products sets the fixed-point grid ``2^(E - bits + 1)``;
  each addend is truncated to that grid by a sign-fill (arithmetic) right
  shift, i.e. rounded toward minus infinity;
* the aligned integers are summed exactly and the sum is rounded to FP32;
* with promotion, every ``promote`` products the accumulator is added into
  a separate FP32 register with an IEEE FP32 add and restarts from zero.

``mode="fp32"`` is the reference accumulation: sequential IEEE float32
additions of the (exact) products.
"""
from __future__ import annotations

import numpy as np


def _floor_to_grid(t: np.ndarray, E: np.ndarray, bits: int) -> np.ndarray:
    quantum = np.exp2(E - (bits - 1))
    return np.floor(t / quantum[:, None]) * quantum[:, None]


def accumulate(products, mode: str = "fixed", chunk: int = 32, bits: int = 14,
               promote: int | None = None) -> np.ndarray:
    """Sum ``products[r, :]`` for each row r the way the chosen unit would.

    products: float64 [R, K] (exact products of FP8 values).
    Returns float64 [R] holding float32-representable values.
    """
    p = np.asarray(products, dtype=np.float64)
    R, K = p.shape
    if mode == "fp32":
        acc = np.zeros(R, dtype=np.float32)
        for k in range(K):
            acc = (acc + p[:, k].astype(np.float32)).astype(np.float32)
        return acc.astype(np.float64)
    if mode != "fixed":
        raise ValueError(mode)
    outer = np.zeros(R, dtype=np.float32)      # promoted FP32 register
    acc = np.zeros(R, dtype=np.float64)        # tensor-core accumulator (fp32 values)
    for k0 in range(0, K, chunk):
        terms = np.concatenate([acc[:, None], p[:, k0:k0 + chunk]], axis=1)
        mx = np.abs(terms).max(axis=1)
        nz = mx > 0
        E = np.where(nz, np.floor(np.log2(np.where(nz, mx, 1.0))), 0.0)
        aligned = _floor_to_grid(terms, E, bits)
        acc = aligned.sum(axis=1).astype(np.float32).astype(np.float64)
        if promote is not None and (k0 + chunk) % promote == 0:
            outer = (outer + acc.astype(np.float32)).astype(np.float32)
            acc = np.zeros(R, dtype=np.float64)
    if promote is not None:
        outer = (outer + acc.astype(np.float32)).astype(np.float32)
        return outer.astype(np.float64)
    return acc


def max_error_over_rms(c, ref) -> float:
    """max |C - Cref| / rms(Cref): the error measure used for the K sweeps."""
    c = np.asarray(c, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(c - ref).max() / np.sqrt(np.mean(ref * ref)))
