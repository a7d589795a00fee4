"""E4M3 codec (test infrastructure; see package docstring).

Format, as the DeepGEMM article's "Was ist fp8?" section names it (E4M3 next
to E5M2) and the OCP 8-bit floating point specification defines it (the
"FN" variant used for training): 1 sign bit, 4 exponent bits with bias 7,
3 mantissa bits; no infinities; exponent 1111 with mantissa 111 is NaN, so
the largest finite magnitude is 1.75 * 2^8 = 448. Exponent 0000 encodes
subnormals m * 2^-9.

Encoding used by the quantizers (the pages name E4M3 but not its rounding;
this is the reading taken): round to
nearest on the exact value with ties to the even code, and saturate every
finite magnitude that would land above 448 to 448 (the ``satfinite`` mode).
The sign bit is copied from the input, so values that round to zero keep
their sign. NaN encodes as 0x7F.
"""
from __future__ import annotations

import numpy as np

BIAS = 7
MAX_FINITE = 448.0
NAN_CODE = 0x7F


def decode(codes) -> np.ndarray:
    """Codes (uint8 array) -> exact values as float64 (NaN for NaN codes)."""
    c = np.asarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m.astype(np.float64) * 2.0 ** (1 - BIAS - 3)  # m/8 * 2^(1-bias)
    nor = (1.0 + m.astype(np.float64) / 8.0) * np.exp2((e - BIAS).astype(np.float64))
    mag = np.where(e == 0, sub, nor)
    val = np.where(sign == 1, -mag, mag)
    return np.where((c & 0x7F) == NAN_CODE, np.nan, val)


# All finite non-negative values in code order 0x00..0x7E (strictly increasing).
_POS = decode(np.arange(0x7F))


def encode(values) -> np.ndarray:
    """float values -> E4M3 codes (uint8), RNE ties-to-even-code, satfinite."""
    v = np.asarray(values, dtype=np.float64)
    mag = np.abs(v)
    # Index of the largest representable magnitude <= |v| (|v| < 448 here).
    lo = np.clip(np.searchsorted(_POS, mag, side="right") - 1, 0, len(_POS) - 2)
    hi = lo + 1
    d_lo = mag - _POS[lo]
    d_hi = _POS[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= MAX_FINITE, 0x7E, code)
    code = code | np.where(np.signbit(v), 0x80, 0)
    code = np.where(np.isnan(v), NAN_CODE, code)
    return code.astype(np.uint8)


def ulp(value) -> np.ndarray:
    """Spacing of E4M3 values at |value| (<= 448): 2^-9 below 2^-6, else 2^(e-3)."""
    mag = np.abs(np.asarray(value, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(mag, 2.0 ** -6)))
    return np.exp2(e - 3)
