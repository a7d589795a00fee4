"""Round-to-nearest-even to bfloat16 (test infrastructure; see package docstring).

The DeepSeek-V3 report excerpt (page 1, third paragraph) has the FP8 GEMMs
emit BF16 or FP32. BF16 keeps the top 16 bits of an FP32 word; the value is
first rounded to FP32 (RNE), then to 8 significant bits (RNE on the FP32
bit pattern). Returned as float64 for comparison.
"""
from __future__ import annotations

import numpy as np


def round_bf16(x) -> np.ndarray:
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    out = rounded.astype(np.uint32).view(np.float32).astype(np.float64)
    return np.where(np.isfinite(f), out, f.astype(np.float64))
