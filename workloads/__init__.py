"""Seeded synthetic inputs for the fine-grained FP8 GEMM path.

This module only draws random numbers and lays out buffers. It holds none
of the method's arithmetic (no scaling, no rounding to FP8, no products), so
both the oracle-side tests and the CUDA path can take their inputs from it.

Shapes and value distributions follow the workloads the pages describe:

* DeepSeek-V3 report (page 1, third paragraph; page 2, third paragraph):
  activations quantized per 1x128 tile, decode batches of at most 256 tokens
  per expert.
* DeepGEMM article (page 4, Table 1): dense shapes M=64..4096, N=2112..7168,
  K=2048..7168.

Every generator takes an explicit seed. Large dense arrays are drawn with a
torch generator on the requested device; discrete choices (outlier rows or
channels, expert counts, permutations) are drawn with numpy's PCG64 on the
host, so they are identical on every device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 128


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, std: float = 1.0, device="cpu",
           dtype=torch.float32) -> torch.Tensor:
    """N(0, std^2) samples, drawn in fp32 and then cast to ``dtype``."""
    g = _gen(device, seed)
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def with_outlier_rows(x: torch.Tensor, frac: float, factor: float, seed: int) -> torch.Tensor:
    """Multiply ceil(frac * rows) seeded rows of a 2-D tensor by ``factor``."""
    rows = x.shape[0]
    n = max(1, math.ceil(frac * rows))
    idx = np.random.default_rng(seed).choice(rows, size=n, replace=False)
    x[torch.as_tensor(np.sort(idx), device=x.device)] *= factor
    return x


def with_outlier_channels(x: torch.Tensor, frac: float, factor: float, seed: int) -> torch.Tensor:
    """Multiply ceil(frac * cols) seeded columns (last dim) by ``factor``."""
    cols = x.shape[-1]
    n = max(1, math.ceil(frac * cols))
    idx = np.random.default_rng(seed).choice(cols, size=n, replace=False)
    x[..., torch.as_tensor(np.sort(idx), device=x.device)] *= factor
    return x


def activations(M: int, K: int, seed: int, device="cpu", dtype=torch.bfloat16,
                outlier_frac: float = 0.01, outlier_factor: float = 30.0) -> torch.Tensor:
    """Prefill/decode activations: N(0,1) with a seeded 1% of channels x30."""
    x = normal((M, K), seed, 1.0, device, torch.float32)
    with_outlier_channels(x, outlier_frac, outlier_factor, seed + 7)
    return x.to(dtype)


def weights(shape, seed: int, device="cpu", dtype=torch.bfloat16, std: float = 0.02) -> torch.Tensor:
    """Linear / expert weights: N(0, 0.02^2)."""
    return normal(shape, seed, std, device, dtype)


def tiny_inputs(seed: int = 1000, device="cpu"):
    """The small dense case: A[128,512], B[256,512] fp32 N(0,1), 2% of A rows x50."""
    a = normal((128, 512), seed, 1.0, device)
    with_outlier_rows(a, 0.02, 50.0, seed + 1)
    b = normal((256, 512), seed + 2, 1.0, device)
    return a, b


def zipf_counts(total: int, experts: int, s: float, seed: int) -> np.ndarray:
    """Token counts per expert: Multinomial(total, p_e ~ e^-s), ids permuted."""
    rng = np.random.default_rng(seed)
    p = np.arange(1, experts + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    counts = rng.multinomial(total, p)
    return counts[rng.permutation(experts)].astype(np.int64)


@dataclass
class ContigLayout:
    """Token rows sorted by expert, each expert's segment padded to 128 rows.

    ``m_indices[row]`` is the expert id of the row, or -1 for a padding row.
    """
    counts: np.ndarray
    padded: np.ndarray
    offsets: np.ndarray
    m_indices: np.ndarray
    m_total: int = field(init=False)

    def __post_init__(self):
        self.m_total = int(self.padded.sum())


def contig_layout(counts: np.ndarray, align: int = BLOCK) -> ContigLayout:
    counts = np.asarray(counts, dtype=np.int64)
    padded = (counts + align - 1) // align * align
    offsets = np.concatenate([[0], np.cumsum(padded)])
    m_idx = np.full(int(padded.sum()), -1, dtype=np.int32)
    for e, c in enumerate(counts):
        m_idx[offsets[e]:offsets[e] + c] = e
    return ContigLayout(counts, padded, offsets[:-1], m_idx)


def masked_counts(experts: int, max_m: int, seed: int, low: int = 1) -> np.ndarray:
    """Per-expert valid token counts, uniform on {low..max_m}."""
    return np.random.default_rng(seed).integers(low, max_m + 1, size=experts).astype(np.int32)


def zero_rows_beyond(x: torch.Tensor, counts, rows_per_group: int) -> torch.Tensor:
    """For x viewed as [G, rows_per_group, ...], zero rows >= counts[g] (masked padding)."""
    v = x.view(len(counts), rows_per_group, *x.shape[1:]) if x.dim() == 2 else x
    for g, c in enumerate(counts):
        v[g, int(c):] = 0
    return x


# Named workloads. Sizes are the ones the DeepGEMM article's Table 1 and the
# DeepSeek-V3 report's decode discussion describe; seeds are fixed per case.
PREFILL_M, PREFILL_K = 4096, 7168
PREFILL_NS = (2112, 24576, 7168, 4096)
DECODE_CASES = ((64, 7168, 16384), (128, 7168, 16384), (64, 4096, 7168), (128, 4096, 7168))
CONTIG_CASES = ((8, 8192, 4096, 7168), (8, 8192, 7168, 2048))  # experts, tokens, N, K
MASKED_CASE = (16, 256, 4096, 7168)  # experts, max tokens per expert, N, K
