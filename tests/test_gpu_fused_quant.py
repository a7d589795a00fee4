"""Fused 1x128 quantization of the GEMM output (fp8_gemm_dense_quant).

The epilogue quantizes the BF16-rounded result per 1x128 tile for the next
layer (DeepSeek-V3 report excerpt, page 1, paragraph 3; the request to fuse
the FP8 cast with data movement, page 2, last paragraph). Checks:

* the BF16 result it also writes matches the oracle's FP64 product of the
  oracle-quantized operands within the GEMM tolerance;
* its codes and scales are bit-identical to the standalone 1x128 quantizer
  applied to that BF16 result (the standalone quantizer is bit-exact against
  the oracle in test_gpu_quant.py);
* against the oracle alone: every tile's largest code is +-448 (amax maps to
  448 when scales are not powers of two), each scale is within the GEMM
  tolerance of the oracle's amax(Cref)/448 for that tile, and the dequantized
  values q*s stay within E4M3 rounding of Cref.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import e4m3, gemm, quant
from parity import compare_gemm, dev, pad_rows_scale, to_np32

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    x = wl.activations(M, K, seed, device="cpu")
    w = wl.weights((N, K), seed + 1, device="cpu")
    qa, sa = quant.quant_1x128(to_np32(x))
    qb, sb = quant.quant_128x128(to_np32(w))
    return qa, sa, qb, sb, dev(qa), dev(pad_rows_scale(sa, M)), dev(qb), dev(sb)


@pytest.mark.parametrize("M,N,K,pow2", [
    (256, 512, 512, False),
    (200, 384, 1024, True),     # ragged rows, power-of-2 scales; N ends halfway through a 256-column tile
    (64, 1024, 2048, False),    # decode-sized: K split over the SMs (Stream-K)
    (1024, 2048, 1024, False),  # several tiles per CTA
])
def test_fused_quant(lib, M, N, K, pow2):
    qa, sa, qb, sb, qa_d, sa_d, qb_d, sb_d = _operands(M, N, K, 5000 + M + N)
    q, s, c = lib.fp8_gemm_dense_quant(qa_d, sa_d, qb_d, sb_d, pow2=pow2, with_bf16=True)
    lib.check()
    cref = gemm.gemm_dense(qa, sa, qb, sb)
    compare_gemm(c, cref, True)
    # bit-identical to quantizing the BF16 result with the standalone kernel
    q2, s2 = lib.fp8_quant_1x128(c, pow2=pow2)
    torch.cuda.synchronize()
    assert torch.equal(q, q2), "codes differ from fp8_quant_1x128 of the BF16 result"
    assert torch.equal(s[:, :M], s2[:, :M]), "scales differ from fp8_quant_1x128 of the BF16 result"
    # the oracle's view of the same tiles
    qn = q.cpu().numpy()
    sn = s.cpu().numpy()[:, :M].astype(np.float64)          # [N/128, M]
    vals = e4m3.decode(qn)
    tiles = np.abs(vals).reshape(M, N // 128, 128).max(axis=2)
    if not pow2:
        assert np.all(tiles == 448.0), "a tile's largest code is not 448"
    else:
        assert np.all(tiles <= 448.0) and np.all(tiles >= 224.0), "pow2 tiles must land in [224, 448]"
    amax_ref = np.abs(cref).reshape(M, N // 128, 128).max(axis=2) / 448.0   # [M, N/128]
    if not pow2:
        rel = np.abs(sn.T - amax_ref) / amax_ref
        assert rel.max() < 1e-2, f"scale off the oracle's amax/448 by {rel.max():.2e}"
    deq = vals * np.repeat(sn.T, 128, axis=1)
    # E4M3 keeps 4 significant bits: relative rounding <= 2^-4 of |C| per element
    err = np.abs(deq - cref)
    # plus the GEMM tolerance between the BF16 result and Cref
    bound = (2.0 ** -4 + 1e-2) * np.abs(cref) + np.repeat(sn.T, 128, axis=1) * 2.0 ** -9 + \
        1e-2 * np.sqrt(np.mean(cref ** 2))
    assert np.all(err <= bound), f"{int((err > bound).sum())} dequantized values outside E4M3 rounding of Cref"


def test_fused_quant_writes_nothing_past_its_outputs(lib):
    # N = 384 leaves the last 256-column tile half empty: its second half has
    # no codes or scales to write. Canaries after q and s must survive.
    M, N, K = 256, 384, 1024
    qa, sa, qb, sb, qa_d, sa_d, qb_d, sb_d = _operands(M, N, K, 5201)
    qbuf = torch.full((M * N + 4096,), 0x5A, dtype=torch.uint8, device="cuda")
    sbuf = torch.full(((N // 128) * M + 4096,), -7.0, dtype=torch.float32, device="cuda")
    q = qbuf[:M * N].view(M, N)
    s = sbuf[:(N // 128) * M].view(N // 128, M)
    lib.fp8_gemm_dense_quant_out(qa_d, sa_d, qb_d, sb_d, q, s, workspace=lib.gemm_workspace(M, N, K))
    lib.check()
    assert torch.all(qbuf[M * N:] == 0x5A), "codes written past q"
    assert torch.all(sbuf[(N // 128) * M:] == -7.0), "scales written past s"


def test_fused_quant_without_bf16_output(lib):
    M, N, K = 512, 768, 1024
    qa, sa, qb, sb, qa_d, sa_d, qb_d, sb_d = _operands(M, N, K, 5101)
    q, s = lib.fp8_gemm_dense_quant(qa_d, sa_d, qb_d, sb_d)
    c = lib.fp8_gemm_dense(qa_d, sa_d, qb_d, sb_d)
    q2, s2 = lib.fp8_quant_1x128(c)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s[:, :M], s2[:, :M])


def test_fused_quant_rejects_bad_shapes(lib):
    t = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    f = torch.zeros(1024, dtype=torch.float32, device="cuda")
    with pytest.raises(lib.Fp8fgError) as ei:
        lib.fp8_gemm_dense_quant_out(t.view(32, 128), f, t.view(32, 128), f, t.view(32, 128), f)  # N=32
    assert ei.value.code == lib.ERR_UNSUPPORTED_SHAPE


@pytest.mark.slow
def test_fused_quant_prefill_sampled(lib):
    # the dense prefill shape whose output feeds the next layer: M=4096,
    # N=7168, K=7168; checked on sampled rows and column blocks
    M, N, K = wl.PREFILL_M, 7168, wl.PREFILL_K
    x = wl.activations(M, K, 1001, device="cuda")
    w = wl.weights((N, K), 2000 + N, device="cuda")
    qa_d, sa_d = lib.fp8_quant_1x128(x)
    qb_d, sb_d = lib.fp8_quant_128x128(w)
    q, s, c = lib.fp8_gemm_dense_quant(qa_d, sa_d, qb_d, sb_d, with_bf16=True)
    q2, s2 = lib.fp8_quant_1x128(c)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(s[:, :M], s2[:, :M])
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(M, 48, replace=False))
    qa, sa = quant.quant_1x128(to_np32(x[rows]))
    for nb in (0, 29, N // 128 - 1):
        cols = slice(nb * 128, nb * 128 + 128)
        qb, sb = quant.quant_128x128(to_np32(w[cols]))
        compare_gemm(c[rows][:, cols], gemm.gemm_dense(qa, sa, qb, sb), True)
