"""GPU parity of the three quantizers against the oracle: bit-exact bytes and scales."""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle import quant
from parity import dev, ld4, to_np32

pytestmark = pytest.mark.gpu


def _check_1x128(fg, x, pow2):
    q, s = fg.fp8_quant_1x128(x, pow2=pow2)
    torch.cuda.synchronize()
    M, K = x.shape
    qo, so = quant.quant_1x128(to_np32(x), pow2)
    qg = q.cpu().numpy()
    sg = s.cpu().numpy()[:, :M]
    assert np.array_equal(sg.view(np.uint32), so.view(np.uint32)), "scales differ"
    diff = np.argwhere(qg != qo)
    assert diff.size == 0, f"{len(diff)} bytes differ, first at {diff[:3].tolist()}"


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("shape,dtype", [((128, 512), torch.float32), ((1, 128), torch.bfloat16),
                                         ((37, 384), torch.bfloat16), ((300, 1024), torch.float32),
                                         ((64, 7168), torch.bfloat16), ((129, 2048), torch.bfloat16)])
def test_quant_1x128_matches_oracle(lib, shape, dtype, pow2):
    x = wl.activations(*shape, seed=101 + shape[0], device="cuda", dtype=dtype)
    _check_1x128(lib, x, pow2)


def test_quant_1x128_tiny_config(lib):
    a, _ = wl.tiny_inputs(1000, device="cuda")
    for pow2 in (False, True):
        _check_1x128(lib, a, pow2)


def test_quant_1x128_edge_values(lib):
    x = torch.zeros((8, 640), dtype=torch.float32)
    x[1, :128] = 448.0                      # exact max
    x[2, :128] = -0.0                        # negative zeros only
    x[3, 5] = 1e-42                          # subnormal amax
    x[3, 6] = -3e-43
    x[4, :128] = torch.linspace(-1, 1, 128)  # spans ties after scaling
    x[5, 128:256] = 3.0e38                   # huge
    x[5, 300] = -3.0e38
    x[6, 256:384] = torch.tensor([2.0 ** -10] * 127 + [448.0 * 2 ** -10])  # tie with zero
    x[7] = torch.randn(640) * 1e-20
    x = x.cuda()
    for pow2 in (False, True):
        _check_1x128(lib, x, pow2)


def test_quant_1x128_strided_rows(lib):
    base = wl.activations(64, 1024, seed=7, device="cuda", dtype=torch.bfloat16)
    x = base[:, :512]  # ldx = 1024
    q, s = lib.fp8_quant_1x128(x)
    qo, so = quant.quant_1x128(to_np32(x))
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(s.cpu().numpy()[:, :64], so)


@pytest.mark.slow
def test_quant_1x128_prefill_sampled_rows(lib):
    x = wl.activations(wl.PREFILL_M, wl.PREFILL_K, seed=1001, device="cuda")
    q, s = lib.fp8_quant_1x128(x)
    rows = np.random.default_rng(0).choice(wl.PREFILL_M, 96, replace=False)
    rows = np.concatenate([[0, wl.PREFILL_M - 1], rows])
    qo, so = quant.quant_1x128(to_np32(x[rows]))
    assert np.array_equal(q[rows].cpu().numpy(), qo)
    assert np.array_equal(s[:, rows].cpu().numpy(), so)


def _check_128x128(fg, w, pow2=False):
    q, s = fg.fp8_quant_128x128(w, pow2=pow2)
    qo, so = quant.quant_128x128(to_np32(w), pow2)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32)), "scales differ"
    diff = np.argwhere(q.cpu().numpy() != qo)
    assert diff.size == 0, f"{len(diff)} bytes differ, first at {diff[:3].tolist()}"


@pytest.mark.parametrize("shape,dtype", [((256, 512), torch.float32), ((200, 256), torch.bfloat16),
                                         ((3, 130, 384), torch.bfloat16), ((1, 8, 128), torch.float32),
                                         ((2112, 1024), torch.bfloat16)])
def test_quant_128x128_matches_oracle(lib, shape, dtype):
    w = wl.weights(shape, seed=202 + shape[-2], device="cuda", dtype=dtype)
    _check_128x128(lib, w)


def test_quant_128x128_pow2_and_zero_block(lib):
    w = wl.weights((260, 384), seed=5, device="cuda", dtype=torch.float32)
    w[128:256, 128:256] = 0
    _check_128x128(lib, w, pow2=True)
    _check_128x128(lib, w, pow2=False)


@pytest.mark.slow
def test_quant_128x128_expert_weights_sampled_blocks(lib):
    # 8 experts x 4096 x 7168 bf16: check three whole 128-row slabs per expert pair
    w = wl.weights((8, 4096, 7168), seed=3001, device="cuda")
    q, s = lib.fp8_quant_128x128(w)
    for g, nb in [(0, 0), (3, 17), (7, 31)]:
        rows = slice(nb * 128, nb * 128 + 128)
        qo, so = quant.quant_128x128(to_np32(w[g, rows]))
        assert np.array_equal(q[g, rows].cpu().numpy(), qo)
        assert np.array_equal(s[g, nb].cpu().numpy(), so[0])


# ---------------------------------------------------------------- 128x1
def _check_requant(fg, src_dev, s_src_dev, oracle_src, oracle_s, G, valid=None, pow2=False):
    vr = None if valid is None else torch.tensor(valid, dtype=torch.int32, device="cuda")
    qT, sT = fg.fp8_requant_128x1(src_dev, s_src_dev, vr, pow2)
    qTg = qT.cpu().numpy().reshape(G, *qT.shape[-2:])
    sTg = sT.cpu().numpy().reshape(G, *sT.shape[-2:])
    for g in range(G):
        qo, so = quant.requant_128x1(oracle_src[g], None if oracle_s is None else oracle_s[g],
                                     None if valid is None else valid[g], pow2)
        C = qo.shape[0]
        assert np.array_equal(sTg[g][:, :C].view(np.uint32), so.view(np.uint32)), f"group {g} scales differ"
        diff = np.argwhere(qTg[g] != qo)
        assert diff.size == 0, f"group {g}: {len(diff)} bytes differ, first {diff[:3].tolist()}"


@pytest.mark.parametrize("pow2", [False, True])
def test_requant_from_fp8_source(lib, pow2):
    G, T, C = 2, 256, 384
    x = wl.activations(G * T, C, seed=401, device="cpu", dtype=torch.float32).view(G, T, C)
    qs, ss = [], []
    for g in range(G):
        q, s = quant.quant_1x128(x[g].numpy())     # oracle-made FP8 source
        qs.append(q)
        ss.append(s)
    q_dev = dev(np.stack(qs))
    s_pad = np.zeros((G, C // 128, ld4(T)), np.float32)
    for g in range(G):
        s_pad[g, :, :T] = ss[g]
    _check_requant(lib, q_dev.view(torch.float8_e4m3fn), dev(s_pad), np.stack(qs), np.stack(ss), G, pow2=pow2)


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_requant_from_float_source_with_valid_rows(lib, pow2, dtype):
    G, T, C = 3, 256, 256
    g_ = wl.normal((G, T, C), seed=402, device="cuda", dtype=dtype)
    valid = [256, 100, 0]
    _check_requant(lib, g_, None, to_np32(g_), None, G, valid=valid, pow2=pow2)


@pytest.mark.slow
def test_requant_prefill_activation_sampled(lib):
    T, C = wl.PREFILL_M, wl.PREFILL_K
    x = wl.activations(T, C, seed=1001, device="cpu", dtype=torch.float32)
    # oracle-quantize two 128-token blocks; requant them on the GPU in place of the full matrix
    q_full = torch.zeros((T, C), dtype=torch.uint8)
    s_full = np.ones((C // 128, ld4(T)), np.float32)
    blocks = [0, 31]
    for tb in blocks:
        q, s = quant.quant_1x128(x[tb * 128:(tb + 1) * 128].numpy())
        q_full[tb * 128:(tb + 1) * 128] = torch.from_numpy(q)
        s_full[:, tb * 128:(tb + 1) * 128] = s
    qT, sT = lib.fp8_requant_128x1(q_full.cuda().view(torch.float8_e4m3fn), dev(s_full), pow2=True)
    for tb in blocks:
        q, s = quant.quant_1x128(x[tb * 128:(tb + 1) * 128].numpy())
        qo, so = quant.requant_128x1(q, s, None, True)
        assert np.array_equal(qT[:, tb * 128:(tb + 1) * 128].cpu().numpy(), qo)
        assert np.array_equal(sT[tb, :C].cpu().numpy(), so[0])


# ---------------------------------------------------------------- many chunks per CTA
# The quantizers are persistent: one CTA per SM walks its chunks through a
# ring of 3-12 shared-memory stages. These sizes give every CTA more chunks
# than stages, so stages are refilled and barrier phases flip several times.
@pytest.mark.slow
@pytest.mark.parametrize("pow2", [False, True])
def test_quant_1x128_ring_wrap(lib, pow2):
    x = wl.activations(2432, 8192, seed=5, device="cuda")  # BF16: 19 x 64 chunks, 6 stages
    _check_1x128(lib, x, pow2)


@pytest.mark.slow
def test_quant_1x128_fp32_ring_wrap(lib):
    x = wl.activations(1216, 8192, seed=8, device="cuda", dtype=torch.float32)  # 19 x 64 chunks of 64 rows
    _check_1x128(lib, x, False)


@pytest.mark.slow
def test_quant_128x128_ring_wrap(lib):
    w = wl.weights((2, 1408, 8192), seed=7, device="cuda")  # 2 x 11 x 64 blocks, 6 stages
    _check_128x128(lib, w)


@pytest.mark.slow
@pytest.mark.parametrize("pow2", [False, True])
def test_requant_ring_wrap(lib, pow2):
    T, C = 4096, 8192  # E4M3 source: 32 x 64 tiles, 11 stages
    x = wl.activations(T, C, seed=6, device="cpu", dtype=torch.float32).numpy()
    q, s = quant.quant_1x128(x)
    s_pad = np.zeros((C // 128, ld4(T)), np.float32)
    s_pad[:, :T] = s
    _check_requant(lib, dev(q).view(torch.float8_e4m3fn)[None], dev(s_pad)[None], q[None], s[None], 1, pow2=pow2)


@pytest.mark.slow
def test_requant_bf16_ring_wrap_with_valid_rows(lib):
    G, T, C = 3, 1024, 4096  # BF16 source: 3 x 8 x 32 tiles, 6 stages; 1.5 groups valid
    g_ = wl.normal((G, T, C), seed=9, device="cuda", dtype=torch.bfloat16)
    _check_requant(lib, g_, None, to_np32(g_), None, G, valid=[1024, 500, 0], pow2=True)


# ---------------------------------------------------------------- bounded waits
def _expect_timeout(fg, call):
    fg.check()
    try:
        fg.debug_set(1, 50_000_000)   # 50 ms wait limit
        fg.debug_set(2, 0)            # every producer skips its first fill
        call()
        with pytest.raises(fg.Fp8fgError) as ei:
            fg.check()
        assert ei.value.code == fg.ERR_TIMEOUT
    finally:
        fg.debug_set(2, -1)
        fg.debug_set(1, 0)


def test_quantizer_timeouts_report_error_and_context_survives(lib):
    x = wl.activations(256, 1024, seed=11, device="cuda")
    w = wl.weights((256, 1024), seed=12, device="cuda")
    _expect_timeout(lib, lambda: lib.fp8_quant_1x128(x))
    _expect_timeout(lib, lambda: lib.fp8_quant_128x128(w))
    _expect_timeout(lib, lambda: lib.fp8_requant_128x1(x))
    # the context is intact and the next calls are exact
    _check_1x128(lib, x, False)
    _check_128x128(lib, w)
    _check_requant(lib, x, None, to_np32(x)[None], None, 1)


@pytest.mark.parametrize("pow2", [False, True])
def test_requant_signed_zeros_and_zero_channels(lib, pow2):
    # E4M3 source holding +0 (0x00) and -0 (0x80) codes, an all-zero channel
    # and an all-(-0) token block; BF16 source with -0 entries.
    T, C = 256, 256
    rng = np.random.default_rng(77)
    q = rng.integers(0, 256, size=(T, C), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x7E                 # no NaN codes
    q[:, 5] = 0x00
    q[:, 6] = 0x80
    q[128:, 200] = 0x80
    q[rng.random((T, C)) < 0.05] = 0x80
    s = np.exp2(rng.integers(-8, 8, size=(C // 128, T))).astype(np.float32) * 0.75
    s_pad = np.zeros((C // 128, ld4(T)), np.float32)
    s_pad[:, :T] = s
    _check_requant(lib, dev(q).view(torch.float8_e4m3fn)[None], dev(s_pad)[None], q[None], s[None], 1, pow2=pow2)
    xb = wl.normal((T, C), seed=78, device="cuda", dtype=torch.bfloat16)
    xb[:, 10] = -0.0
    xb[:64, 11] = 0.0
    xb[64:, 11] = -0.0
    _check_requant(lib, xb, None, to_np32(xb)[None], None, 1, pow2=pow2)
