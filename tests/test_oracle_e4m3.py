"""Pins for the oracle's E4M3 codec and BF16 rounding (CPU only).

The codec is checked against two library implementations of the same
format (torch.float8_e4m3fn and ml_dtypes.float8_e4m3fn), against closed-form
values of the OCP E4M3 definition, and on every tie point.
"""
import ml_dtypes
import numpy as np
import torch

from oracle import bf16, e4m3


def _torch_decode(codes):
    t = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _torch_encode(values):
    v = np.clip(np.asarray(values, np.float32), -448.0, 448.0)
    t = torch.from_numpy(v).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_decode_all_codes_match_torch_and_ml_dtypes():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3.decode(codes)
    ref_t = _torch_decode(codes)
    ref_m = codes.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    for ref in (ref_t, ref_m):
        assert np.array_equal(np.isnan(ours), np.isnan(ref))
        ok = ~np.isnan(ref)
        assert np.array_equal(ours[ok], ref[ok])


def test_decode_closed_forms():
    d = lambda c: float(e4m3.decode(np.array([c], np.uint8))[0])  # noqa: E731
    assert d(0x7E) == 448.0            # largest finite
    assert d(0xFE) == -448.0
    assert d(0x01) == 2.0 ** -9        # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9    # largest subnormal
    assert d(0x08) == 2.0 ** -6        # smallest normal
    assert d(0x38) == 1.0
    assert d(0x40) == 2.0
    assert d(0x77) == 240.0
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x80) == 0.0 and np.signbit(d(0x80))


def test_encode_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    assert np.array_equal(e4m3.encode(e4m3.decode(codes)), codes)


def test_encode_ties_and_neighbours_match_torch():
    pos = e4m3.decode(np.arange(0x7F))
    mids = (pos[:-1] + pos[1:]) / 2  # exact in float32 (<= 5 significant bits)
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)
    up = np.nextafter(m32, np.float32(np.inf))
    dn = np.nextafter(m32, np.float32(-np.inf))
    vals = np.concatenate([m32, up, dn, pos.astype(np.float32)])
    vals = np.concatenate([vals, -vals])
    assert np.array_equal(e4m3.encode(vals), _torch_encode(vals))
    mine_m = vals.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(e4m3.encode(vals), mine_m)


def test_encode_dense_sweep_matches_torch():
    rng = np.random.default_rng(5)
    mag = np.exp2(rng.uniform(-14, 9, 400_000)).astype(np.float32)
    sign = np.where(rng.random(mag.size) < 0.5, -1, 1).astype(np.float32)
    vals = mag * sign
    vals = vals[np.abs(vals) <= 448]
    assert np.array_equal(e4m3.encode(vals), _torch_encode(vals))


def test_encode_saturates_and_keeps_sign_of_zero():
    big = np.array([448.0, 449.0, 464.0, 479.9, 480.0, 1e6, 3.0e38], np.float32)
    assert np.all(e4m3.encode(big) == 0x7E)
    assert np.all(e4m3.encode(-big) == 0xFE)
    tiny = np.array([-0.0, -1e-10, -2.0 ** -11], np.float32)
    assert np.all(e4m3.encode(tiny) == 0x80)
    assert np.all(e4m3.encode(-tiny) == 0x00)
    # exactly half the smallest subnormal is a tie with zero (even code)
    assert e4m3.encode(np.float32(2.0 ** -10)) == 0x00
    assert e4m3.encode(np.float32(np.nextafter(np.float32(2.0 ** -10), np.float32(1)))) == 0x01


def test_ulp_closed_form():
    assert e4m3.ulp(1.0) == 0.125
    assert e4m3.ulp(448.0) == 32.0
    assert e4m3.ulp(2.0 ** -7) == 2.0 ** -9
    assert e4m3.ulp(0.0) == 2.0 ** -9


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-30, 30, 200_000))).astype(np.float32)
    # add exact ties: bf16 value + half ulp
    b = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    ties = (b.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(bf16.round_bf16(x), ref)
