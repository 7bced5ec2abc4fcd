"""Pins of the FP8 (E4M3) oracle: the format's defining values, exhaustive
round trips, rounding ties, saturation, and the decode's reduction to plain
attention when every value is exactly representable."""
import numpy as np
import pytest

from oracle import fp8 as F
from paged_kv_cache_283_gb300.inputs import f32_to_bf16_bits


def test_defining_values():
    # E4M3: bias 7, 3 mantissa bits, largest finite 448 = 0x7E, NaN 0x7F,
    # smallest normal 2^-6 = 0x08, smallest subnormal 2^-9 = 0x01, 1.0 = 0x38
    dec = F.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x7E, 0xBE, 0x80], np.uint8))
    assert dec.tolist() == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 448.0, -1.75, -0.0]
    assert np.isnan(F.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    assert F.e4m3_encode(np.array([1.0, 448.0, -448.0, 2.0 ** -9, 0.0])).tolist() == [0x38, 0x7E, 0xFE, 0x01, 0x00]


def test_exhaustive_round_trip():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    assert np.array_equal(F.e4m3_encode(F.e4m3_decode(codes)), codes)


def test_ties_to_even_and_saturation():
    # between 1.0 (0x38) and 1.125 (0x39): 1.0625 ties -> even code 0x38
    # between 1.125 (0x39) and 1.25 (0x3A): 1.1875 ties -> 0x3A
    assert F.e4m3_encode(np.array([1.0625, 1.1875, 1.07, -1.0625])).tolist() == [0x38, 0x3A, 0x39, 0xB8]
    # between 416 (0x7D) and 448 (0x7E): 432 ties -> 0x7E (even); beyond 448 saturates
    assert F.e4m3_encode(np.array([432.0, 460.0, 1e6, -1e30])).tolist() == [0x7E, 0x7E, 0x7E, 0xFE]
    assert F.e4m3_encode(np.array([np.nan])).tolist() == [0x7F]


def test_quantize_rows():
    x = np.array([[448.0, -224.0, 1.0, 0.0], [0.0, 0.0, 0.0, 0.0], [-3.0, 1.5, 0.75, 0.1]])
    codes, scale = F.quantize_fp8(f32_to_bf16_bits(x.astype(np.float32)))
    assert scale[0] == np.float32(1.0) and scale[1] == 0.0
    assert codes[0].tolist() == [0x7E, 0xF6, 0x38, 0x00] and not codes[1].any()
    s2 = np.float32(np.float32(3.0) / np.float32(448.0))
    assert scale[2] == s2 and F.e4m3_decode(codes[2, :1]) == -448.0
    # round trip within half an E4M3 step (relative 2^-4) of each value
    back = F.dequantize_fp8(codes, scale)
    assert np.all(np.abs(back - x) <= np.abs(x) * 2.0 ** -4 + 2.0 ** -10)


def test_fp8_decode_equals_plain_attention_when_exact():
    from oracle import attention as A
    rng = np.random.default_rng(3)
    nb, hkv, bs, d, hq = 5, 2, 16, 8, 4
    # rows whose largest magnitude is 448 and all entries E4M3 values: scale 1
    pick = F.e4m3_decode(rng.integers(0, 0x7E, size=(nb, hkv, bs, d)).astype(np.uint8))
    pick = pick * np.where(rng.random(pick.shape) < 0.5, -1, 1)
    pick[..., 0] = 448.0
    kb = f32_to_bf16_bits(pick.astype(np.float32))
    vb = f32_to_bf16_bits((pick[..., ::-1]).astype(np.float32).copy())
    kq, ks = F.quantize_fp8(kb)
    vq, vs = F.quantize_fp8(vb)
    assert np.all(ks == 1.0) and np.all(vs == 1.0)
    q = f32_to_bf16_bits(rng.standard_normal((2, hq, d)).astype(np.float32))
    tables = [np.array([4, 0]), np.array([2, 1, 3])]
    ctx = np.array([20, 40])
    got = F.decode_fp8(q, kq, vq, ks, vs, tables, ctx, 0.01, bs)
    want = A.decode(q, pick, pick[..., ::-1], tables, ctx, 0.01, bs)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_fp8_cache_write_places_rows():
    rng = np.random.default_rng(4)
    nb, hkv, bs, d = 4, 2, 16, 8
    key = f32_to_bf16_bits(rng.standard_normal((3, hkv, d)).astype(np.float32))
    z8 = np.zeros((nb, hkv, bs, d), np.uint8)
    zs = np.zeros((nb, hkv, bs), np.float32)
    kc, vc, ks, vs = F.reshape_and_cache_fp8(key, key, z8, z8, zs, zs, np.array([17, -1, 63]), bs)
    cq, cs = F.quantize_fp8(key)
    assert np.array_equal(kc[1, :, 1], cq[0]) and np.array_equal(vs[3, :, 15], cs[2])
    assert np.count_nonzero(ks) == 2 * hkv
