"""Pins of the INT8 KV quantiser (oracle/quant.py): exact values worked by
hand, the round-trip error bound, and the cache write."""
import numpy as np

from oracle import quant as Q
from paged_kv_cache_283_gb300.inputs import f32_to_bf16_bits


def _bits(vals):
    return f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def test_worked_example():
    # amax 2.0 -> scale 2/127; 1.0 / (2/127) = 63.5 -> 64 (half to even);
    # -0.5 -> -31.75 -> -32; 2.0 -> 127; 0 -> 0
    codes, scale = Q.quantize_int8(_bits([[1.0, -0.5, 2.0, 0.0]]))
    assert scale[0] == np.float32(2.0) / np.float32(127.0)
    assert codes.tolist() == [[64, -32, 127, 0]]


def test_ties_round_to_even_and_sign_symmetry():
    # amax 127 -> scale 1: x/scale is x itself, halves go to the even integer
    x = _bits([[127.0, 0.5, 1.5, 2.5, -2.5, -127.0]])
    codes, scale = Q.quantize_int8(x)
    assert scale[0] == 1.0
    assert codes.tolist() == [[127, 0, 2, 2, -2, -127]]


def test_zero_row():
    codes, scale = Q.quantize_int8(_bits([[0.0] * 8]))
    assert scale[0] == 0.0 and not codes.any()


def test_round_trip_error_bound():
    rng = np.random.default_rng(9)
    x = _bits(rng.standard_normal((64, 128)).astype(np.float32) * 3)
    codes, scale = Q.quantize_int8(x)
    back = Q.dequantize(codes, scale)
    xf = x.astype(np.uint32) << 16
    xf = xf.view(np.float32).astype(np.float64)
    # half a quantisation step, plus fp32 rounding of the scale and the division
    bound = scale.astype(np.float64)[:, None] * (0.5 + 1e-5)
    assert np.all(np.abs(back - xf) <= bound)
    assert np.all(np.abs(codes) <= 127)
    assert np.all(np.max(np.abs(codes), axis=1) == 127)   # the largest value maps to 127


def test_cache_write_places_codes_and_scales():
    rng = np.random.default_rng(10)
    nb, hkv, bs, d = 4, 2, 16, 8
    kc = np.zeros((nb, hkv, bs, d), np.int8)
    ks = np.zeros((nb, hkv, bs), np.float32)
    key = _bits(rng.standard_normal((3, hkv, d)))
    kc2, vc2, ks2, vs2 = Q.reshape_and_cache_int8(key, key, kc, kc, ks, ks, [17, -1, 63], bs)
    cq, cs = Q.quantize_int8(key)
    assert np.array_equal(kc2[1, :, 1], cq[0]) and np.array_equal(ks2[1, :, 1], cs[0])
    assert np.array_equal(kc2[3, :, 15], cq[2]) and np.array_equal(vs2[3, :, 15], cs[2])
    assert np.count_nonzero(ks2) == 2 * hkv


def test_int8_decode_equals_plain_attention_when_codes_are_exact():
    # q and K rows whose largest entry is 127 and the rest integers: their
    # scales are exactly 1, the codes are the values themselves, and the INT8
    # decode must equal ordinary attention on the dequantised pools
    from oracle import attention as A
    rng = np.random.default_rng(12)
    nb, hkv, bs, d, hq = 6, 2, 16, 8, 4
    def ints(shape):
        x = rng.integers(-100, 100, size=shape).astype(np.float32)
        x[..., 0] = 127.0
        return x
    kf, vf, qf = ints((nb, hkv, bs, d)), ints((nb, hkv, bs, d)), ints((2, hq, d))
    kq, ks = Q.quantize_int8(_bits(kf))
    vq, vs = Q.quantize_int8(_bits(vf))
    assert np.all(ks == 1.0) and np.array_equal(kq.astype(np.float32), kf)
    tables = np.array([[3, 0, 5], [1, 2, 4]])
    ctx = np.array([40, 17])
    scale = 1.0 / 4096
    got = Q.decode_int8(_bits(qf), kq, vq, ks, vs, tables, ctx, scale, bs)
    want = A.decode(qf.astype(np.float64), kf, Q.dequantize(vq, vs), tables, ctx, scale, bs)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_int8_decode_empty_sequence():
    z8 = np.zeros((2, 1, 16, 8), np.int8)
    zs = np.zeros((2, 1, 16), np.float32)
    out = Q.decode_int8(_bits(np.ones((1, 2, 8))), z8, z8, zs, zs, np.array([[0]]),
                        np.array([0]), 1.0, 16)
    assert not out.any()


def test_int8_scheme_error_on_normal_data():
    # How far the INT8 scheme moves the decode output from the bf16 cache's
    # on N(0, 1) data.  One code step is amax / 127, about 3.5 / 127 of a
    # standard deviation for D = 128, so values and q carry a rounding error
    # of roughly step / sqrt(12) = 0.8 % rms; the softmax-weighted mean
    # inherits an error of that order.  A normwise 3 % per output row bounds
    # it with room; a wrong scale (e.g. a dropped k or q scale) is off by
    # orders of magnitude.
    from oracle import attention as A
    from oracle.cache import reshape_and_cache
    from paged_kv_cache_283_gb300 import inputs as I
    ctx = [64, 300, 1024, 2048]
    w = I.random_case(77, len(ctx), ctx, 32, 8, 128, num_blocks=512)
    bs = w.block_size
    tables = [list(range(i * 128, i * 128 + 128)) for i in range(len(ctx))]
    slots = np.array([t[(n - 1) // bs] * bs + (n - 1) % bs for t, n in zip(tables, ctx)])
    kc, vc = reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, slots, bs)
    full = A.decode(w.q, kc, vc, tables, np.array(ctx), w.scale, bs)
    kq, ks = Q.quantize_int8(w.k_cache)
    vq, vs = Q.quantize_int8(w.v_cache)
    kq, vq, ks, vs = Q.reshape_and_cache_int8(w.key, w.value, kq, vq, ks, vs, slots, bs)
    got = Q.decode_int8(w.q, kq, vq, ks, vs, tables, np.array(ctx), w.scale, bs)
    err = np.linalg.norm(got - full, axis=-1) / np.linalg.norm(full, axis=-1)
    assert err.max() < 3e-2
    assert err.mean() > 1e-4  # the codes really are lossy here
