"""FP8 (E4M3) KV cache, restated (oracle, test-only).

The walkthrough's size formula only lets one stored number cost p = 1 byte;
besides INT8 (``quant``), the other 1-byte format is FP8.  Reading (the pages
give no scheme): E4M3 as NVIDIA's FP8 "e4m3" (1 sign bit, 4 exponent bits with
bias 7, 3 mantissa bits, no infinities, exponent and mantissa all ones is NaN,
largest finite 448, subnormals down to 2^-9); every (token, KV head) row has
one fp32 scale = amax / 448 (fp32 division), code = E4M3 of fp32(x / scale)
rounded to nearest, ties to even, saturated to +-448; an all-zero row has
scale 0 and codes 0.  Dequantised value = decode(code) * scale.  Decode keeps
q unquantised: scores are scale * q . (decode(k_code) * k_scale) and the
softmax weights mix decode(v_code) * v_scale.
"""
import numpy as np

from .attention import as_f64


def _e4m3_table():
    """Values of the 127 non-negative finite codes 0x00..0x7E, by code."""
    vals = np.empty(127)
    for code in range(127):
        e, m = code >> 3, code & 7
        vals[code] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_TABLE = _e4m3_table()


def e4m3_decode(codes):
    """uint8 codes -> float64 values (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag = c & 0x7F
    out = np.where(mag == 0x7F, np.nan, _TABLE[np.minimum(mag, 126)])
    return np.where(c & 0x80, -out, out)


def e4m3_encode(x):
    """float values -> uint8 codes: nearest finite E4M3 value, ties to the even
    code, magnitudes beyond 448 saturated to 448, NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # nearest of the sorted table (it is increasing in the code)
    hi = np.clip(np.searchsorted(_TABLE, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_hi, d_lo = np.abs(_TABLE[hi] - a), np.abs(a - _TABLE[lo])
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= 448.0, 126, pick)
    code = pick.astype(np.int64) | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize_fp8(x_bits):
    """bf16 bits [..., D] -> (codes uint8 [..., D], scales float32 [...])."""
    x = as_f64(x_bits).astype(np.float32)                 # exact: bf16 fits fp32
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(448.0)).astype(np.float32)  # fp32 division
    safe = np.where(scale > 0, scale, np.float32(1.0))
    y = (x / safe[..., None]).astype(np.float32)           # fp32 division
    codes = np.where(scale[..., None] > 0, e4m3_encode(y), 0).astype(np.uint8)
    return codes, scale


def dequantize_fp8(codes, scales):
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def reshape_and_cache_fp8(key, value, k_codes, v_codes, k_scales, v_scales, slot_mapping,
                          block_size, inplace=False):
    """The cache write into an FP8 pool: pools [NB, Hkv, bs, D] uint8 (E4M3
    codes), scales [NB, Hkv, bs] float32; key/value [T, Hkv, D] bf16 bits."""
    kc = k_codes if inplace else np.array(k_codes, copy=True)
    vc = v_codes if inplace else np.array(v_codes, copy=True)
    ks = k_scales if inplace else np.array(k_scales, copy=True)
    vs = v_scales if inplace else np.array(v_scales, copy=True)
    kq, kscale = quantize_fp8(key)
    vq, vscale = quantize_fp8(value)
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        kc[blk, :, off, :] = kq[t]
        vc[blk, :, off, :] = vq[t]
        ks[blk, :, off] = kscale[t]
        vs[blk, :, off] = vscale[t]
    return kc, vc, ks, vs


def decode_fp8(q_bits, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens,
               scale, block_size):
    """Paged decode over an FP8 cache in float64; q unquantised.  Returns
    out [B, Hq, D]; an empty sequence gives zeros."""
    q = as_f64(q_bits)
    B, hq, d = q.shape
    hkv = k_codes.shape[1]
    group = hq // hkv
    out = np.zeros((B, hq, d))
    for b in range(B):
        n = int(context_lens[b])
        if n == 0:
            continue
        pos = np.arange(n)
        phys = np.asarray(block_tables[b], dtype=np.int64)[pos // block_size]
        off = pos % block_size
        K = dequantize_fp8(k_codes[phys, :, off, :], k_scales[phys, :, off])   # [n, Hkv, D]
        V = dequantize_fp8(v_codes[phys, :, off, :], v_scales[phys, :, off])
        for h in range(hq):
            g = h // group
            s = scale * (K[:, g, :] @ q[b, h])
            w = np.exp(s - s.max())
            out[b, h] = (w @ V[:, g, :]) / w.sum()
    return out
