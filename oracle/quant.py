"""INT8 KV cache: quantisation and dequantisation (oracle, test-only).

"LLM serving (vLLM, quantized inference): Visual walkthrough", Step 1: the
cost of one stored number, p, is 2 bytes in FP16/BF16 and 1 byte in INT8;
every KV-cache size scales with p.  The pages give no scaling scheme.  The
reading used: symmetric INT8 with one fp32 scale per (token, KV head), so
that a token can be written once and never re-quantised as the cache grows:

    amax  = max_d |x_d|                     (x the token's bf16 values in fp32)
    scale = amax / 127                      (fp32, round to nearest)
    code  = clamp(round_half_even(x_d / scale), -127, 127)   (fp32 division)
    x_d  ~= code * scale

with scale = 0 and all codes 0 when amax = 0.  Every step is one IEEE fp32
operation, so a faithful implementation reproduces the codes exactly.
"""
import numpy as np

from .bf16 import bf16_bits_to_f64


def quantize_int8(x_bits):
    """bf16 bits [..., D] -> (codes int8 [..., D], scales float32 [...])."""
    x = bf16_bits_to_f64(np.asarray(x_bits)).astype(np.float32)   # exact
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    q = np.rint((x / safe[..., None]).astype(np.float32))
    q = np.clip(q, -127, 127)
    q = np.where(scale[..., None] > 0, q, 0)
    return q.astype(np.int8), scale


def dequantize(codes, scales):
    """codes int8 [..., D], scales float32 [...] -> float64 values (exact)."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]


def reshape_and_cache_int8(key, value, k_codes, v_codes, k_scales, v_scales, slot_mapping,
                           block_size, inplace=False):
    """The cache write into an INT8 pool: pools [NB, Hkv, bs, D] int8, scales
    [NB, Hkv, bs] float32; key/value [T, Hkv, D] bf16 bits."""
    kc = k_codes if inplace else np.array(k_codes, copy=True)
    vc = v_codes if inplace else np.array(v_codes, copy=True)
    ks = k_scales if inplace else np.array(k_scales, copy=True)
    vs = v_scales if inplace else np.array(v_scales, copy=True)
    kq, kscale = quantize_int8(key)
    vq, vscale = quantize_int8(value)
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        kc[blk, :, off, :] = kq[t]
        vc[blk, :, off, :] = vq[t]
        ks[blk, :, off] = kscale[t]
        vs[blk, :, off] = vscale[t]
    return kc, vc, ks, vs


def decode_int8(q_bits, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens,
                scale, block_size):
    """Paged decode over an INT8 cache, float64 except where the method is
    integer: each query head is quantised by the same rule as the cache, the
    scores are scale * q_scale * k_scale_j * (integer dot of the codes), and
    the softmax weights mix the dequantised values (codes * v_scale).
    Returns out [B, Hq, D] float64; an empty sequence gives zeros."""
    qc, qs = quantize_int8(q_bits)                     # [B, Hq, D], [B, Hq]
    B, hq, d = qc.shape
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
        kc = k_codes[phys, :, off, :].astype(np.int64)        # [n, Hkv, D]
        ks = k_scales[phys, :, off].astype(np.float64)        # [n, Hkv]
        V = dequantize(v_codes[phys, :, off, :], v_scales[phys, :, off])
        for h in range(hq):
            g = h // group
            dots = kc[:, g, :] @ qc[b, h].astype(np.int64)    # exact integers
            s = scale * float(qs[b, h]) * ks[:, g] * dots
            w = np.exp(s - s.max())
            out[b, h] = (w @ V[:, g, :]) / w.sum()
    return out
