"""FP8 (E4M3) KV cache on the GPU: the quantising cache write bit-exact against
the oracle's codes and scales, and FP8 decode (whole-sequence and split-K)
within the parity tolerance of the oracle's FP8 decode, including pools whose
bytes past each context are NaN codes."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import fp8 as OF
from paged_kv_cache_283_gb300 import inputs as I
from paged_kv_cache_283_gb300 import pa

from gpu_helpers import assert_close, bf16_to_f64, both_tables, dev_bf16, v_pool_logical, v_pool_stored

pytestmark = pytest.mark.gpu


def _i64(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).cuda()


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _dev_pools(kq, vq, ks, vs):
    """Device pools from logical codes (V goes to its storage order)."""
    return (torch.from_numpy(kq).cuda(), torch.from_numpy(v_pool_stored(vq, True)).cuda(),
            torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda())


@pytest.mark.parametrize("d", [128, 64])
def test_fp8_cache_write_bit_exact(d):
    rng = np.random.default_rng(d + 1)
    nb, hkv, T = 9, 4, 30
    key = I.normal_bf16(rng, (T, hkv, d))
    val = I.normal_bf16(rng, (T, hkv, d))
    key[3] = 0                                   # an all-zero row: scale 0
    big = I.f32_to_bf16_bits((rng.standard_normal((hkv, d)) * 1e4).astype(np.float32))
    val[7] = big                                 # large values: scale >> 1
    kq = rng.integers(0, 256, size=(nb, hkv, 16, d)).astype(np.uint8)
    vq = rng.integers(0, 256, size=(nb, hkv, 16, d)).astype(np.uint8)
    ks = rng.standard_normal((nb, hkv, 16)).astype(np.float32)
    vs = rng.standard_normal((nb, hkv, 16)).astype(np.float32)
    slots = rng.choice(nb * 16, size=T, replace=False).astype(np.int64)
    slots[[5, 11]] = -1
    want = OF.reshape_and_cache_fp8(key, val, kq, vq, ks, vs, slots, 16)
    dk, dv, dks, dvs = _dev_pools(kq, vq, ks, vs)
    pa.pa_clear_device_error()
    pa.pa_reshape_and_cache_fp8(dev_bf16(key), dev_bf16(val), dk, dv, dks, dvs, _i64(slots))
    torch.cuda.synchronize()
    got = (dk.cpu().numpy(), v_pool_logical(dv.cpu().numpy(), True), dks.cpu().numpy(),
           dvs.cpu().numpy())
    for g, exp in zip(got, want):
        assert np.array_equal(g, exp)
    assert pa.pa_get_device_error() == 0


def _fp8_step(w, split, nan_tail=False):
    bt_m, sl_m, bt_p, sl_p = both_tables(w)
    kq, ks = OF.quantize_fp8(w.k_cache)
    vq, vs = OF.quantize_fp8(w.v_cache)
    if nan_tail:
        # every position past a sequence's context holds NaN codes and NaN scales
        for b, c in enumerate(w.context_lens.tolist()):
            c_after = c  # the new token sits at c - 1
            blk = bt_m[b][(c_after - 1) // 16]
            off = c_after % 16
            if off:
                kq[blk, :, off:, :] = 0x7F
                vq[blk, :, off:, :] = 0xFF
                ks[blk, :, off:] = np.nan
                vs[blk, :, off:] = np.nan
    dk, dv, dks, dvs = _dev_pools(kq, vq, ks, vs)
    pa.pa_reshape_and_cache_fp8(dev_bf16(w.key), dev_bf16(w.value), dk, dv, dks, dvs, _i64(sl_p))
    q = dev_bf16(w.q)
    out = torch.empty_like(q)
    bt, ctx = _i32(bt_p), _i32(w.context_lens)
    if split is None:
        pa.pa_decode_fp8(out, q, dk, dv, dks, dvs, bt, ctx, w.scale)
    else:
        ws = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim,
                                 int(w.context_lens.max()), split)
        pa.pa_decode_splitk_fp8(*ws, q, dk, dv, dks, dvs, bt, ctx, w.scale, partition_size=split)
        pa.pa_splitk_reduce(out, *ws, ctx, partition_size=split)
    torch.cuda.synchronize()
    kq2, vq2, ks2, vs2 = OF.reshape_and_cache_fp8(w.key, w.value, kq, vq, ks, vs, sl_m, 16)
    ref = OF.decode_fp8(w.q, kq2, vq2, ks2, vs2, bt_m, w.context_lens, w.scale, 16)
    return bf16_to_f64(out), ref


@pytest.mark.parametrize("idx", [1, 2])
@pytest.mark.parametrize("split", [None, 512, 16])
def test_fp8_decode_step(idx, split):
    w = I.workload(idx)
    pa.pa_clear_device_error()
    got, ref = _fp8_step(w, split)
    assert_close(got, ref, f"fp8 workload {idx} split={split}")
    assert pa.pa_get_device_error() == 0


EDGE = [1, 15, 16, 17, 33, 512, 513, 2112]


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (128, 16, 8), (128, 64, 8), (64, 4, 2),
                                      (64, 16, 4)])
@pytest.mark.parametrize("split", [None, 64])
def test_fp8_edge_contexts_nan_tail(d, hq, hkv, split):
    w = I.random_case(3000 + d + hq, len(EDGE), EDGE, hq, hkv, d)
    pa.pa_clear_device_error()
    got, ref = _fp8_step(w, split, nan_tail=True)
    assert_close(got, ref, f"fp8 edge d={d} hq={hq} split={split}")
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (128, 64, 8), (64, 4, 2)])
@pytest.mark.parametrize("split", [None, 64])
def test_fp8_q_magnitudes(d, hq, hkv, split):
    """q heads far outside f16's range (|q| ~ 1e5 and ~ 1e-6), an all-zero head
    and a head whose elements span 1e-3 .. 1e3: the scores must keep their
    relative precision whatever the magnitude of q."""
    w = I.random_case(4000 + d + hq, len(EDGE), EDGE, hq, hkv, d)
    rng = np.random.default_rng(d + hq)
    q = (w.q.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    q[:, 0::4] *= 1e5
    q[:, 1::4] *= 1e-6
    q[:, 2] = 0.0
    q[:, 3::4] *= 10.0 ** rng.uniform(-3, 3, size=q[:, 3::4].shape)
    w.q = I.f32_to_bf16_bits(q.astype(np.float32))
    pa.pa_clear_device_error()
    got, ref = _fp8_step(w, split)
    assert_close(got, ref, f"fp8 q magnitudes d={d} hq={hq} split={split}")
    assert pa.pa_get_device_error() == 0
