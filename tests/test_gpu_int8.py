"""INT8 KV cache on the GPU: the quantising cache write bit-exact against the
oracle's codes and scales, and INT8 decode (whole-sequence and split-K)
within the parity tolerance of the oracle's INT8 decode."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import quant as OQ
from paged_kv_cache_283_gb300 import inputs as I
from paged_kv_cache_283_gb300 import pa

from gpu_helpers import (assert_close, bf16_to_f64, both_tables, dev_bf16, model_tables,
                         v_pool_logical, v_pool_stored)

pytestmark = pytest.mark.gpu


def _i64(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).cuda()


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _pools(w, rng):
    """INT8 pools holding the workload's K/V, quantised by the oracle."""
    kq, ks = OQ.quantize_int8(w.k_cache)
    vq, vs = OQ.quantize_int8(w.v_cache)
    return kq, vq, ks, vs


def _dev_pools(kq, vq, ks, vs):
    """Device pools from logical codes (V goes to its storage order)."""
    return (torch.from_numpy(kq).cuda(), torch.from_numpy(v_pool_stored(vq, False)).cuda(),
            torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda())


@pytest.mark.parametrize("d", [128, 64])
def test_int8_cache_write_bit_exact(d):
    rng = np.random.default_rng(d)
    nb, hkv, T = 9, 4, 30
    key = I.normal_bf16(rng, (T, hkv, d))
    val = I.normal_bf16(rng, (T, hkv, d))
    key[3] = 0                                   # an all-zero row: scale 0
    kq = rng.integers(-128, 128, size=(nb, hkv, 16, d), dtype=np.int8)
    vq = rng.integers(-128, 128, size=(nb, hkv, 16, d), dtype=np.int8)
    ks = rng.standard_normal((nb, hkv, 16)).astype(np.float32)
    vs = rng.standard_normal((nb, hkv, 16)).astype(np.float32)
    slots = rng.choice(nb * 16, size=T, replace=False).astype(np.int64)
    slots[[5, 11]] = -1
    want = OQ.reshape_and_cache_int8(key, val, kq, vq, ks, vs, slots, 16)
    dk, dv, dks, dvs = _dev_pools(kq, vq, ks, vs)
    pa.pa_clear_device_error()
    pa.pa_reshape_and_cache_int8(dev_bf16(key), dev_bf16(val), dk, dv, dks, dvs, _i64(slots))
    torch.cuda.synchronize()
    got = (dk.cpu().numpy(), v_pool_logical(dv.cpu().numpy(), False), dks.cpu().numpy(),
           dvs.cpu().numpy())
    for g, exp in zip(got, want):
        assert np.array_equal(g, exp)
    assert pa.pa_get_device_error() == 0


def _int8_step(w, split, rng):
    bt_m, sl_m, bt_p, sl_p = both_tables(w)
    kq, vq, ks, vs = _pools(w, rng)
    dk, dv, dks, dvs = _dev_pools(kq, vq, ks, vs)
    pa.pa_reshape_and_cache_int8(dev_bf16(w.key), dev_bf16(w.value), dk, dv, dks, dvs,
                                 _i64(sl_p))
    q = dev_bf16(w.q)
    out = torch.empty_like(q)
    bt, ctx = _i32(bt_p), _i32(w.context_lens)
    if split is None:
        pa.pa_decode_int8(out, q, dk, dv, dks, dvs, bt, ctx, w.scale)
    else:
        ws = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim,
                                 int(w.context_lens.max()), split)
        pa.pa_decode_splitk_int8(*ws, q, dk, dv, dks, dvs, bt, ctx, w.scale,
                                 partition_size=split)
        pa.pa_splitk_reduce(out, *ws, ctx, partition_size=split)
    torch.cuda.synchronize()
    kq2, vq2, ks2, vs2 = OQ.reshape_and_cache_int8(w.key, w.value, kq, vq, ks, vs, sl_m, 16)
    ref = OQ.decode_int8(w.q, kq2, vq2, ks2, vs2, bt_m, w.context_lens, w.scale, 16)
    return bf16_to_f64(out), ref


@pytest.mark.parametrize("idx", [1, 2])
@pytest.mark.parametrize("split", [None, 512, 16])
def test_int8_decode_step(idx, split):
    w = I.workload(idx)
    got, ref = _int8_step(w, split, np.random.default_rng(idx))
    assert_close(got, ref, f"int8 workload {idx} split={split}")
    assert pa.pa_get_device_error() == 0


EDGE = [1, 15, 16, 17, 33, 512, 513, 2112]


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (128, 16, 8), (128, 64, 8), (64, 4, 2),
                                      (64, 16, 4)])
@pytest.mark.parametrize("split", [None, 64])
def test_int8_edge_contexts(d, hq, hkv, split):
    w = I.random_case(2000 + d + hq, len(EDGE), EDGE, hq, hkv, d)
    got, ref = _int8_step(w, split, np.random.default_rng(d + hq))
    assert_close(got, ref, f"int8 edge d={d} hq={hq} split={split}")
    assert pa.pa_get_device_error() == 0
