"""Copy-on-write on the GPU: pa_copy_blocks bit-exact against the oracle's
copy, and a parallel-sampling decode (one prompt forked into several samples
that each write into the shared, partly filled last block) against the
oracle run through the same allocator script."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import attention as OA
from oracle import cache as OC
from oracle.allocator import BlockAllocatorModel
from paged_kv_cache_283_gb300 import inputs as I
from paged_kv_cache_283_gb300 import pa

from gpu_helpers import assert_close, bf16_to_f64, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def _i64(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).cuda()


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


@pytest.mark.parametrize("layers,hkv,d", [(3, 8, 128), (1, 2, 64), (70, 1, 64)])
def test_copy_blocks_bit_exact(layers, hkv, d):
    rng = np.random.default_rng(layers + d)
    nb = 12
    ks = [rng.integers(0, 1 << 16, size=(nb, hkv, 16, d), dtype=np.uint16) for _ in range(layers)]
    vs = [rng.integers(0, 1 << 16, size=(nb, hkv, 16, d), dtype=np.uint16) for _ in range(layers)]
    pairs = np.array([[2, 7], [0, 11], [5, 5], [9, 3]], dtype=np.int64)
    want_k, want_v = OC.copy_blocks(ks, vs, pairs)
    dk = [dev_bf16(k) for k in ks]
    dv = [dev_bf16(v) for v in vs]
    pa.pa_clear_device_error()
    pa.pa_copy_blocks(dk, dv, _i64(pairs))
    torch.cuda.synchronize()
    for l in range(layers):
        assert np.array_equal(host_bits(dk[l]), want_k[l])
        assert np.array_equal(host_bits(dv[l]), want_v[l])
    assert pa.pa_get_device_error() == 0


def test_copy_blocks_rejects_bad_ids_without_writing():
    rng = np.random.default_rng(8)
    ks = [rng.integers(0, 1 << 16, size=(4, 2, 16, 64), dtype=np.uint16)]
    dk, dv = [dev_bf16(ks[0])], [dev_bf16(ks[0])]
    pa.pa_clear_device_error()
    pa.pa_copy_blocks(dk, dv, _i64([[1, 9], [-1, 2]]))
    assert pa.pa_get_device_error() == pa.PA_DEVERR_BLOCK_ID
    assert np.array_equal(host_bits(dk[0]), ks[0])
    pa.pa_clear_device_error()


@pytest.mark.parametrize("split", [None, 512])
def test_parallel_sampling_copy_on_write(split):
    # one 1000-token prompt (last block holds 8 tokens) forked into 4 samples;
    # 6 decode steps in which every sample (and the prompt's own sequence)
    # appends a token, attends, and the copies the allocator asks for are made
    rng = np.random.default_rng(283)
    hq, hkv, d, bs = 32, 8, 128, 16
    nb = 200
    order = rng.permutation(nb).astype(np.int32)
    k0 = I.normal_bf16(rng, (nb, hkv, bs, d))
    v0 = I.normal_bf16(rng, (nb, hkv, bs, d))
    model = BlockAllocatorModel(nb, bs, order)
    real = pa.BlockAllocator(nb, bs, order)
    seqs = [0, 1, 2, 3, 4]
    for a in (model, real):
        a.add_seq(0)
        a.reserve(0, 1000)
        for s in seqs[1:]:
            a.fork(0, s)
    kc_o, vc_o = k0.copy(), v0.copy()
    kc_d, vc_d = dev_bf16(k0), dev_bf16(v0)
    pa.pa_clear_device_error()
    copies = 0
    for step in range(6):
        want = model.append_slots(seqs)
        slots, src, dst = real.append_slots(seqs)
        assert [w[0] for w in want] == slots.tolist()
        assert [w[1] for w in want] == src.tolist() and [w[2] for w in want] == dst.tolist()
        pairs = np.array([[s, t] for s, t in zip(src, dst) if s >= 0], dtype=np.int64)
        copies += len(pairs)
        key = I.normal_bf16(rng, (len(seqs), hkv, d))
        val = I.normal_bf16(rng, (len(seqs), hkv, d))
        q = I.normal_bf16(rng, (len(seqs), hq, d))
        # oracle: copy, write, attend
        if len(pairs):
            (kc_o,), (vc_o,) = OC.copy_blocks([kc_o], [vc_o], pairs, inplace=True)
        kc_o, vc_o = OC.reshape_and_cache(key, val, kc_o, vc_o, slots, bs, inplace=True)
        mb = max(len(model.block_table(s)) for s in seqs)
        bt = np.full((len(seqs), mb), 0, dtype=np.int32)
        for i, s in enumerate(seqs):
            t = model.block_table(s)
            bt[i, :len(t)] = t
        ctx = np.array([model.seq_len(s) for s in seqs], dtype=np.int32)
        ref = OA.decode(q, kc_o, vc_o, bt, ctx, 1 / np.sqrt(d), bs)
        # CUDA path: the same three calls
        if len(pairs):
            pa.pa_copy_blocks([kc_d], [vc_d], _i64(pairs))
        pa.pa_reshape_and_cache(dev_bf16(key), dev_bf16(val), kc_d, vc_d, _i64(slots))
        bt_p, ctx_p = real.block_tables(seqs, mb)
        assert np.array_equal(np.where(bt_p >= 0, bt_p, 0), bt) and np.array_equal(ctx_p, ctx)
        out = torch.empty(len(seqs), hq, d, dtype=torch.bfloat16, device="cuda")
        qd = dev_bf16(q)
        if split is None:
            pa.pa_decode(out, qd, kc_d, vc_d, _i32(bt), _i32(ctx), 1 / np.sqrt(d))
        else:
            ws = pa.splitk_workspace(len(seqs), hq, d, int(ctx.max()), split)
            pa.pa_decode_splitk(*ws, qd, kc_d, vc_d, _i32(bt), _i32(ctx), 1 / np.sqrt(d),
                                partition_size=split)
            pa.pa_splitk_reduce(out, *ws, _i32(ctx), partition_size=split)
        torch.cuda.synchronize()
        assert_close(bf16_to_f64(out), ref, f"parallel sampling step {step}")
    # five sequences shared the partly filled last block: the first four to
    # write each moved to a copy, the fifth then held the original alone
    assert copies == 4
    assert np.array_equal(host_bits(kc_d), kc_o) and np.array_equal(host_bits(vc_d), vc_o)
    assert pa.pa_get_device_error() == 0
