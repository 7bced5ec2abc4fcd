"""CUDA path (libpa.so through the C ABI) against the float64 CPU oracle.

Cache writes must match bit for bit; attention outputs must pass the
tolerance gate of gpu_helpers.assert_close.  Every workload of the bench's
config list is covered at full size (sampled heads where the oracle would be
slow), plus edge-case contexts, ragged tails, block relabelling, shared vs
duplicated prefixes, split-K partition statistics and the device error word.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import attention as OA
from oracle import cache as OC
from paged_kv_cache_283_gb300 import inputs as I
from paged_kv_cache_283_gb300 import pa

from gpu_helpers import (assert_close, bf16_to_f64, both_tables, dev_bf16, host_bits,
                         model_tables)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pa.lib()
    pa.pa_clear_device_error()
    yield
    torch.cuda.synchronize()


def _dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _dev_i64(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).cuda()


def _run_decode(q, kc, vc, bt, ctx, scale, split=None):
    """pa_decode, or pa_decode_splitk(partition=split) + pa_splitk_reduce."""
    out = torch.empty_like(q)
    if split is None:
        pa.pa_decode(out, q, kc, vc, bt, ctx, scale)
    else:
        max_ctx = int(ctx.max().item()) if ctx.numel() else 0
        ws = pa.splitk_workspace(q.shape[0], q.shape[1], q.shape[2], max_ctx, split)
        pa.pa_decode_splitk(*ws, q, kc, vc, bt, ctx, scale, partition_size=split)
        pa.pa_splitk_reduce(out, *ws, ctx, partition_size=split)
    torch.cuda.synchronize()
    return out


def _assert_no_device_error():
    assert pa.pa_get_device_error() == 0


# ---------------------------------------------------------------------------
# cache write

@pytest.mark.parametrize("d,hkv", [(128, 8), (64, 2), (72, 3)])
def test_reshape_random_slots_bit_exact(d, hkv):
    rng = np.random.default_rng(d + hkv)
    nb, bs, T = 11, 16, 37
    kc = rng.integers(0, 1 << 16, size=(nb, hkv, bs, d), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(nb, hkv, bs, d), dtype=np.uint16)
    key = rng.integers(0, 1 << 16, size=(T, hkv, d), dtype=np.uint16)
    val = rng.integers(0, 1 << 16, size=(T, hkv, d), dtype=np.uint16)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[[3, 10, 36]] = -1
    want_k, want_v = OC.reshape_and_cache(key, val, kc, vc, slots, bs)
    dk, dv = dev_bf16(kc), dev_bf16(vc)
    pa.pa_reshape_and_cache(dev_bf16(key), dev_bf16(val), dk, dv, _dev_i64(slots))
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(dk), want_k)
    assert np.array_equal(host_bits(dv), want_v)
    _assert_no_device_error()


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_reshape_workload_step_bit_exact(idx):
    w = I.workload(idx)
    if idx == 4:
        bt, slots = _shared_prefix_tables(w)[:2]
    else:
        _, slots, _, slots_p = both_tables(w)
    dk, dv = dev_bf16(w.k_cache), dev_bf16(w.v_cache)
    before_k = dk.clone()
    pa.pa_reshape_and_cache(dev_bf16(w.key), dev_bf16(w.value), dk, dv, _dev_i64(slots))
    torch.cuda.synchronize()
    blk = slots // 16
    off = slots % 16
    got_k = host_bits(dk[torch.from_numpy(blk).cuda(), :, torch.from_numpy(off).cuda(), :])
    got_v = host_bits(dv[torch.from_numpy(blk).cuda(), :, torch.from_numpy(off).cuda(), :])
    assert np.array_equal(got_k, w.key) and np.array_equal(got_v, w.value)
    # every other row is untouched
    mask = torch.ones(dk.shape[0], dk.shape[2], dtype=torch.bool, device="cuda")
    mask[torch.from_numpy(blk).cuda(), torch.from_numpy(off).cuda()] = False
    a = dk.permute(0, 2, 1, 3)[mask]
    b = before_k.permute(0, 2, 1, 3)[mask]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    _assert_no_device_error()


# ---------------------------------------------------------------------------
# decode: one full step (cache write, then attention) against the oracle

def _oracle_step(w, bt, slots, kc_bits, vc_bits, q_bits, key, val, heads=None, seqs=None):
    """Oracle: write the new tokens, then attend; returns {(b): [Hq, D]}."""
    kc, vc = OC.reshape_and_cache(key, val, kc_bits, vc_bits, slots, w.block_size, inplace=True)
    out = {}
    for b in (range(w.num_seqs) if seqs is None else seqs):
        out[b] = OA.decode_sequence(q_bits[b], kc, vc, bt[b], int(w.context_lens[b]), w.scale,
                                    w.block_size, q_heads=heads)
    return out


def _gpu_step(w, bt, slots, kc_bits, vc_bits, q_bits, key, val, split=None):
    dk, dv = dev_bf16(kc_bits), dev_bf16(vc_bits)
    pa.pa_reshape_and_cache(dev_bf16(key), dev_bf16(val), dk, dv, _dev_i64(slots))
    out = _run_decode(dev_bf16(q_bits), dk, dv, _dev_i32(bt), _dev_i32(w.context_lens), w.scale,
                      split)
    return bf16_to_f64(out)


def _compare(got, ref, heads, what):
    for b, r in ref.items():
        hs = range(r.shape[0]) if heads is None else heads
        for h in hs:
            assert_close(got[b, h][None], r[h][None], f"{what} seq {b} head {h}")


@pytest.mark.parametrize("idx", [1, 2])
@pytest.mark.parametrize("split", [None, 512, 16])
def test_decode_step_full(idx, split):
    w = I.workload(idx)
    bt_m, sl_m, bt_p, sl_p = both_tables(w)
    got = _gpu_step(w, bt_p, sl_p, w.k_cache, w.v_cache, w.q, w.key, w.value, split)
    ref = _oracle_step(w, bt_m, sl_m, w.k_cache.copy(), w.v_cache.copy(), w.q, w.key, w.value)
    _compare(got, ref, None, f"workload {idx} split={split}")
    _assert_no_device_error()


@pytest.mark.parametrize("split", [512, None])
def test_decode_long_context_sampled(split):
    w = I.long_splitk()
    bt_m, sl_m, bt_p, sl_p = both_tables(w)
    got = _gpu_step(w, bt_p, sl_p, w.k_cache, w.v_cache, w.q, w.key, w.value, split)
    heads = [0, 13, 31]
    ref = _oracle_step(w, bt_m, sl_m, w.k_cache, w.v_cache, w.q, w.key, w.value, heads=heads)
    _compare(got, ref, heads, f"long-context split={split}")
    _assert_no_device_error()


def _shared_prefix_tables(w):
    """Tables / new-token slots of the shared-prefix workload, both allocators."""
    from oracle.allocator import BlockAllocatorModel
    m = BlockAllocatorModel(w.num_blocks, 16, w.free_order)
    a = pa.BlockAllocator(w.num_blocks, 16, w.free_order)
    for al in (m, a):
        al.add_seq(-1)
        al.reserve(-1, w.prefix_len)
        for b, s in enumerate(w.suffix_lens.tolist()):
            al.fork(-1, b)
            al.reserve(b, s - 1)
        al.free_seq(-1)
    sl_m = np.array([x[0] for x in m.append_slots(range(w.num_seqs))], dtype=np.int64)
    sl_p, src, _ = a.append_slots(list(range(w.num_seqs)))
    assert np.all(src == -1)  # the suffix is private: no copy-on-write
    bt_p, ctx = a.block_tables(list(range(w.num_seqs)), w.max_blocks_per_seq)
    bt_m = np.full_like(bt_p, -1)
    for b in range(w.num_seqs):
        t = m.block_table(b)
        bt_m[b, :len(t)] = t
    assert np.array_equal(bt_m, bt_p) and np.array_equal(sl_m, sl_p)
    assert np.array_equal(ctx, w.context_lens)
    return bt_p, sl_p, m


@pytest.mark.parametrize("split", [None, 512])
def test_shared_prefix_full_and_equals_duplicated(split):
    w = I.shared_prefix()
    bt, slots, _ = _shared_prefix_tables(w)
    got = _gpu_step(w, bt, slots, w.k_cache, w.v_cache, w.q, w.key, w.value, split)
    ref = _oracle_step(w, bt, slots, w.k_cache.copy(), w.v_cache.copy(), w.q, w.key, w.value)
    _compare(got, ref, None, f"shared prefix split={split}")
    # duplicated layout: every sequence owns a private copy of the prefix
    nbl = int(w.blocks_per_seq().sum())
    kd = np.empty((nbl,) + w.k_cache.shape[1:], dtype=np.uint16)
    vd = np.empty_like(kd)
    btd = np.full_like(bt, -1)
    nxt = 0
    for b in range(w.num_seqs):
        k = int(w.blocks_per_seq()[b])
        kd[nxt:nxt + k] = w.k_cache[bt[b, :k]]
        vd[nxt:nxt + k] = w.v_cache[bt[b, :k]]
        btd[b, :k] = np.arange(nxt, nxt + k)
        nxt += k
    slots_d = btd[np.arange(w.num_seqs), (w.context_lens - 1) // 16] * 16 + (w.context_lens - 1) % 16
    got_d = _gpu_step(w, btd, slots_d.astype(np.int64), kd, vd, w.q, w.key, w.value, split)
    assert np.array_equal(got, got_d)  # same arithmetic order: bit-identical
    _assert_no_device_error()


def test_32_layer_step_sampled_layers():
    w = I.llama8b_32layer_batch256()
    bt_m, sl_m, bt_p, sl_p = both_tables(w)
    base_k, base_v = dev_bf16(w.k_cache), dev_bf16(w.v_cache)
    for layer in (0, 17, 31):
        order = I.layer_block_order(w, layer)
        q, key, val = I.layer_inputs(w, layer)
        ord_dev = torch.from_numpy(order).cuda()
        dk = base_k.index_select(0, ord_dev)
        dv = base_v.index_select(0, ord_dev)
        pa.pa_reshape_and_cache(dev_bf16(key), dev_bf16(val), dk, dv, _dev_i64(sl_p))
        got = bf16_to_f64(_run_decode(dev_bf16(q), dk, dv, _dev_i32(bt_p),
                                      _dev_i32(w.context_lens), w.scale))
        ref = _oracle_step(w, bt_m, sl_m, w.k_cache[order], w.v_cache[order], q, key, val)
        _compare(got, ref, None, f"32-layer step, layer {layer}")
    _assert_no_device_error()


# ---------------------------------------------------------------------------
# edge cases and invariants

EDGE_CTX = [1, 15, 16, 17, 31, 32, 33, 127, 512, 513, 2112, 4113]


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (128, 16, 8), (128, 64, 8), (64, 4, 2),
                                      (64, 16, 4)])
@pytest.mark.parametrize("split", [None, 16, 512, 64])
def test_edge_contexts(d, hq, hkv, split):
    w = I.random_case(1000 + d + hq, len(EDGE_CTX), EDGE_CTX, hq, hkv, d)
    bt_m, sl_m, bt_p, sl_p = both_tables(w)
    got = _gpu_step(w, bt_p, sl_p, w.k_cache, w.v_cache, w.q, w.key, w.value, split)
    ref = _oracle_step(w, bt_m, sl_m, w.k_cache.copy(), w.v_cache.copy(), w.q, w.key, w.value)
    _compare(got, ref, None, f"edge d={d} hq={hq} hkv={hkv} split={split}")
    _assert_no_device_error()


@pytest.mark.parametrize("split", [None, 512])
def test_zero_length_sequence_gives_zeros(split):
    w = I.random_case(77, 3, [0, 20, 0], 8, 2, 128)
    bt, _ = model_tables(w, step_append=False)
    bt[bt < 0] = 0
    out = _run_decode(dev_bf16(w.q), dev_bf16(w.k_cache), dev_bf16(w.v_cache), _dev_i32(bt),
                      _dev_i32(w.context_lens), w.scale, split)
    got = bf16_to_f64(out)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    ref = OA.decode_sequence(w.q[1], w.k_cache, w.v_cache, bt[1], 20, w.scale, 16)
    assert_close(got[1], ref, "ctx 20 next to empty sequences")
    _assert_no_device_error()


@pytest.mark.parametrize("split", [None, 512])
def test_block_relabelling_is_bit_identical(split):
    w = I.random_case(88, 5, [700, 1, 16, 2049, 333], 32, 8, 128)
    bt, _ = model_tables(w, step_append=False)
    out1 = _run_decode(dev_bf16(w.q), dev_bf16(w.k_cache), dev_bf16(w.v_cache), _dev_i32(bt),
                       _dev_i32(w.context_lens), w.scale, split)
    perm = np.random.default_rng(89).permutation(w.num_blocks)
    kp = np.empty_like(w.k_cache)
    vp = np.empty_like(w.v_cache)
    kp[perm] = w.k_cache
    vp[perm] = w.v_cache
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2 = _run_decode(dev_bf16(w.q), dev_bf16(kp), dev_bf16(vp), _dev_i32(bt2),
                       _dev_i32(w.context_lens), w.scale, split)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    ref = OA.decode(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.scale, 16)
    assert_close(bf16_to_f64(out1), ref, "relabelled pool")


def test_splitk_partition_statistics():
    w = I.random_case(99, 3, [1500, 512, 37], 32, 8, 128)
    bt, _ = model_tables(w, step_append=False)
    q, kc, vc = dev_bf16(w.q), dev_bf16(w.k_cache), dev_bf16(w.v_cache)
    ws_o, ws_m, ws_l = pa.splitk_workspace(3, 32, 128, 1500, 512)
    pa.pa_decode_splitk(ws_o, ws_m, ws_l, q, kc, vc, _dev_i32(bt), _dev_i32(w.context_lens),
                        w.scale, partition_size=512)
    torch.cuda.synchronize()
    o, m, l = ws_o.cpu().numpy(), ws_m.cpu().numpy(), ws_l.cpu().numpy()
    for b, n in enumerate(w.context_lens.tolist()):
        rm, rl, ro = OA.partition_stats(w.q[b], w.k_cache, w.v_cache, bt[b], n, w.scale, 16, 512)
        np_ = rm.shape[1]
        np.testing.assert_allclose(m[b, :, :np_], rm, rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(l[b, :, :np_], rl, rtol=1e-4)
        assert_close(o[b, :, :np_], ro, f"partition outputs seq {b}")
    _assert_no_device_error()


def test_device_error_word_reports_bad_indices():
    w = I.random_case(5, 2, [40, 20], 8, 2, 64)
    bt, _ = model_tables(w, step_append=False)
    q, kc, vc = dev_bf16(w.q), dev_bf16(w.k_cache), dev_bf16(w.v_cache)
    pa.pa_clear_device_error()
    bad = bt.copy()
    bad[0, 1] = w.num_blocks + 5             # outside the pool: read as block 0
    out = torch.empty_like(q)
    pa.pa_decode(out, q, kc, vc, _dev_i32(bad), _dev_i32(w.context_lens), w.scale)
    assert pa.pa_get_device_error() == pa.PA_DEVERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    pa.pa_clear_device_error()
    long_ctx = np.array([40, bt.shape[1] * 16 + 50], dtype=np.int32)   # beyond the table
    full = np.where(bt >= 0, bt, 0)      # padding made valid: only the length is wrong
    pa.pa_decode(out, q, kc, vc, _dev_i32(full), _dev_i32(long_ctx), w.scale)
    assert pa.pa_get_device_error() == pa.PA_DEVERR_CONTEXT_LEN
    pa.pa_clear_device_error()
    slots = np.array([3, w.num_blocks * 16 + 7], dtype=np.int64)      # second one out of range
    key = dev_bf16(w.key)
    before = host_bits(kc)
    pa.pa_reshape_and_cache(key, dev_bf16(w.value), kc, vc, _dev_i64(slots))
    assert pa.pa_get_device_error() == pa.PA_DEVERR_SLOT
    after = host_bits(kc)
    assert np.array_equal(after[0, :, 3], w.key[0])
    after[0, :, 3] = before[0, :, 3]
    assert np.array_equal(after, before)
    pa.pa_clear_device_error()
    assert pa.pa_get_device_error() == 0


def test_binding_rejects_cpu_tensors():
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pa.pa_decode(q, q, torch.zeros(1, 2, 16, 64, dtype=torch.bfloat16),
                     torch.zeros(1, 2, 16, 64, dtype=torch.bfloat16),
                     torch.zeros(1, 1, dtype=torch.int32), torch.ones(1, dtype=torch.int32), 1.0)


@pytest.mark.parametrize("case", ["many_seqs", "long_partition"])
def test_splitk_large_batch_and_long_partitions(case):
    # A batch of 1100 short sequences, and partitions of 512 blocks.
    if case == "many_seqs":
        rng = np.random.default_rng(3030)
        ctx = rng.integers(1, 80, size=1100)
        w = I.random_case(3031, 1100, ctx, 8, 2, 64)
        split = 32
    else:
        w = I.random_case(3032, 3, [9000, 4100, 17], 16, 8, 128)
        split = 8192
    bt_m, sl_m, bt_p, sl_p = both_tables(w)
    got = _gpu_step(w, bt_p, sl_p, w.k_cache, w.v_cache, w.q, w.key, w.value, split)
    ref = _oracle_step(w, bt_m, sl_m, w.k_cache.copy(), w.v_cache.copy(), w.q, w.key, w.value)
    _compare(got, ref, None, f"split-K ({case})")
    _assert_no_device_error()


@pytest.mark.parametrize("split", [16, 48, 256])
def test_splitk_schedule_mixes(split):
    # Many small and a few long sequences: partial partitions of every size,
    # sequences with no full partition, and an empty one.
    rng = np.random.default_rng(split)
    ctx = np.concatenate([rng.integers(1, 40, size=60), rng.integers(1000, 3000, size=6), [0]])
    w = I.random_case(5000 + split, len(ctx), ctx, 32, 8, 128)
    bt, _ = model_tables(w, step_append=False)
    bt[bt < 0] = 0
    out = _run_decode(dev_bf16(w.q), dev_bf16(w.k_cache), dev_bf16(w.v_cache), _dev_i32(bt),
                      _dev_i32(w.context_lens), w.scale, split)
    ref = OA.decode(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.scale, 16)
    assert_close(bf16_to_f64(out), ref, f"schedule mix, partition {split}")
    _assert_no_device_error()


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("split", [False, True])
def test_decode_step_object_matches_oracle(split, fused):
    # pa.DecodeStep: the same cache write + attention with pre-marshalled
    # calls; called twice with new inputs written into the same buffers
    w = I.random_case(777, 6, [300, 17, 1, 2049, 512, 96], 32, 8, 128)
    bt_m, sl_m, bt_p, sl_p = both_tables(w)
    kc, vc = dev_bf16(w.k_cache), dev_bf16(w.v_cache)
    key, val, q = dev_bf16(w.key), dev_bf16(w.value), dev_bf16(w.q)
    slots, bt, ctx = _dev_i64(sl_p), _dev_i32(bt_p), _dev_i32(w.context_lens)
    out = torch.empty_like(q)
    step = pa.DecodeStep(key, val, kc, vc, slots, q, bt, ctx, out, w.scale, split=split,
                         partition_size=256, max_context_len=int(w.context_lens.max()),
                         fused=fused)
    kc_o, vc_o = w.k_cache.copy(), w.v_cache.copy()
    rng = np.random.default_rng(778)
    for it in range(2):
        if it == 1:
            nk, nv, nq = (I.normal_bf16(rng, w.key.shape), I.normal_bf16(rng, w.value.shape),
                          I.normal_bf16(rng, w.q.shape))
            key.copy_(dev_bf16(nk))
            val.copy_(dev_bf16(nv))
            q.copy_(dev_bf16(nq))
        else:
            nk, nv, nq = w.key, w.value, w.q
        step()
        torch.cuda.synchronize()
        kc_o, vc_o = OC.reshape_and_cache(nk, nv, kc_o, vc_o, sl_m, 16, inplace=True)
        ref = OA.decode(nq, kc_o, vc_o, bt_m, w.context_lens, w.scale, 16)
        assert_close(bf16_to_f64(out), ref, f"DecodeStep split={split} fused={fused} call {it}")
    _assert_no_device_error()


@pytest.mark.parametrize("kv_len_case", ["mixed", "long"])
def test_decode_step_object_auto_partition_and_order(kv_len_case):
    # pa.DecodeStep with partition_size=None and the host lengths: the fused
    # step picks its partition size and a longest-first order
    lens = [300, 17, 1, 2049, 512, 96] if kv_len_case == "mixed" else [9000, 40, 4100, 700]
    w = I.random_case(779 + len(lens), len(lens), lens, 32, 8, 128)
    bt_m, sl_m, bt_p, sl_p = both_tables(w)
    kc, vc = dev_bf16(w.k_cache), dev_bf16(w.v_cache)
    key, val, q = dev_bf16(w.key), dev_bf16(w.value), dev_bf16(w.q)
    out = torch.empty_like(q)
    step = pa.DecodeStep(key, val, kc, vc, _dev_i64(sl_p), q, _dev_i32(bt_p),
                         _dev_i32(w.context_lens), out, w.scale, partition_size=None,
                         host_context_lens=w.context_lens)
    assert step.partition_size in (256, 384, 512, 640, 768, 1024, 1536, 2048, 4096)
    step()
    torch.cuda.synchronize()
    kc_o, vc_o = OC.reshape_and_cache(w.key, w.value, w.k_cache.copy(), w.v_cache.copy(), sl_m,
                                      16, inplace=True)
    ref = OA.decode(w.q, kc_o, vc_o, bt_m, w.context_lens, w.scale, 16)
    assert_close(bf16_to_f64(out), ref, f"DecodeStep auto ({kv_len_case})")
    _assert_no_device_error()
