"""The fused decode step (pa_decode_step, _int8, _fp8: cache write + decode +
split-K merge in one launch) against the float64 oracle: the pools after the
call bit-exact against the oracle's cache write, the outputs within the
parity tolerance of the oracle's decode over the written cache.  Also: padding
slots, empty sequences, a slot that is not its sequence's position (refused,
PA_DEVERR_SLOT), attention without a write, the arrival counters left at zero,
and repeated calls."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import attention as OA
from oracle import cache as OC
from oracle import fp8 as OF
from oracle import quant as OQ
from paged_kv_cache_283_gb300 import inputs as I
from paged_kv_cache_283_gb300 import pa

from gpu_helpers import assert_close, bf16_to_f64, both_tables, dev_bf16, host_bits, \
    v_pool_logical, v_pool_stored

pytestmark = pytest.mark.gpu


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _i64(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).cuda()


class _Case:
    """One workload on both sides: oracle pools (numpy) and device pools."""

    def __init__(self, w, kv):
        self.w, self.kv = w, kv
        self.bt_m, self.sl_m, self.bt_p, self.sl_p = both_tables(w)
        if kv == "bf16":
            self.host = [w.k_cache.copy(), w.v_cache.copy()]
            self.dev = [dev_bf16(w.k_cache), dev_bf16(w.v_cache)]
        else:
            quant = OF.quantize_fp8 if kv == "fp8" else OQ.quantize_int8
            kq, ks = quant(w.k_cache)
            vq, vs = quant(w.v_cache)
            self.host = [kq, vq, ks, vs]
            self.dev = [torch.from_numpy(kq).cuda(), torch.from_numpy(v_pool_stored(vq, kv == "fp8")).cuda(),
                        torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()]

    def oracle_write(self, key, val, slots):
        w = self.w
        if self.kv == "bf16":
            self.host = list(OC.reshape_and_cache(key, val, self.host[0], self.host[1], slots,
                                                  w.block_size))
        else:
            write = OF.reshape_and_cache_fp8 if self.kv == "fp8" else OQ.reshape_and_cache_int8
            self.host = list(write(key, val, *self.host, slots, w.block_size))

    def oracle_decode(self, q, ctx=None):
        w = self.w
        ctx = w.context_lens if ctx is None else ctx
        if self.kv == "bf16":
            return OA.decode(q, self.host[0], self.host[1], self.bt_m, ctx, w.scale,
                             w.block_size)
        dec = OF.decode_fp8 if self.kv == "fp8" else OQ.decode_int8
        return dec(q, *self.host, self.bt_m, ctx, w.scale, w.block_size)

    def device_pools(self):
        """Device pools in the oracle's (logical) layout, for bit comparison."""
        if self.kv == "bf16":
            return [host_bits(self.dev[0]), host_bits(self.dev[1])]
        return [self.dev[0].cpu().numpy(), v_pool_logical(self.dev[1].cpu().numpy(), self.kv == "fp8"),
                self.dev[2].cpu().numpy(), self.dev[3].cpu().numpy()]

    def run(self, q, key, val, slots, split, ctx=None, counters=None, workspace=None):
        w = self.w
        out = torch.empty_like(q)
        ctx_d = _i32(w.context_lens if ctx is None else ctx)
        kw = {}
        if self.kv != "bf16":
            kw = {"k_scales": self.dev[2], "v_scales": self.dev[3]}
        if split:
            if workspace is None:
                workspace = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim,
                                                max(1, int(w.context_lens.max())), split)
            if counters is None:
                counters = pa.step_counters(w.num_seqs, w.num_kv_heads)
        pa.pa_decode_step(out, q, self.dev[0], self.dev[1], _i32(self.bt_p), ctx_d, w.scale,
                          key=key, value=val, slot_mapping=slots, partition_size=split or 0,
                          workspace=workspace, counters=counters, **kw)
        torch.cuda.synchronize()
        return out, counters


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("idx", [1, 2])
@pytest.mark.parametrize("split", [0, 512, 128, 16])
def test_fused_step_matches_oracle(kv, idx, split):
    """split 512 and 128 (at most 16 partitions): merged in the launch; split
    16 (up to 128 partitions): merged by a second launch."""
    w = I.workload(idx)
    c = _Case(w, kv)
    pa.pa_clear_device_error()
    out, counters = c.run(dev_bf16(w.q), dev_bf16(w.key), dev_bf16(w.value), _i64(c.sl_p), split)
    c.oracle_write(w.key, w.value, c.sl_m)
    for got, want in zip(c.device_pools(), c.host):
        assert np.array_equal(got, want), "pool bytes after the fused cache write"
    assert_close(bf16_to_f64(out), c.oracle_decode(w.q), f"fused {kv} workload {idx} split={split}")
    if split:
        assert int(counters.abs().sum().item()) == 0, "arrival counters left nonzero"
    assert pa.pa_get_device_error() == 0


EDGE = [1, 15, 16, 17, 33, 512, 513, 2112]


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (128, 64, 8), (64, 4, 2)])
@pytest.mark.parametrize("split", [0, 256, 64])
def test_fused_step_edges(kv, d, hq, hkv, split):
    """Edge contexts (one token, block and partition boundaries) with some
    sequences' slots as padding (-1): those keep the pool's old row."""
    w = I.random_case(6000 + d + hq, len(EDGE), EDGE, hq, hkv, d)
    c = _Case(w, kv)
    slots_m = c.sl_m.copy()
    slots_m[[1, 5]] = -1
    slots_p = c.sl_p.copy()
    slots_p[[1, 5]] = -1
    pa.pa_clear_device_error()
    out, counters = c.run(dev_bf16(w.q), dev_bf16(w.key), dev_bf16(w.value), _i64(slots_p), split)
    c.oracle_write(w.key, w.value, slots_m)
    for got, want in zip(c.device_pools(), c.host):
        assert np.array_equal(got, want)
    assert_close(bf16_to_f64(out), c.oracle_decode(w.q), f"fused edges {kv} d={d} split={split}")
    if split:
        assert int(counters.abs().sum().item()) == 0
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("split", [0, 48])
def test_fused_step_empty_sequences_and_no_write(split):
    """Empty sequences give zeros; with no key / value / slots the call is a
    plain decode and the pools are untouched."""
    ctx = np.array([0, 40, 0, 200, 7], dtype=np.int32)
    w = I.random_case(6100 + split, len(ctx), np.maximum(ctx, 1), 16, 4, 128)
    c = _Case(w, "bf16")
    before = [x.copy() for x in c.host]
    pa.pa_clear_device_error()
    out, counters = c.run(dev_bf16(w.q), None, None, None, split, ctx=ctx)
    for got, want in zip(c.device_pools(), before):
        assert np.array_equal(got, want), "a call without a write changed the pools"
    ref = c.oracle_decode(w.q, ctx)
    assert np.all(ref[ctx == 0] == 0)
    assert_close(bf16_to_f64(out), ref, f"fused empty/no-write split={split}")
    if split:
        assert int(counters.abs().sum().item()) == 0
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("split", [0, 64])
def test_fused_step_refuses_foreign_slot(split):
    """A slot that is not its sequence's position n - 1 is not written and
    raises PA_DEVERR_SLOT; the other sequences are unaffected."""
    w = I.random_case(6200, 4, [100, 300, 17, 64], 32, 8, 128)
    c = _Case(w, "bf16")
    slots_p = c.sl_p.copy()
    slots_m = c.sl_m.copy()
    slots_p[2] = slots_p[0] + 1 if slots_p[0] % 16 != 15 else slots_p[0] - 1  # another position
    slots_m[2] = -1  # the oracle: sequence 2's new token is not written
    pa.pa_clear_device_error()
    out, _ = c.run(dev_bf16(w.q), dev_bf16(w.key), dev_bf16(w.value), _i64(slots_p), split)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_SLOT
    pa.pa_clear_device_error()
    c.oracle_write(w.key, w.value, slots_m)
    for got, want in zip(c.device_pools(), c.host):
        assert np.array_equal(got, want)
    assert_close(bf16_to_f64(out), c.oracle_decode(w.q), f"foreign slot split={split}")


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_fused_step_repeated_calls(kv):
    """Three calls on the same buffers (counters and workspace reused): each
    writes its token and attends over the cache as the oracle has it then."""
    w = I.random_case(6300, 6, [300, 17, 1, 2049, 512, 96], 32, 8, 128)
    c = _Case(w, kv)
    ws = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim, int(w.context_lens.max()), 256)
    counters = pa.step_counters(w.num_seqs, w.num_kv_heads)
    rng = np.random.default_rng(6301)
    key, val, q = dev_bf16(w.key), dev_bf16(w.value), dev_bf16(w.q)
    slots = _i64(c.sl_p)
    pa.pa_clear_device_error()
    for it in range(3):
        nk, nv, nq = (w.key, w.value, w.q) if it == 0 else (
            I.normal_bf16(rng, w.key.shape), I.normal_bf16(rng, w.value.shape),
            I.normal_bf16(rng, w.q.shape))
        key.copy_(dev_bf16(nk))
        val.copy_(dev_bf16(nv))
        q.copy_(dev_bf16(nq))
        out, _ = c.run(q, key, val, slots, 256, counters=counters, workspace=ws)
        c.oracle_write(nk, nv, c.sl_m)
        assert_close(bf16_to_f64(out), c.oracle_decode(nq), f"fused {kv} call {it}")
        assert int(counters.abs().sum().item()) == 0
    assert pa.pa_get_device_error() == 0


def test_fused_step_long_context_matches_separate_kernels():
    """The long-context workload (8K..128K tokens, up to 256 partitions, so
    the merge is a second launch) against pa_decode_splitk + pa_splitk_reduce
    on the same written cache (that path is pinned to the oracle elsewhere)."""
    w = I.long_splitk()
    bt_m, sl_m, bt_p, sl_p = both_tables(w)
    kc, vc = dev_bf16(w.k_cache), dev_bf16(w.v_cache)
    q, key, val = dev_bf16(w.q), dev_bf16(w.key), dev_bf16(w.value)
    bt, ctx, slots = _i32(bt_p), _i32(w.context_lens), _i64(sl_p)
    ws = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim, int(w.context_lens.max()), 512)
    counters = pa.step_counters(w.num_seqs, w.num_kv_heads)
    pa.pa_clear_device_error()
    out = torch.empty_like(q)
    pa.pa_decode_step(out, q, kc, vc, bt, ctx, w.scale, key=key, value=val, slot_mapping=slots,
                      partition_size=512, workspace=ws, counters=counters)
    ref = torch.empty_like(q)
    pa.pa_decode_splitk(*ws, q, kc, vc, bt, ctx, w.scale, partition_size=512)
    pa.pa_splitk_reduce(ref, *ws, ctx, partition_size=512)
    torch.cuda.synchronize()
    a, b = out.float(), ref.float()
    assert torch.all((a - b).abs() <= 2.0 ** -7 * b.abs() + 1e-6), "fused vs separate merge"
    # and the written rows are the new tokens
    kh = host_bits(kc)
    for bi, si in enumerate(sl_p):
        assert np.array_equal(kh[si // 16, :, si % 16], w.key[bi])
    assert int(counters.abs().sum().item()) == 0
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("kind", ["longest", "random", "stale"])
@pytest.mark.parametrize("split", [256, 64])
def test_fused_step_work_order(kind, split):
    """A split-K launch in a given work order (pa_splitk_order's longest-first,
    a random permutation, or the order made for other context lengths) gives
    the same attention: every item runs whatever the order."""
    w = I.random_case(6400 + split, len(EDGE), EDGE, 32, 8, 128)
    c = _Case(w, "bf16")
    maxp = -(-int(w.context_lens.max()) // split)
    if kind == "longest":
        order = pa.splitk_order(w.context_lens, split, maxp)
    elif kind == "random":
        order = np.random.default_rng(split).permutation(w.num_seqs * maxp).astype(np.int32)
    else:
        other = np.random.default_rng(7).integers(0, 3000, size=w.num_seqs).astype(np.int32)
        order = pa.splitk_order(other, split, maxp)
    ws = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim, int(w.context_lens.max()),
                             split)
    counters = pa.step_counters(w.num_seqs, w.num_kv_heads)
    q = dev_bf16(w.q)
    out = torch.empty_like(q)
    pa.pa_clear_device_error()
    pa.pa_decode_step(out, q, c.dev[0], c.dev[1], _i32(c.bt_p), _i32(w.context_lens), w.scale,
                      key=dev_bf16(w.key), value=dev_bf16(w.value), slot_mapping=_i64(c.sl_p),
                      partition_size=split, workspace=ws, counters=counters,
                      order=_i32(order))
    torch.cuda.synchronize()
    c.oracle_write(w.key, w.value, c.sl_m)
    for got, want in zip(c.device_pools(), c.host):
        assert np.array_equal(got, want)
    assert_close(bf16_to_f64(out), c.oracle_decode(w.q), f"order {kind} split={split}")
    assert int(counters.abs().sum().item()) == 0
    assert pa.pa_get_device_error() == 0


def test_fused_step_order_entry_out_of_range():
    """An order entry outside [0, B * max_partitions) sets PA_DEVERR_ORDER and
    its CTA does nothing (no wait, no fault)."""
    w = I.random_case(6500, 4, [100, 300, 17, 64], 32, 8, 128)
    c = _Case(w, "bf16")
    split = 64
    maxp = -(-int(w.context_lens.max()) // split)
    order = pa.splitk_order(w.context_lens, split, maxp)
    order[-1] = w.num_seqs * maxp + 5
    ws = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim, int(w.context_lens.max()),
                             split)
    counters = pa.step_counters(w.num_seqs, w.num_kv_heads)
    q = dev_bf16(w.q)
    out = torch.empty_like(q)
    pa.pa_clear_device_error()
    pa.pa_decode_step(out, q, c.dev[0], c.dev[1], _i32(c.bt_p), _i32(w.context_lens), w.scale,
                      partition_size=split, workspace=ws, counters=counters, order=_i32(order))
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() & pa.PA_DEVERR_ORDER
    # the displaced item never arrived, so a counter may be left nonzero:
    # recovery re-zeroes them, and the next call (valid order, same counters
    # and workspace) is exact again
    assert pa.recover_step_counters(counters) & pa.PA_DEVERR_ORDER
    assert int(counters.abs().sum().item()) == 0 and pa.pa_get_device_error() == 0
    good = _i32(pa.splitk_order(w.context_lens, split, maxp))
    pa.pa_decode_step(out, q, c.dev[0], c.dev[1], _i32(c.bt_p), _i32(w.context_lens), w.scale,
                      partition_size=split, workspace=ws, counters=counters, order=good)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert_close(bf16_to_f64(out), c.oracle_decode(w.q), "call after recovering the counters")
    assert int(counters.abs().sum().item()) == 0


def test_decode_step_object_contexts_grow_past_the_first_plan():
    """DecodeStep with partition_size=None plans its partition size and order
    from the first call's contexts (4 sequences of at most 100 tokens: one
    256-token partition each), but its workspace and order cover the block
    tables' capacity (1024 tokens), so later calls whose contexts grow to 3
    and 4 partitions stay exact.  Each call appends one token per sequence
    (after reserving the positions skipped) and is checked against the
    oracle."""
    from oracle.allocator import BlockAllocatorModel
    nb, hkv, hq, d, cap = 320, 8, 32, 128, 64
    rng = np.random.default_rng(6700)
    free = rng.permutation(nb).astype(np.int32)
    kc_h = I.normal_bf16(rng, (nb, hkv, 16, d))
    vc_h = I.normal_bf16(rng, (nb, hkv, 16, d))
    plan_ctx = [[40, 17, 100, 64], [300, 18, 600, 65], [700, 19, 1024, 300]]
    a = pa.BlockAllocator(nb, 16, free)
    m = BlockAllocatorModel(nb, 16, free)
    B = len(plan_ctx[0])
    for al in (a, m):
        for b in range(B):
            al.add_seq(b)
    kc, vc = dev_bf16(kc_h), dev_bf16(vc_h)
    q = torch.empty(B, hq, d, dtype=torch.bfloat16, device="cuda")
    key = torch.empty(B, hkv, d, dtype=torch.bfloat16, device="cuda")
    val = torch.empty_like(key)
    out = torch.empty_like(q)
    bt_d = torch.zeros(B, cap, dtype=torch.int32, device="cuda")
    ctx_d = torch.zeros(B, dtype=torch.int32, device="cuda")
    slots_d = torch.zeros(B, dtype=torch.int64, device="cuda")
    step = None
    pa.pa_clear_device_error()
    for it, ctx in enumerate(plan_ctx):
        ctx = np.array(ctx, dtype=np.int32)
        for b in range(B):
            grow = int(ctx[b]) - 1 - a.seq_len(b)
            a.reserve(b, grow)
            m.reserve(b, grow)
        slots, _, _ = a.append_slots(list(range(B)))
        slots_m = np.array([x[0] for x in m.append_slots(range(B))], dtype=np.int64)
        bt, ctx_a = a.block_tables(list(range(B)), cap)
        bt_m = np.full_like(bt, -1)
        for b in range(B):
            t = m.block_table(b)
            bt_m[b, :len(t)] = t
        assert np.array_equal(slots, slots_m) and np.array_equal(bt, bt_m)
        assert np.array_equal(ctx_a, ctx)
        nq, nk, nv = (I.normal_bf16(rng, (B, hq, d)), I.normal_bf16(rng, (B, hkv, d)),
                      I.normal_bf16(rng, (B, hkv, d)))
        q.copy_(dev_bf16(nq))
        key.copy_(dev_bf16(nk))
        val.copy_(dev_bf16(nv))
        bt_d.copy_(torch.from_numpy(np.maximum(bt, 0)))
        ctx_d.copy_(torch.from_numpy(ctx))
        slots_d.copy_(torch.from_numpy(slots))
        if step is None:
            step = pa.DecodeStep(key, val, kc, vc, slots_d, q, bt_d, ctx_d, out, 1 / np.sqrt(d),
                                 partition_size=None, host_context_lens=ctx)
            assert step.partition_size == 256
            assert step.workspace[1].shape[2] == cap * 16 // 256
        step()
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0, f"call {it}"
        kc_h, vc_h = OC.reshape_and_cache(nk, nv, kc_h, vc_h, slots_m, 16)
        ref = OA.decode(nq, kc_h, vc_h, bt_m, ctx, 1 / np.sqrt(d), 16)
        assert_close(bf16_to_f64(out), ref, f"DecodeStep call {it}, contexts {ctx.tolist()}")


@pytest.mark.parametrize("kv", ["bf16", "int8"])
def test_fused_step_early_read_chain(kv):
    """PA_STEP_EARLY_READ: two launches back to back on one stream, the second
    (layer 2, its own pools) with early reads and with q = the first launch's
    output, so its q must be read only after waiting for the first kernel.
    Both against the oracle; the second's q is the first's output as stored."""
    w = I.random_case(6600, 6, [300, 17, 1, 2049, 512, 96], 32, 8, 128)
    c1, c2 = _Case(w, kv), _Case(w, kv)
    split = 256
    maxp = -(-int(w.context_lens.max()) // split)
    order = _i32(pa.splitk_order(w.context_lens, split, maxp))
    ws1 = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim, int(w.context_lens.max()),
                              split)
    ws2 = pa.splitk_workspace(w.num_seqs, w.num_q_heads, w.head_dim, int(w.context_lens.max()),
                              split)
    cnt1 = pa.step_counters(w.num_seqs, w.num_kv_heads)
    cnt2 = pa.step_counters(w.num_seqs, w.num_kv_heads)
    q1 = dev_bf16(w.q)
    out1, out2 = torch.empty_like(q1), torch.empty_like(q1)
    bt, ctx, slots = _i32(c1.bt_p), _i32(w.context_lens), _i64(c1.sl_p)
    key, val = dev_bf16(w.key), dev_bf16(w.value)
    kw1 = {"k_scales": c1.dev[2], "v_scales": c1.dev[3]} if kv != "bf16" else {}
    kw2 = {"k_scales": c2.dev[2], "v_scales": c2.dev[3]} if kv != "bf16" else {}
    pa.pa_clear_device_error()
    for _ in range(3):  # a few times, so that the second can start early
        pa.pa_decode_step(out1, q1, c1.dev[0], c1.dev[1], bt, ctx, w.scale, key=key, value=val,
                          slot_mapping=slots, partition_size=split, workspace=ws1,
                          counters=cnt1, order=order, **kw1)
        pa.pa_decode_step(out2, out1, c2.dev[0], c2.dev[1], bt, ctx, w.scale, key=key,
                          value=val, slot_mapping=slots, partition_size=split, workspace=ws2,
                          counters=cnt2, order=order, early_read=True, **kw2)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    c1.oracle_write(w.key, w.value, c1.sl_m)
    c2.oracle_write(w.key, w.value, c2.sl_m)
    assert_close(bf16_to_f64(out1), c1.oracle_decode(w.q), f"early-read chain {kv}: first")
    q2 = host_bits(out1)
    assert_close(bf16_to_f64(out2), c2.oracle_decode(q2), f"early-read chain {kv}: second")
