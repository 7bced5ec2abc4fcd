"""The exact launches bench.py times, against the float64 oracle.

For each workload the benchmark reports, the test takes the benchmark's own
setup (bench._setup: tables and slots from the library's allocator, pool
replicas larger than L2 or one pool per layer), its own launch arguments
(bench.step_launch: the split-K partition size pa_splitk_partition_size
chooses, the longest-first work order, early reads) and its own step function
(bench._attn_fns).  It runs the steps eagerly, as the benchmark's warm-up
does, then replays the captured CUDA graphs back to back, as the timed loop
does: every launch with early reads follows the previous replica's or
layer's launch on the same stream.  Then every replica's (or layer's) pools
are compared bit for bit with the oracle's cache write of the same new
tokens, and the outputs with the oracle's decode over the written cache, at
the parity tolerance.  The oracle's block tables and slots come from its own
allocator model, asserted equal to the library's.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import bench  # noqa: E402
from oracle import attention as OA  # noqa: E402
from oracle import cache as OC  # noqa: E402
from oracle import fp8 as OF  # noqa: E402
from oracle import quant as OQ  # noqa: E402
from oracle.allocator import BlockAllocatorModel  # noqa: E402
from paged_kv_cache_283_gb300 import inputs as I  # noqa: E402
from paged_kv_cache_283_gb300 import pa  # noqa: E402

from gpu_helpers import assert_close, bf16_to_f64, host_bits, model_tables, \
    v_pool_logical  # noqa: E402

pytestmark = pytest.mark.gpu


def _model_tables(w):
    """Oracle-side block tables and new-token slots (the allocator model),
    including the shared-prefix workload's fork of one 1024-token prompt."""
    if w.idx != 4:
        return model_tables(w)
    m = BlockAllocatorModel(w.num_blocks, w.block_size, w.free_order)
    m.add_seq(-1)
    m.reserve(-1, w.prefix_len)
    for b, s in enumerate(w.suffix_lens.tolist()):
        m.fork(-1, b)
        m.reserve(b, s - 1)
    m.free_seq(-1)
    slots = np.array([x[0] for x in m.append_slots(range(w.num_seqs))], dtype=np.int64)
    bt = np.full((w.num_seqs, w.max_blocks_per_seq), -1, dtype=np.int32)
    for b in range(w.num_seqs):
        t = m.block_table(b)
        bt[b, :len(t)] = t
    return bt, slots


def _host_pool(pool, kv):
    """A device pool (replica or layer) in the oracle's logical layout."""
    if kv == "bf16":
        return [host_bits(pool[0]), host_bits(pool[1])]
    return [pool[0].cpu().numpy(), v_pool_logical(pool[1].cpu().numpy(), kv == "fp8"),
            pool[2].cpu().numpy(), pool[3].cpu().numpy()]


def _oracle_write(kv, pools, key, val, slots):
    if kv == "bf16":
        return list(OC.reshape_and_cache(key, val, pools[0], pools[1], slots, 16))
    write = OF.reshape_and_cache_fp8 if kv == "fp8" else OQ.reshape_and_cache_int8
    return list(write(key, val, *pools, slots, 16))


def _oracle_decode(kv, pools, q, bt, ctx, scale):
    if kv == "bf16":
        return OA.decode(q, pools[0], pools[1], bt, ctx, scale, 16)
    dec = OF.decode_fp8 if kv == "fp8" else OQ.decode_int8
    return dec(q, *pools, bt, ctx, scale, 16)


def _bench_path(idx, kv, max_layers=None):
    """Runs the benchmark's step for workload ``idx`` (warm-up, then the
    graphs replayed twice per replica).  Returns (state, launch, initial host
    pools per replica and layer, replica whose outputs the out buffers hold,
    out buffers per layer)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    st = bench._setup(idx, dev, 4 * l2, kv, max_layers=max_layers)
    w = st["w"]
    lp = bench.step_launch(idx, w, kv, num_sms=props.multi_processor_count)
    init = None
    if kv != "bf16":  # synthetic 1-byte pools drawn on the device: keep host copies
        init = [[_host_pool(p, kv) for p in rep] for rep in st["replicas"]]
    order = torch.from_numpy(lp["order"]).to(dev) if lp["order"] is not None else None
    step, _, outs = bench._attn_fns(st, lp["attn"], lp["partition"], lp["fused"], order,
                                    lp["early_read"])
    stream = torch.cuda.Stream(dev)
    nrep = len(st["replicas"])
    pa.pa_clear_device_error()
    with torch.cuda.stream(stream):
        for k in range(3):
            step(k % nrep)
    stream.synchronize()
    graphs = [bench._capture(lambda r=r: step(r), stream) for r in range(nrep)]
    bench._time_graphs(graphs, 2 * nrep, stream)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0, "device error word set by the benchmark's step"
    return st, lp, init, (2 * nrep - 1) % nrep, outs


def _check_tables(st, w):
    bt_m, sl_m = _model_tables(w)
    assert np.array_equal(st["bt_host"], bt_m) and np.array_equal(st["slots_host"], sl_m)
    return bt_m, sl_m


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
def test_batch64_bench_launch_matches_oracle(kv):
    """The headline workload (batch 64, contexts U[128, 2048]): one fused
    launch per step with the chosen partition size, longest-first order and
    early reads, over two pool replicas."""
    st, lp, init, last, outs = _bench_path(2, kv)
    w = st["w"]
    assert lp["fused"] and lp["attn"] == "splitk" and lp["early_read"]
    assert lp["partition"] == pa.splitk_partition_size(
        w.context_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, kv, ordered=True)
    assert lp["order"] is not None and lp["plan"].max_partitions <= pa.ORDER_MAX_PARTITIONS
    bt, slots = _check_tables(st, w)
    for r, rep in enumerate(st["replicas"]):
        start = [w.k_cache, w.v_cache] if kv == "bf16" else init[r][0]
        want = _oracle_write(kv, start, w.key, w.value, slots)
        for got, exp in zip(_host_pool(rep[0], kv), want):
            assert np.array_equal(got, exp), f"replica {r}: pool after the fused write"
        if r == last:
            ref = _oracle_decode(kv, want, w.q, bt, w.context_lens, w.scale)
            assert_close(bf16_to_f64(outs[0]), ref,
                         f"batch-64 bench launch {kv} partition {lp['partition']}")


@pytest.mark.parametrize("kv", ["bf16", "int8", "fp8"])
def test_32_layer_bench_launch_matches_oracle(kv):
    """The 32-layer step's launches (partition chosen for batch 256,
    longest first, early reads), chained over the first three layers'
    pools in one stream: each layer's launch starts against the previous
    layer's.  Every layer against the oracle."""
    st, lp, init, _, outs = _bench_path(5, kv, max_layers=3)
    w = st["w"]
    assert len(st["replicas"]) == 1 and len(st["replicas"][0]) == 3
    assert lp["fused"] and lp["early_read"] and lp["order"] is not None
    assert lp["partition"] == pa.splitk_partition_size(
        w.context_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, kv, ordered=True)
    bt, slots = _check_tables(st, w)
    for layer, pool in enumerate(st["replicas"][0]):
        q, key, val = I.layer_inputs(w, layer)
        if kv == "bf16":
            order = I.layer_block_order(w, layer)
            start = [w.k_cache[order], w.v_cache[order]]
        else:
            start = init[0][layer]
        want = _oracle_write(kv, start, key, val, slots)
        for got, exp in zip(_host_pool(pool, kv), want):
            assert np.array_equal(got, exp), f"layer {layer}: pool after the fused write"
        ref = _oracle_decode(kv, want, q, bt, w.context_lens, w.scale)
        assert_close(bf16_to_f64(outs[layer]), ref,
                     f"32-layer bench launch {kv} layer {layer} partition {lp['partition']}")


def test_shared_prefix_bench_launch_matches_oracle():
    """Batch 128 sharing one 1024-token prefix (refcount 128): the
    benchmark's fused launches against the oracle."""
    st, lp, _, last, outs = _bench_path(4, "bf16")
    w = st["w"]
    bt, slots = _check_tables(st, w)
    want = _oracle_write("bf16", [w.k_cache, w.v_cache], w.key, w.value, slots)
    for r, rep in enumerate(st["replicas"]):
        for got, exp in zip(_host_pool(rep[0], "bf16"), want):
            assert np.array_equal(got, exp), f"replica {r}: pool after the fused write"
    ref = _oracle_decode("bf16", want, w.q, bt, w.context_lens, w.scale)
    assert_close(bf16_to_f64(outs[0]), ref, f"shared-prefix bench launch {lp['partition']}")


def test_long_context_bench_launch_matches_oracle_sampled_heads():
    """The long-context batch (8K..128K tokens) as the benchmark runs it:
    512-token partitions fixed by the workload, grid order, early reads, the
    fused launch followed by its second-launch merge.  Pools bit for bit;
    outputs against the oracle on four heads of every sequence (one per
    sampled KV group), each decoded over that KV head's slice of the pools."""
    st, lp, _, last, outs = _bench_path(3, "bf16")
    w = st["w"]
    assert lp["partition"] == 512 and lp["order"] is None and lp["early_read"]
    bt, slots = _check_tables(st, w)
    want = _oracle_write("bf16", [w.k_cache, w.v_cache], w.key, w.value, slots)
    for r, rep in enumerate(st["replicas"]):
        for got, exp in zip(_host_pool(rep[0], "bf16"), want):
            assert np.array_equal(got, exp), f"replica {r}: pool after the fused write"
    got = bf16_to_f64(outs[0])
    G = w.group
    for b in range(w.num_seqs):
        for h in sorted({(4 * b + k) % w.num_q_heads for k in (0, 9, 18, 27)}):
            g = h // G
            ref = OA.decode_sequence(w.q[b][[h]], want[0][:, g:g + 1], want[1][:, g:g + 1],
                                     bt[b], int(w.context_lens[b]), w.scale, 16)
            assert_close(got[b, h][None], ref, f"long context seq {b} head {h}")
