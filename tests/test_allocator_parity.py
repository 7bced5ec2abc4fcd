"""The C++ host allocator (libpa.so, via the binding) against the Python
allocator model of the oracle: the same scripts must give bit-identical
slots, copy-on-write pairs, block tables, refcounts, free lists and errors.
Runs on CPU: the allocator never touches the GPU."""
import numpy as np
import pytest

from oracle.allocator import BlockAllocatorModel, InvalidArg, OutOfBlocks
from paged_kv_cache_283_gb300 import inputs as I
from paged_kv_cache_283_gb300 import pa


@pytest.fixture(scope="module", autouse=True)
def built():
    import os
    if not os.path.exists(pa.LIB_PATH):
        from paged_kv_cache_283_gb300 import build
        build.build()


def _same_state(model, real, live):
    assert list(real.free_list()) == model.free_list()
    for blk in range(model.num_blocks):
        assert real.refcount(blk) == model.refcount(blk)
    for s in live:
        assert list(real.block_table(s)) == model.block_table(s)
        assert real.seq_len(s) == model.seq_len(s)
        assert real.tail_waste(s) == model.tail_waste(s)


def _both(fn_model, fn_real):
    """Run one op on both; they must succeed alike or fail with the same error."""
    try:
        want = fn_model()
        err_m = None
    except OutOfBlocks:
        want, err_m = None, "oob"
    except InvalidArg:
        want, err_m = None, "inval"
    try:
        got = fn_real()
        err_r = None
    except pa.OutOfBlocks:
        got, err_r = None, "oob"
    except pa.PAError as e:
        assert e.status == pa.PA_ERR_INVALID_ARG
        got, err_r = None, "inval"
    assert err_m == err_r
    return want, got


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_scripts_match_model(seed):
    rng = np.random.default_rng(seed)
    nb = 24
    order = rng.permutation(nb)
    model = BlockAllocatorModel(nb, 16, order)
    real = pa.BlockAllocator(nb, 16, order)
    live, next_id = [], 0
    for step in range(2500):
        op = int(rng.integers(0, 12))
        if op < 2 or not live:
            _both(lambda: model.add_seq(next_id), lambda: real.add_seq(next_id))
            live.append(next_id)
            next_id += 1
        elif op < 6:
            s = live[int(rng.integers(len(live)))]
            want, got = _both(lambda: model.append_slot(s), lambda: real.append_slot(s))
            assert want == got
        elif op < 7:
            s = live[int(rng.integers(len(live)))]
            n = int(rng.integers(0, 40))
            want, got = _both(lambda: model.reserve(s, n), lambda: real.reserve(s, n))
            assert want == got
        elif op < 8:
            k = int(rng.integers(1, len(live) + 1))
            seqs = list(rng.choice(live, size=k, replace=False))
            want, got = _both(lambda: model.append_slots(seqs),
                              lambda: real.append_slots(seqs))
            if want is not None:
                assert [w[0] for w in want] == list(got[0])
                assert [w[1] for w in want] == list(got[1])
                assert [w[2] for w in want] == list(got[2])
        elif op < 9:
            p = live[int(rng.integers(len(live)))]
            _both(lambda: model.fork(p, next_id), lambda: real.fork(p, next_id))
            live.append(next_id)
            next_id += 1
        elif op < 10:
            # errors: unknown sequence, duplicate id, duplicate in a batch
            _both(lambda: model.append_slot(10 ** 6), lambda: real.append_slot(10 ** 6))
            _both(lambda: model.add_seq(live[0]), lambda: real.add_seq(live[0]))
            _both(lambda: model.append_slots([live[0], live[0]]),
                  lambda: real.append_slots([live[0], live[0]]))
        else:
            s = live.pop(int(rng.integers(len(live))))
            _both(lambda: model.free_seq(s), lambda: real.free_seq(s))
        _same_state(model, real, live)


def _tables_both(w):
    model = BlockAllocatorModel(w.num_blocks, w.block_size, w.free_order)
    real = pa.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    for b, n in enumerate(w.context_lens.tolist()):
        model.add_seq(b)
        real.add_seq(b)
        model.reserve(b, n - 1)
        real.reserve(b, n - 1)
    # the decode step appends the new token of every sequence
    want = model.append_slots(range(w.num_seqs))
    slots, src, dst = real.append_slots(list(range(w.num_seqs)))
    assert [x[0] for x in want] == slots.tolist()
    assert all(x[1] == -1 for x in want) and np.all(src == -1)
    bt, ctx = real.block_tables(list(range(w.num_seqs)), w.max_blocks_per_seq)
    for b in range(w.num_seqs):
        t = model.block_table(b)
        assert bt[b, :len(t)].tolist() == t and np.all(bt[b, len(t):] == -1)
    assert ctx.tolist() == w.context_lens.tolist()
    return model, real


@pytest.mark.parametrize("idx", [1, 2, 3, 5])
def test_workload_tables_match_model(idx):
    w = I.workload(idx, with_data=False)
    model, real = _tables_both(w)
    used = w.num_blocks - real.num_free()
    assert used == int(w.blocks_per_seq().sum())
    for b in (0, w.num_seqs - 1):
        assert real.tail_waste(b) == (-w.context_lens[b]) % 16


def test_shared_prefix_workload_matches_model():
    w = I.shared_prefix(with_data=False)
    model = BlockAllocatorModel(w.num_blocks, 16, w.free_order)
    real = pa.BlockAllocator(w.num_blocks, 16, w.free_order)
    for a in (model, real):
        a.add_seq(-1)
        a.reserve(-1, w.prefix_len)
        for b, s in enumerate(w.suffix_lens.tolist()):
            a.fork(-1, b)
            a.reserve(b, s)
        a.free_seq(-1)
    _same_state(model, real, range(w.num_seqs))
    assert real.refcount(int(real.block_table(0)[0])) == 128
    used = w.num_blocks - real.num_free()
    assert used == 64 + int(sum(-(-s // 16) for s in w.suffix_lens.tolist()))


def test_invalid_free_order_rejected():
    with pytest.raises(pa.PAError):
        pa.BlockAllocator(4, 16, [0, 1, 1, 2])
    with pytest.raises(pa.PAError):
        pa.BlockAllocator(0, 16)
