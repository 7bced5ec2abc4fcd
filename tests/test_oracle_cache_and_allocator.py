"""Pins of the oracle's cache write (oracle/cache.py) and allocator model
(oracle/allocator.py): hand-worked scripts, the pages' waste numbers, and
invariants under random scripts."""
import numpy as np
import pytest

from oracle.allocator import BlockAllocatorModel, InvalidArg, OutOfBlocks
from oracle.cache import reshape_and_cache


def test_scatter_writes_exactly_the_slots():
    rng = np.random.default_rng(1)
    nb, hkv, bs, d, T = 6, 2, 16, 8, 9
    kc = rng.integers(0, 65535, size=(nb, hkv, bs, d), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(nb, hkv, bs, d), dtype=np.uint16)
    key = rng.integers(0, 65535, size=(T, hkv, d), dtype=np.uint16)
    val = rng.integers(0, 65535, size=(T, hkv, d), dtype=np.uint16)
    slots = np.array([0, 17, 95, -1, 40, 33, -5, 63, 80])
    k2, v2 = reshape_and_cache(key, val, kc, vc, slots, bs)
    written = set()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = s // bs, s % bs
        written.add((blk, off))
        assert np.array_equal(k2[blk, :, off, :], key[t])
        assert np.array_equal(v2[blk, :, off, :], val[t])
    for blk in range(nb):
        for off in range(bs):
            if (blk, off) not in written:
                assert np.array_equal(k2[blk, :, off], kc[blk, :, off])
                assert np.array_equal(v2[blk, :, off], vc[blk, :, off])
    # inputs untouched unless asked
    assert not np.array_equal(k2, kc)


def test_scripted_allocation():
    m = BlockAllocatorModel(8, 16, [5, 2, 7, 0, 1, 3, 4, 6])
    m.add_seq(10)
    assert m.append_slot(10) == (5 * 16 + 0, -1, -1)
    for pos in range(1, 16):
        assert m.append_slot(10) == (5 * 16 + pos, -1, -1)
    assert m.num_free() == 7
    # token 16 opens the second block, taken from the head of the free list
    assert m.append_slot(10) == (2 * 16 + 0, -1, -1)
    assert m.block_table(10) == [5, 2]
    assert m.seq_len(10) == 17 and m.tail_waste(10) == 15
    # fork shares both blocks
    m.fork(10, 11)
    assert m.refcount(5) == 2 and m.refcount(2) == 2
    # the child writes into the shared, partly filled block: copy-on-write
    assert m.append_slot(11) == (7 * 16 + 1, 2, 7)
    assert m.block_table(11) == [5, 7] and m.refcount(2) == 1 and m.refcount(7) == 1
    # the parent now owns block 2 alone: no copy
    assert m.append_slot(10) == (2 * 16 + 1, -1, -1)
    # freeing the parent returns only the block it no longer shares
    m.free_seq(10)
    assert m.refcount(5) == 1 and m.refcount(2) == 0
    assert m.free_list() == [0, 1, 3, 4, 6, 2]
    m.free_seq(11)
    assert m.free_list() == [0, 1, 3, 4, 6, 2, 5, 7]
    assert all(m.refcount(b) == 0 for b in range(8))


def test_fork_on_block_boundary_needs_no_copy():
    m = BlockAllocatorModel(4, 16)
    m.add_seq(0)
    m.reserve(0, 32)
    m.fork(0, 1)
    assert m.append_slot(1) == (2 * 16, -1, -1)     # fresh block, prefix untouched
    assert m.block_table(1) == [0, 1, 2] and m.refcount(0) == 2


@pytest.mark.parametrize("S,waste", [(32, 0), (1, 15), (100, 12)])
def test_allocator_tail_waste_matches_pages(S, waste):
    m = BlockAllocatorModel(16, 16)
    m.add_seq(0)
    m.reserve(0, S)
    assert m.tail_waste(0) == waste
    assert len(m.block_table(0)) == -(-S // 16)


def test_out_of_blocks_leaves_state_unchanged():
    m = BlockAllocatorModel(3, 16, [2, 0, 1])
    m.add_seq(0)
    m.add_seq(1)
    m.reserve(0, 40)                       # 3 blocks: all of the pool
    snap = (m.free_list(), list(m.ref), m.block_table(0), m.seq_len(0))
    with pytest.raises(OutOfBlocks):
        m.append_slot(1)
    with pytest.raises(OutOfBlocks):
        m.reserve(0, 9)                    # 40 + 9 > 48
    m.reserve(0, 8)                        # exactly fills the last block
    with pytest.raises(OutOfBlocks):
        m.append_slots([0, 1])
    assert m.seq_len(0) == 48 and m.block_table(0) == snap[2]
    assert m.free_list() == snap[0]


def test_batch_append_is_all_or_nothing():
    m = BlockAllocatorModel(4, 16)
    for s in range(3):
        m.add_seq(s)
    m.reserve(0, 16)
    m.reserve(1, 5)
    m.reserve(2, 16)
    # seq 0 and 2 need fresh blocks, seq 1 does not; one block (3) is free
    with pytest.raises(OutOfBlocks):
        m.append_slots([0, 1, 2])
    assert [m.seq_len(s) for s in range(3)] == [16, 5, 16]
    out = m.append_slots([1, 0])
    assert out == [(1 * 16 + 5, -1, -1), (3 * 16 + 0, -1, -1)]
    assert m.seq_len(1) == 6 and m.seq_len(0) == 17


def test_invalid_args():
    m = BlockAllocatorModel(4, 16)
    m.add_seq(1)
    with pytest.raises(InvalidArg):
        m.add_seq(1)
    with pytest.raises(InvalidArg):
        m.append_slot(2)
    with pytest.raises(InvalidArg):
        m.fork(1, 1)
    with pytest.raises(InvalidArg):
        m.append_slots([1, 1])
    with pytest.raises(InvalidArg):
        BlockAllocatorModel(3, 16, [0, 1, 1])


def test_shared_prefix_counts_memory_once():
    rng = np.random.default_rng(9)
    suffix = rng.integers(16, 513, size=128)
    need = 64 + int(sum(-(-s // 16) for s in suffix))
    m = BlockAllocatorModel(need + 10, 16)
    m.add_seq(-1)
    m.reserve(-1, 1024)
    for b, s in enumerate(suffix):
        m.fork(-1, b)
        m.reserve(b, int(s))
    m.free_seq(-1)
    used = m.num_blocks - m.num_free()
    assert used == need
    assert all(m.refcount(blk) == 128 for blk in m.block_table(0)[:64])


def test_random_script_invariants():
    rng = np.random.default_rng(77)
    nb = 40
    m = BlockAllocatorModel(nb, 16, rng.permutation(nb))
    live, next_id = [], 0
    for step in range(3000):
        op = rng.integers(0, 10)
        try:
            if op < 2 or not live:
                m.add_seq(next_id)
                live.append(next_id)
                next_id += 1
            elif op < 7:
                m.append_slot(live[rng.integers(len(live))])
            elif op < 8:
                m.fork(live[rng.integers(len(live))], next_id)
                live.append(next_id)
                next_id += 1
            else:
                s = live.pop(rng.integers(len(live)))
                m.free_seq(s)
        except OutOfBlocks:
            pass
        # invariants
        refs = [0] * nb
        for s in live:
            for blk in m.block_table(s):
                refs[blk] += 1
            assert len(m.block_table(s)) == -(-m.seq_len(s) // 16)
        assert refs == m.ref
        free = m.free_list()
        assert len(set(free)) == len(free)
        assert all(refs[b] == 0 for b in free)
        assert len(free) + sum(1 for r in refs if r > 0) == nb


def test_copy_blocks_copies_whole_blocks_in_every_layer():
    from oracle.cache import copy_blocks
    rng = np.random.default_rng(5)
    ks = [rng.integers(0, 65535, size=(6, 2, 16, 8), dtype=np.uint16) for _ in range(3)]
    vs = [rng.integers(0, 65535, size=(6, 2, 16, 8), dtype=np.uint16) for _ in range(3)]
    k2, v2 = copy_blocks(ks, vs, [[1, 4], [5, 0]])
    for l in range(3):
        assert np.array_equal(k2[l][4], ks[l][1]) and np.array_equal(v2[l][4], vs[l][1])
        assert np.array_equal(k2[l][0], ks[l][5]) and np.array_equal(v2[l][0], vs[l][5])
        for blk in (1, 2, 3, 5):
            assert np.array_equal(k2[l][blk], ks[l][blk])
            assert np.array_equal(v2[l][blk], vs[l][blk])


def test_copy_on_write_keeps_branches_apart():
    # a forked sequence that writes into the shared partial block gets its own
    # copy; the parent's view of the block is unchanged
    from oracle.cache import copy_blocks, reshape_and_cache
    rng = np.random.default_rng(6)
    m = BlockAllocatorModel(6, 16, [3, 1, 4, 0, 2, 5])
    m.add_seq(0)
    m.reserve(0, 20)                       # blocks [3, 1], 4 tokens in block 1
    m.fork(0, 1)
    slot, src, dst = m.append_slot(1)
    assert (src, dst) == (1, 4) and slot == 4 * 16 + 4
    kc = rng.integers(0, 65535, size=(6, 1, 16, 4), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(6, 1, 16, 4), dtype=np.uint16)
    (kc2,), (vc2,) = copy_blocks([kc], [vc], [[src, dst]])
    key = rng.integers(0, 65535, size=(1, 1, 4), dtype=np.uint16)
    kc3, vc3 = reshape_and_cache(key, key, kc2, vc2, [slot], 16)
    assert np.array_equal(kc3[4, :, :4], kc[1, :, :4])      # prefix rows copied
    assert np.array_equal(kc3[4, 0, 4], key[0, 0])           # child's new token
    assert np.array_equal(kc3[1], kc[1])                     # parent's block untouched
