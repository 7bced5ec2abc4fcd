"""Automatic prefix caching (host): the C++ allocator against the Python
model, the behaviour the dev.to page describes ("Prefix Caching and Chunked
Prefill"), and the block names against SHA-256 itself."""
import hashlib

import numpy as np
import pytest

from oracle.allocator import InvalidArg, OutOfBlocks, PrefixCachingAllocatorModel
from paged_kv_cache_283_gb300 import pa


@pytest.fixture(scope="module", autouse=True)
def built():
    import os
    if not os.path.exists(pa.LIB_PATH):
        from paged_kv_cache_283_gb300 import build
        build.build()


def _pair(nb, bs=16, order=None):
    m = PrefixCachingAllocatorModel(nb, bs, order)
    r = pa.BlockAllocator(nb, bs, order)
    r.enable_prefix_cache()
    return m, r


def _same(m, r, live):
    assert list(r.free_list()) == m.free_list()
    assert list(r.evictable_list()) == m.evictable_list()
    for b in range(m.num_blocks):
        assert r.refcount(b) == m.refcount(b)
    for s in live:
        assert list(r.block_table(s)) == m.block_table(s)
        assert r.seq_len(s) == m.seq_len(s)


def test_names_are_sha256():
    # FIPS 180-4 example "abc"; a salt longer than one 64-byte block; chaining
    assert pa.pa_prefix_root_hash(b"abc").hex() == \
        "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad"
    assert pa.pa_prefix_root_hash(b"") == bytes(32)
    long_salt = bytes(range(200))
    assert pa.pa_prefix_root_hash(long_salt) == hashlib.sha256(long_salt).digest()
    rng = np.random.default_rng(1)
    parent = bytes(32)
    for n in (0, 1, 16, 100):
        tok = rng.integers(-2**31, 2**31 - 1, size=n).astype(np.int32)
        want = hashlib.sha256(parent + tok.astype("<i4").tobytes()).digest()
        got = pa.pa_prefix_block_hash(parent, tok)
        assert got == want == PrefixCachingAllocatorModel.block_name(parent, tok)
        parent = got


def test_shared_prompt_prefix_is_reused():
    m, r = _pair(64)
    rng = np.random.default_rng(2)
    a = rng.integers(0, 32000, size=100)
    for al in (m, r):
        assert al.add_seq_prompt(0, a) == 0                  # cold cache
    b = np.concatenate([a[:96], rng.integers(0, 32000, size=30)])
    assert m.add_seq_prompt(1, b) == r.add_seq_prompt(1, b) == 96   # 6 whole blocks
    assert m.block_table(1)[:6] == m.block_table(0)[:6]
    # one token changed early breaks the chain from its block on
    c = a.copy()
    c[40] += 1
    assert m.add_seq_prompt(2, c) == r.add_seq_prompt(2, c) == 32
    c[5] += 1
    assert m.add_seq_prompt(3, c) == r.add_seq_prompt(3, c) == 0
    _same(m, r, [0, 1, 2, 3])


def test_salt_keeps_tenants_apart():
    m, r = _pair(32)
    p = np.arange(64)
    for al in (m, r):
        assert al.add_seq_prompt(0, p, salt=b"tenant-a") == 0
        assert al.add_seq_prompt(1, p, salt=b"tenant-b") == 0
        assert al.add_seq_prompt(2, p, salt=b"tenant-a") == 64
        assert al.add_seq_prompt(3, p) == 0
    _same(m, r, [0, 1, 2, 3])


def test_released_blocks_stay_cached_then_are_evicted_lru():
    m, r = _pair(12, order=list(range(12)))
    rng = np.random.default_rng(3)
    a, b = rng.integers(0, 1000, size=48), rng.integers(0, 1000, size=48)
    for al in (m, r):
        al.add_seq_prompt(0, a)                 # blocks 0-2, named
        al.add_seq_prompt(1, b)                 # blocks 3-5, named
        al.free_seq(0)
        al.free_seq(1)
    assert m.num_free() == 6 and m.evictable_list() == [0, 1, 2, 3, 4, 5]
    assert r.num_free() == 6 and list(r.evictable_list()) == [0, 1, 2, 3, 4, 5]
    # the prompt comes back: a hit on cached-but-evictable blocks
    assert m.add_seq_prompt(2, a) == r.add_seq_prompt(2, a) == 48
    assert m.evictable_list() == [3, 4, 5]
    # 8 fresh blocks: 6 from the free list, then the 2 least recently used
    new = rng.integers(5000, 6000, size=128)
    assert m.add_seq_prompt(3, new) == r.add_seq_prompt(3, new) == 0
    assert m.evictable_list() == [5] == list(r.evictable_list())
    # b's chain lost its first block, so nothing of b is found any more
    blocks3 = m.block_table(3)
    for al in (m, r):
        al.free_seq(3)                          # its 8 named blocks become evictable
    assert m.num_free() == 0 and m.evictable_list() == [5] + blocks3
    assert m.add_seq_prompt(4, b) == r.add_seq_prompt(4, b) == 0
    assert m.block_table(4) == [5] + blocks3[:2]   # the three least recently used
    _same(m, r, [2, 4])


def test_out_of_blocks_leaves_everything_unchanged():
    m, r = _pair(4)
    for al in (m, r):
        al.add_seq_prompt(0, np.arange(48))
    snap = (m.free_list(), m.evictable_list(), list(m.ref))
    for al, exc in ((m, OutOfBlocks), (r, pa.OutOfBlocks)):
        with pytest.raises(exc):
            al.add_seq_prompt(1, np.arange(100, 140))      # 3 blocks, 1 free
    assert (m.free_list(), m.evictable_list(), list(m.ref)) == snap
    _same(m, r, [0])
    with pytest.raises(InvalidArg):
        m.add_seq_prompt(0, [1, 2])
    with pytest.raises(pa.PAError):
        r.add_seq_prompt(0, [1, 2])


def test_enable_only_when_empty():
    r = pa.BlockAllocator(8, 16)
    r.add_seq(0)
    with pytest.raises(pa.PAError):
        r.enable_prefix_cache()
    r2 = pa.BlockAllocator(8, 16)
    with pytest.raises(pa.PAError):
        r2.add_seq_prompt(0, [1, 2, 3])                    # caching is off


def test_system_prompt_stored_once():
    m, r = _pair(1000)
    rng = np.random.default_rng(4)
    system = rng.integers(0, 32000, size=1024)
    private = 0
    for s in range(40):
        tail = rng.integers(0, 32000, size=int(rng.integers(1, 300)))
        prompt = np.concatenate([system, tail])
        want = 0 if s == 0 else 1024
        assert m.add_seq_prompt(s, prompt) == r.add_seq_prompt(s, prompt) == want
        private += -(-len(tail) // 16)
    assert m.num_blocks - m.num_free() == 64 + private
    assert r.refcount(int(r.block_table(0)[0])) == 40
    _same(m, r, range(40))


@pytest.mark.parametrize("seed", [5, 6])
def test_random_scripts_match_model(seed):
    rng = np.random.default_rng(seed)
    nb = 40
    order = rng.permutation(nb)
    m, r = _pair(nb, order=order)
    stems = [rng.integers(0, 50, size=64) for _ in range(3)]
    live, nxt = [], 0
    for step in range(1500):
        op = int(rng.integers(0, 10))
        try:
            if op < 3 or not live:
                stem = stems[int(rng.integers(3))][: int(rng.integers(0, 65))]
                tail = rng.integers(0, 50, size=int(rng.integers(0, 40)))
                salt = [b"", b"x"][int(rng.integers(2))]
                prompt = np.concatenate([stem, tail]).astype(np.int32)
                try:
                    want = m.add_seq_prompt(nxt, prompt, salt)
                except OutOfBlocks:
                    with pytest.raises(pa.OutOfBlocks):
                        r.add_seq_prompt(nxt, prompt, salt)
                    continue
                assert r.add_seq_prompt(nxt, prompt, salt) == want
                live.append(nxt)
                nxt += 1
            elif op < 6:
                s = live[int(rng.integers(len(live)))]
                try:
                    want = m.append_slot(s)
                except OutOfBlocks:
                    with pytest.raises(pa.OutOfBlocks):
                        r.append_slot(s)
                    continue
                assert r.append_slot(s) == want
            elif op < 7:
                p = live[int(rng.integers(len(live)))]
                m.fork(p, nxt)
                r.fork(p, nxt)
                live.append(nxt)
                nxt += 1
            else:
                s = live.pop(int(rng.integers(len(live))))
                m.free_seq(s)
                r.free_seq(s)
        finally:
            pass
        _same(m, r, live)
