"""Pins of the attention oracle (oracle/attention.py) with no GPU.

* brute force: dense attention written with explicit Python loops on
  contiguous K/V, the pool filled block by block from those arrays;
* a library routine: torch's scaled_dot_product_attention in float64 on CPU;
* closed forms: equal keys give the mean of V, one token gives v0;
* invariants: any relabelling of physical blocks, shared vs duplicated prefix;
* the partition / log-sum-exp path against the unsplit result.
"""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle.bf16 import bf16_bits_to_f64
from paged_kv_cache_283_gb300 import inputs as I


def brute_force_dense(q, K, V, scale):
    """softmax(scale q.K) V, all loops explicit; q [Hq][D], K/V [n][Hkv][D]."""
    hq, d = len(q), len(q[0])
    hkv = len(K[0])
    grp = hq // hkv
    out = []
    for h in range(hq):
        kvh = h // grp
        scores = []
        for j in range(len(K)):
            acc = 0.0
            for c in range(d):
                acc += q[h][c] * K[j][kvh][c]
            scores.append(scale * acc)
        mx = max(scores)
        ws = [math.exp(s - mx) for s in scores]
        tot = sum(ws)
        row = []
        for c in range(d):
            acc = 0.0
            for j in range(len(K)):
                acc += ws[j] * V[j][kvh][c]
            row.append(acc / tot)
        out.append(row)
    return out


def place_into_pool(seqs_k, seqs_v, num_blocks, hkv, d, bs, free_order):
    """Lay contiguous per-sequence K/V into a paged pool, walking block by block."""
    kp = np.zeros((num_blocks, hkv, bs, d))
    vp = np.zeros((num_blocks, hkv, bs, d))
    tables = []
    it = iter(free_order)
    for K, V in zip(seqs_k, seqs_v):
        table = []
        n = len(K)
        nblocks = (n + bs - 1) // bs
        for lb in range(nblocks):
            phys = int(next(it))
            table.append(phys)
            for off in range(bs):
                j = lb * bs + off
                if j < n:
                    kp[phys, :, off, :] = K[j]
                    vp[phys, :, off, :] = V[j]
        tables.append(table)
    width = max(len(t) for t in tables)
    bt = np.full((len(tables), width), -1, dtype=np.int64)
    for b, t in enumerate(tables):
        bt[b, :len(t)] = t
    return kp, vp, bt


def _contiguous_case(seed, ctxs, hq, hkv, d):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((len(ctxs), hq, d))
    ks = [rng.standard_normal((n, hkv, d)) for n in ctxs]
    vs = [rng.standard_normal((n, hkv, d)) for n in ctxs]
    return q, ks, vs


@pytest.mark.parametrize("ctxs,hq,hkv,d", [([1, 37], 4, 2, 64), ([16, 17, 5], 4, 4, 8),
                                           ([33, 2], 8, 2, 16)])
def test_oracle_vs_brute_force(ctxs, hq, hkv, d):
    bs = 16
    q, ks, vs = _contiguous_case(7, ctxs, hq, hkv, d)
    need = sum((n + bs - 1) // bs for n in ctxs)
    nb = need + 3
    order = np.random.default_rng(8).permutation(nb)
    kp, vp, bt = place_into_pool(ks, vs, nb, hkv, d, bs, order)
    scale = 1.0 / math.sqrt(d)
    got = A.decode(q, kp, vp, bt, np.array(ctxs), scale, bs)
    for b in range(len(ctxs)):
        want = brute_force_dense(q[b].tolist(), ks[b].tolist(), vs[b].tolist(), scale)
        np.testing.assert_allclose(got[b], np.array(want), rtol=1e-12, atol=1e-13)


def test_oracle_vs_torch_sdpa():
    torch = pytest.importorskip("torch")
    bs, hq, hkv, d = 16, 8, 2, 32
    ctxs = [50, 1, 16, 129]
    q, ks, vs = _contiguous_case(11, ctxs, hq, hkv, d)
    nb = sum((n + bs - 1) // bs for n in ctxs) + 5
    order = np.random.default_rng(12).permutation(nb)
    kp, vp, bt = place_into_pool(ks, vs, nb, hkv, d, bs, order)
    scale = 0.37
    got = A.decode(q, kp, vp, bt, np.array(ctxs), scale, bs)
    for b, n in enumerate(ctxs):
        qt = torch.tensor(q[b], dtype=torch.float64)[:, None, :]          # [Hq,1,D]
        kt = torch.tensor(ks[b], dtype=torch.float64).permute(1, 0, 2)     # [Hkv,n,D]
        vt = torch.tensor(vs[b], dtype=torch.float64).permute(1, 0, 2)
        kt = kt.repeat_interleave(hq // hkv, dim=0)
        vt = vt.repeat_interleave(hq // hkv, dim=0)
        want = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        np.testing.assert_allclose(got[b], want[:, 0, :].numpy(), rtol=1e-11, atol=1e-12)


def test_tiny_workload_vs_brute_force_from_bits():
    w = I.tiny()
    from oracle.allocator import BlockAllocatorModel
    m = BlockAllocatorModel(w.num_blocks, w.block_size, w.free_order)
    for b, n in enumerate(w.context_lens):
        m.add_seq(b)
        m.reserve(b, int(n))
    bt = np.full((w.num_seqs, w.max_blocks_per_seq), -1)
    for b in range(w.num_seqs):
        t = m.block_table(b)
        bt[b, :len(t)] = t
    got = A.decode(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.scale, w.block_size)
    kf = bf16_bits_to_f64(w.k_cache)
    vf = bf16_bits_to_f64(w.v_cache)
    qf = bf16_bits_to_f64(w.q)
    for b, n in enumerate(w.context_lens.tolist()):
        K, V = [], []
        for lb, phys in enumerate(m.block_table(b)):
            for off in range(w.block_size):
                if lb * w.block_size + off < n:
                    K.append(kf[phys, :, off, :].tolist())
                    V.append(vf[phys, :, off, :].tolist())
        want = brute_force_dense(qf[b].tolist(), K, V, w.scale)
        np.testing.assert_allclose(got[b], np.array(want), rtol=1e-12, atol=1e-13)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(3)
    kp = rng.standard_normal((4, 2, 16, 8))
    vp = rng.standard_normal((4, 2, 16, 8))
    q = rng.standard_normal((1, 4, 8)) * 50
    out = A.decode(q, kp, vp, np.array([[2]]), np.array([1]), 1.0, 16)
    for h in range(4):
        assert np.array_equal(out[0, h], vp[2, h // 2, 0])


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(4)
    kp = np.broadcast_to(rng.standard_normal((1, 2, 1, 8)), (5, 2, 16, 8)).copy()
    vp = rng.standard_normal((5, 2, 16, 8))
    q = rng.standard_normal((1, 4, 8))
    table = np.array([[3, 0, 4]])
    n = 40
    out = A.decode(q, kp, vp, table, np.array([n]), 0.5, 16)
    rows = [vp[table[0, j // 16], :, j % 16, :] for j in range(n)]
    mean = np.mean(np.stack(rows), axis=0)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], mean[h // 2], rtol=1e-13, atol=1e-14)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(5)
    kp = rng.standard_normal((3, 1, 16, 4)) * 0.01
    vp = rng.standard_normal((3, 1, 16, 4))
    q = np.ones((1, 1, 4))
    kp[1, 0, 7, :] = 100.0      # logical position 16 + 7 = 23 under table [2, 1]
    out = A.decode(q, kp, vp, np.array([[2, 1]]), np.array([30]), 1.0, 16)
    np.testing.assert_allclose(out[0, 0], vp[1, 0, 7], rtol=0, atol=1e-12)


def test_empty_sequence_gives_zeros():
    rng = np.random.default_rng(6)
    kp = rng.standard_normal((2, 1, 16, 4))
    out = A.decode(rng.standard_normal((2, 2, 4)), kp, kp, np.array([[0], [1]]),
                   np.array([0, 3]), 1.0, 16)
    assert np.all(out[0] == 0.0)
    assert np.all(np.isfinite(out[1]))


def test_block_permutation_invariance():
    w = I.random_case(21, 3, [40, 16, 77], 8, 2, 32)
    bt = _fifo_tables(w)
    out = A.decode(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.scale, 16)
    perm = np.random.default_rng(22).permutation(w.num_blocks)
    kp = np.empty_like(w.k_cache)
    vp = np.empty_like(w.v_cache)
    kp[perm] = w.k_cache
    vp[perm] = w.v_cache
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
    out2 = A.decode(w.q, kp, vp, bt2, w.context_lens, w.scale, 16)
    assert np.array_equal(out, out2)


def test_shared_prefix_equals_duplicated():
    rng = np.random.default_rng(31)
    bs, hkv, d, hq = 16, 2, 16, 4
    prefix_blocks = 3
    suffix = [5, 16, 20]
    nb_shared = prefix_blocks + sum((s + bs - 1) // bs for s in suffix)
    kp = rng.standard_normal((nb_shared, hkv, bs, d))
    vp = rng.standard_normal((nb_shared, hkv, bs, d))
    tables_s, nxt = [], prefix_blocks
    for s in suffix:
        own = list(range(nxt, nxt + (s + bs - 1) // bs))
        nxt += len(own)
        tables_s.append(list(range(prefix_blocks)) + own)
    # duplicated layout: each sequence gets its own copy of the prefix blocks
    kd, vd, tables_d = [], [], []
    for t in tables_s:
        base = len(kd)
        for phys in t:
            kd.append(kp[phys])
            vd.append(vp[phys])
        tables_d.append(list(range(base, base + len(t))))
    kd, vd = np.stack(kd), np.stack(vd)
    width = max(len(t) for t in tables_s)
    pad = lambda ts: np.array([t + [-1] * (width - len(t)) for t in ts])
    ctx = np.array([prefix_blocks * bs + s for s in suffix])
    q = rng.standard_normal((3, hq, d))
    o1 = A.decode(q, kp, vp, pad(tables_s), ctx, 0.25, bs)
    o2 = A.decode(q, kd, vd, pad(tables_d), ctx, 0.25, bs)
    assert np.array_equal(o1, o2)
    assert len(kd) > nb_shared  # the shared pool stores the prefix once


def _fifo_tables(w):
    order = list(w.free_order)
    bt = np.full((w.num_seqs, w.max_blocks_per_seq), -1, dtype=np.int64)
    pos = 0
    for b, n in enumerate(w.context_lens.tolist()):
        k = (n + w.block_size - 1) // w.block_size
        bt[b, :k] = order[pos:pos + k]
        pos += k
    return bt


@pytest.mark.parametrize("psize", [16, 48, 512])
def test_partition_merge_equals_unsplit(psize):
    w = I.random_case(41, 3, [700, 16, 515], 8, 2, 32)
    bt = _fifo_tables(w)
    out = A.decode(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.scale, 16)
    kf = bf16_bits_to_f64(w.k_cache)
    qf = bf16_bits_to_f64(w.q)
    for b, n in enumerate(w.context_lens.tolist()):
        m, l, o = A.partition_stats(w.q[b], w.k_cache, w.v_cache, bt[b], n, w.scale, 16, psize)
        assert m.shape[1] == -(-n // psize)
        for h in range(8):
            merged = A.lse_merge(m[h], l[h], o[h])
            np.testing.assert_allclose(merged, out[b, h], rtol=1e-12, atol=1e-14)
            # m_p is the largest score of its partition, recomputed by loops
            for p in range(m.shape[1]):
                best = -math.inf
                for j in range(p * psize, min(n, (p + 1) * psize)):
                    phys = bt[b][j // 16]
                    s = w.scale * float(np.dot(qf[b, h], kf[phys, h // 4, j % 16]))
                    best = max(best, s)
                assert abs(best - m[h, p]) <= 1e-12 * max(1.0, abs(best))
            assert np.all(l[h] >= 1.0)  # the maximising token contributes exp(0)


def test_single_partition_is_identity():
    w = I.random_case(42, 2, [100, 3], 4, 2, 16)
    bt = _fifo_tables(w)
    out = A.decode(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.scale, 16)
    for b, n in enumerate(w.context_lens.tolist()):
        m, l, o = A.partition_stats(w.q[b], w.k_cache, w.v_cache, bt[b], n, w.scale, 16, 512)
        assert m.shape[1] == 1
        np.testing.assert_allclose(o[:, 0, :], out[b], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(A.lse_merge(m[0], l[0], o[0]), out[b, 0], rtol=1e-13)
