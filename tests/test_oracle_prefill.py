"""Pins of the prefill oracle: brute force, the decode oracle (n = 1), closed
forms, chunking invariance, block relabelling and torch SDPA in float64."""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import prefill as P
from paged_kv_cache_283_gb300.inputs import normal_bf16


def _case(seed, ctx, hq=4, hkv=2, d=16, bs=16, extra=3):
    rng = np.random.default_rng(seed)
    nblk = -(-ctx // bs)
    nb = nblk + extra
    table = rng.permutation(nb)[:nblk]
    kc = normal_bf16(rng, (nb, hkv, bs, d))
    vc = normal_bf16(rng, (nb, hkv, bs, d))
    return rng, table, kc, vc


def test_brute_force_loops():
    ctx, n, hq, hkv, d, bs = 37, 9, 4, 2, 8, 16
    rng, table, kc, vc = _case(1, ctx, hq, hkv, d, bs)
    q = normal_bf16(rng, (n, hq, d))
    got = P.prefill_sequence(q, kc, vc, table, ctx, 0.3, bs)
    qf, kf, vf = A.as_f64(q), A.as_f64(kc), A.as_f64(vc)
    for i in range(n):
        p = ctx - n + i
        for h in range(hq):
            g = h // (hq // hkv)
            scores = []
            for j in range(p + 1):
                blk, off = table[j // bs], j % bs
                scores.append(0.3 * sum(qf[i, h, x] * kf[blk, g, off, x] for x in range(d)))
            mx = max(scores)
            wts = [math.exp(s - mx) for s in scores]
            for x in range(d):
                num = sum(wts[j] * vf[table[j // bs], g, j % bs, x] for j in range(p + 1))
                assert got[i, h, x] == pytest.approx(num / sum(wts), rel=1e-12, abs=1e-12)


def test_one_token_is_a_decode_step():
    ctx, hq, hkv, d, bs = 50, 8, 2, 16, 16
    rng, table, kc, vc = _case(2, ctx, hq, hkv, d, bs)
    q = normal_bf16(rng, (1, hq, d))
    got = P.prefill_sequence(q, kc, vc, table, ctx, 0.25, bs)
    want = A.decode(q, kc, vc, [table], np.array([ctx]), 0.25, bs)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_first_prompt_token_returns_its_value():
    ctx, bs = 20, 16
    rng, table, kc, vc = _case(3, ctx)
    q = normal_bf16(rng, (ctx, 4, 16))
    got = P.prefill_sequence(q, kc, vc, table, ctx, 0.5, bs)
    v0 = A.as_f64(vc[table[0], :, 0, :])          # [Hkv, D]
    for h in range(4):
        assert np.array_equal(got[0, h], v0[h // 2])


def test_chunks_equal_the_whole_prompt():
    ctx, bs = 70, 16
    rng, table, kc, vc = _case(4, ctx)
    q = normal_bf16(rng, (ctx, 4, 16))
    whole = P.prefill_sequence(q, kc, vc, table, ctx, 0.4, bs)
    a = P.prefill_sequence(q[:23], kc, vc, table, 23, 0.4, bs)
    b = P.prefill_sequence(q[23:61], kc, vc, table, 61, 0.4, bs)
    c = P.prefill_sequence(q[61:], kc, vc, table, ctx, 0.4, bs)
    np.testing.assert_allclose(np.concatenate([a, b, c]), whole, rtol=1e-12, atol=1e-13)


def test_block_relabelling_and_batch():
    bs = 16
    rng = np.random.default_rng(5)
    nb, hkv, d = 12, 2, 16
    kc = normal_bf16(rng, (nb, hkv, bs, d))
    vc = normal_bf16(rng, (nb, hkv, bs, d))
    tables = [np.array([3, 7, 1]), np.array([0, 11])]
    ctx, n = np.array([40, 20]), np.array([5, 20])
    q = normal_bf16(rng, (25, 4, d))
    got = P.prefill(q, kc, vc, tables, ctx, n, 0.3, bs)
    perm = rng.permutation(nb)                        # physical block i -> perm[i]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    got2 = P.prefill(q, kc2, vc2, [perm[t] for t in tables], ctx, n, 0.3, bs)
    assert np.array_equal(got, got2)
    np.testing.assert_allclose(got[:5], P.prefill_sequence(q[:5], kc, vc, tables[0], 40, 0.3, bs),
                               rtol=0, atol=0)


def test_torch_sdpa_float64():
    torch = pytest.importorskip("torch")
    ctx, n, hq, hkv, d, bs = 45, 12, 8, 2, 32, 16
    rng, table, kc, vc = _case(6, ctx, hq, hkv, d, bs)
    q = normal_bf16(rng, (n, hq, d))
    got = P.prefill_sequence(q, kc, vc, table, ctx, 0.2, bs)
    K = A.gather_sequence(kc, table, ctx, bs)          # [ctx, Hkv, D]
    V = A.gather_sequence(vc, table, ctx, bs)
    g = hq // hkv
    Kh = torch.from_numpy(np.repeat(K, g, axis=1)).permute(1, 0, 2)   # [Hq, ctx, D]
    Vh = torch.from_numpy(np.repeat(V, g, axis=1)).permute(1, 0, 2)
    Qh = torch.from_numpy(A.as_f64(q)).permute(1, 0, 2)               # [Hq, n, D]
    pos = torch.arange(ctx - n, ctx)[:, None]
    mask = torch.arange(ctx)[None, :] <= pos
    ref = torch.nn.functional.scaled_dot_product_attention(Qh, Kh, Vh, attn_mask=mask,
                                                           scale=0.2)
    np.testing.assert_allclose(got, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


def test_bad_lengths():
    rng, table, kc, vc = _case(7, 10)
    q = normal_bf16(rng, (11, 4, 16))
    with pytest.raises(ValueError):
        P.prefill_sequence(q, kc, vc, table, 10, 0.1, 16)
    with pytest.raises(ValueError):
        P.prefill(q[:3], kc, vc, [table], np.array([10]), np.array([4]), 0.1, 16)
