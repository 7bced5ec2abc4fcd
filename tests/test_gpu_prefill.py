"""Paged chunked-prefill attention on the GPU (pa_prefill, tcgen05) against the
float64 prefill oracle: ragged chunks at ragged offsets spanning several query
tiles and key chunks, every supported group size, a chunk of one token (a
decode step), NaN in the unused tail of the last block, and the host checks."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import prefill as OP
from paged_kv_cache_283_gb300 import pa
from paged_kv_cache_283_gb300.inputs import normal_bf16

from gpu_helpers import assert_close, bf16_to_f64, dev_bf16

pytestmark = pytest.mark.gpu

BS = 16


def _case(seed, chunks, hq, hkv, d=128, nan_tail=False):
    """chunks: [(prior context, new tokens)] per sequence."""
    rng = np.random.default_rng(seed)
    ctx = np.array([p + n for p, n in chunks], dtype=np.int32)
    qlen = np.array([n for _, n in chunks], dtype=np.int32)
    nblk = -(-ctx // BS)
    nb = int(nblk.sum()) + 7
    perm = rng.permutation(nb)
    mb = int(nblk.max())
    tables = np.full((len(chunks), mb), -1, dtype=np.int32)
    at = 0
    for b, k in enumerate(nblk.tolist()):
        tables[b, :k] = perm[at:at + k]
        at += k
    kc = normal_bf16(rng, (nb, hkv, BS, d))
    vc = normal_bf16(rng, (nb, hkv, BS, d))
    if nan_tail:  # positions past each context hold NaN
        for b, c in enumerate(ctx.tolist()):
            if c % BS:
                blk = tables[b, c // BS]
                kc[blk, :, c % BS:, :] = 0x7FC0
                vc[blk, :, c % BS:, :] = 0x7FC0
    q = normal_bf16(rng, (int(qlen.sum()), hq, d))
    return ctx, qlen, tables, kc, vc, q


def _run(ctx, qlen, tables, kc, vc, q, scale):
    qsl = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    dq = dev_bf16(q)
    out = torch.full_like(dq, float("nan"))
    pa.pa_clear_device_error()
    pa.pa_prefill(out, dq, dev_bf16(kc), dev_bf16(vc), torch.from_numpy(tables).cuda(),
                  torch.from_numpy(ctx).cuda(), torch.from_numpy(qsl).cuda(),
                  int(qlen.max()), scale)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    ref = OP.prefill(q, kc, vc, tables, ctx, qlen, scale, BS)
    return bf16_to_f64(out), ref


MIXED = [(0, 5), (0, 37), (100, 1), (13, 40), (300, 200), (0, 128), (1000, 33), (7, 129)]


@pytest.mark.parametrize("hq,hkv", [(8, 2), (32, 8), (16, 16), (16, 8), (64, 8)])
def test_prefill_mixed_chunks(hq, hkv):
    ctx, qlen, tables, kc, vc, q = _case(hq * 7 + hkv, MIXED, hq, hkv)
    got, ref = _run(ctx, qlen, tables, kc, vc, q, 1.0 / np.sqrt(128.0))
    assert_close(got, ref, f"prefill hq={hq} hkv={hkv}")


def test_prefill_nan_past_context():
    ctx, qlen, tables, kc, vc, q = _case(11, [(3, 10), (0, 21), (40, 7)], 8, 2, nan_tail=True)
    got, ref = _run(ctx, qlen, tables, kc, vc, q, 0.088)
    assert_close(got, ref, "prefill with NaN past the context")


def test_prefill_llama8b_chunks():
    # Llama-3.1-8B heads, 4 chunks of 256 tokens at different depths
    chunks = [(0, 256), (256, 256), (1100, 256), (2000, 256)]
    ctx, qlen, tables, kc, vc, q = _case(12, chunks, 32, 8)
    got, ref = _run(ctx, qlen, tables, kc, vc, q, 1.0 / np.sqrt(128.0))
    assert_close(got, ref, "prefill llama8b chunks")


def test_prefill_one_token_matches_decode():
    ctx, qlen, tables, kc, vc, q = _case(13, [(50, 1), (0, 1), (700, 1)], 32, 8)
    got, ref = _run(ctx, qlen, tables, kc, vc, q, 0.1)
    assert_close(got, ref, "prefill n=1")
    out = torch.empty(q.shape[0], 32, 128, dtype=torch.bfloat16, device="cuda")
    pa.pa_decode(out, dev_bf16(q), dev_bf16(kc), dev_bf16(vc), torch.from_numpy(tables).cuda(),
                 torch.from_numpy(ctx).cuda(), 0.1)
    torch.cuda.synchronize()
    assert_close(bf16_to_f64(out), got, "decode vs prefill n=1")


def test_prefill_host_checks():
    dq = torch.zeros(4, 8, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(2, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    c = torch.ones(1, dtype=torch.int32, device="cuda")
    qsl = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PAError):
        pa.pa_prefill(torch.empty_like(dq), dq, kc, kc, t, c, qsl, 4, 0.1)  # head_dim 64
    assert pa.lib().pa_prefill_supported(128, 4, 16) == 1
    assert pa.lib().pa_prefill_supported(128, 3, 16) == 0


def test_prefill_full_step_sampled():
    """The 16 x 512-token chunked-prefill step the bench times, at full size;
    the oracle checks sampled rows one by one (a row at position p is the
    one-token chunk of the context p + 1)."""
    from oracle.allocator import BlockAllocatorModel
    from paged_kv_cache_283_gb300 import inputs as I
    w = I.chunked_prefill()
    B = len(w.context_lens)
    m = BlockAllocatorModel(w.num_blocks, w.block_size, w.free_order)
    for b, n in enumerate(w.context_lens.tolist()):
        m.add_seq(b)
        m.reserve(b, n)
    tables = [m.block_table(b) for b in range(B)]
    alloc = pa.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    for b, n in enumerate(w.context_lens.tolist()):
        alloc.add_seq(b)
        alloc.reserve(b, n)
    mb = max(len(t) for t in tables)
    bt, ctx = alloc.block_tables(list(range(B)), mb)
    for b in range(B):
        assert list(bt[b, :len(tables[b])]) == list(tables[b])
    qsl = np.concatenate([[0], np.cumsum(w.query_lens)]).astype(np.int32)
    dq = dev_bf16(w.q)
    out = torch.full_like(dq, float("nan"))
    pa.pa_clear_device_error()
    pa.pa_prefill(out, dq, dev_bf16(w.k_cache), dev_bf16(w.v_cache), torch.from_numpy(bt).cuda(),
                  torch.from_numpy(ctx.astype(np.int32)).cuda(), torch.from_numpy(qsl).cuda(),
                  int(w.query_lens.max()), w.scale)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    got = bf16_to_f64(out)
    assert np.all(np.isfinite(got))
    rows, refs = [], []
    for b in range(B):
        n, c = int(w.query_lens[b]), int(w.context_lens[b])
        for i in (0, 1, 31, 32, 255, n - 1):
            pos = c - n + i
            refs.append(OP.prefill_sequence(w.q[qsl[b] + i:qsl[b] + i + 1], w.k_cache, w.v_cache,
                                            tables[b], pos + 1, w.scale, w.block_size)[0])
            rows.append(got[qsl[b] + i])
    assert_close(np.stack(rows), np.stack(refs), "full chunked-prefill step, sampled rows")
