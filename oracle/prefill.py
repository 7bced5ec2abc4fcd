"""Paged (chunked) prefill attention, restated plainly in float64 (oracle,
test-only).

What is computed, and where it comes from:

* Prefill runs all prompt tokens through the model at once; decode then adds
  one token per step ("How LLM Inference Serving Works", section "Two Phases:
  Prefill and Decode").  Chunked prefill splits a long prompt into pieces that
  share steps with decodes, under a per-step token budget (section "Chunked
  prefill").  A chunk of ``n`` new tokens of a sequence whose context,
  chunk included, is ``ctx`` tokens long holds positions ctx - n .. ctx - 1;
  its keys and values are written into the paged cache first (the cache
  write of the decode path), then every new token attends.
* The query of a token is compared against the keys of the tokens before it
  and mixes their values with the softmax weights (section "What the KV
  Cache Is, and How Big It Gets"); as in the decode oracle the token also
  attends to itself, so the query at position p sees keys 0 .. p (causal).
  With n = 1 this is exactly one decode step.
* Keys and values are found through the sequence's block table, as in
  ``attention.gather_sequence``; grouped-query heads as in ``attention``
  (query head h reads KV head h // (Hq / Hkv)).

Inputs may be raw bf16 bit patterns (uint16) or float arrays.
"""
import numpy as np

from .attention import as_f64, gather_sequence


def prefill_sequence(q_seq, k_cache, v_cache, table_row, ctx, scale, block_size):
    """Outputs [n, Hq, D] (float64) of the n = len(q_seq) newest tokens of one
    sequence with context length ``ctx`` (n <= ctx).  Query i sits at position
    ctx - n + i and attends to the keys at positions 0 .. ctx - n + i."""
    q_seq = as_f64(q_seq)
    n, hq, d = q_seq.shape
    if n == 0:
        return np.zeros((0, hq, d))
    if not 0 < n <= ctx:
        raise ValueError("need 0 < n <= ctx")
    hkv = k_cache.shape[1]
    group = hq // hkv
    K = gather_sequence(k_cache, table_row, ctx, block_size)   # [ctx, Hkv, D]
    V = gather_sequence(v_cache, table_row, ctx, block_size)
    pos = ctx - n + np.arange(n)                                # query positions
    visible = np.arange(ctx)[None, :] <= pos[:, None]           # [n, ctx]
    out = np.empty((n, hq, d))
    for h in range(hq):
        g = h // group
        s = scale * (q_seq[:, h, :] @ K[:, g, :].T)             # [n, ctx]
        s = np.where(visible, s, -np.inf)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        out[:, h, :] = (w @ V[:, g, :]) / w.sum(axis=1, keepdims=True)
    return out


def prefill(q, k_cache, v_cache, block_tables, context_lens, query_lens, scale, block_size):
    """A batch of chunks: q [T, Hq, D] holds the sequences' new tokens back to
    back (sequence b owns query_lens[b] rows, in order).  Returns [T, Hq, D]."""
    q = np.asarray(q)
    outs = []
    row = 0
    for b, (ctx, n) in enumerate(zip(np.asarray(context_lens).tolist(),
                                     np.asarray(query_lens).tolist())):
        outs.append(prefill_sequence(q[row:row + n], k_cache, v_cache, block_tables[b],
                                     int(ctx), scale, block_size))
        row += n
    if row != q.shape[0]:
        raise ValueError("query_lens must sum to the number of query rows")
    return np.concatenate(outs, axis=0) if outs else np.zeros((0,) + q.shape[1:])
