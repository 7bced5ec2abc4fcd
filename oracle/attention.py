"""Paged decode attention, restated plainly in float64 (oracle, test-only).

What is computed, and where it comes from:

* The query of the newest token is compared against the keys of the earlier
  tokens, and the result is a weighted mix of their values ("How LLM Inference
  Serving Works", section "What the KV Cache Is, and How Big It Gets").  The
  pages never print the formula; the plainest reading, used here, is
  softmax(scale * K q) V with the scale chosen by the caller.
* Grouped-query attention: 32 query heads share 8 KV heads (same section).
  The grouping is not stated; query head h reads KV head h // G with
  G = Hq / Hkv (contiguous groups).
* The K and V of a sequence live in fixed-size physical blocks anywhere in the
  pool, and a per-sequence block table maps logical block j to its physical
  block ("PagedAttention: Virtual Memory for the KV Cache"; "Visual
  walkthrough", Step 7).  Token j of a sequence therefore sits in physical
  block table[j // bs] at offset j % bs.  The pool layout (not stated on the
  pages) is [num_blocks, Hkv, bs, D].
* Paging changes where bytes live, not the arithmetic ("Visual walkthrough",
  quick self-check: the FLOPs are unchanged), so the oracle first gathers each
  sequence into contiguous K/V and then runs dense attention on it.
* Split over partitions: attention over a long context can be evaluated per
  contiguous partition of ``partition_size`` tokens, keeping per partition
  m = max score, l = sum exp(score - m) and o = sum exp(score - m) v / l; the
  partitions are combined with weights l_p * exp(m_p - M), M = max m_p.  This
  is the textbook log-sum-exp identity, not something the pages print.
* An empty sequence (context length 0) has nothing to attend to; its output is
  taken as zeros.

Inputs may be raw bf16 bit patterns (uint16) or float arrays; bit patterns are
decoded exactly after gathering, so only the rows a sequence uses are ever
widened to float64.
"""
import numpy as np

from .bf16 import bf16_bits_to_f64


def as_f64(x):
    """Float64 view of a bf16-bit-pattern (uint16) or floating-point array."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return x.astype(np.float64)


def gather_sequence(cache, table_row, ctx, block_size):
    """Rows [ctx, Hkv, D] of one sequence, in logical order, via its block table."""
    pos = np.arange(ctx)
    phys = np.asarray(table_row, dtype=np.int64)[pos // block_size]
    off = pos % block_size
    # Two index arrays separated by a slice: numpy puts the broadcast index
    # dimension first, giving [ctx, Hkv, D].
    return as_f64(cache[phys, :, off, :])


def softmax_attention(qh, K, V, scale):
    """softmax(scale * K @ qh) @ V for one query head; K, V are [n, D], n >= 1."""
    s = scale * (K @ qh)
    w = np.exp(s - s.max())
    return (w @ V) / w.sum()


def decode_sequence(q_b, k_cache, v_cache, table_row, ctx, scale, block_size,
                    q_heads=None):
    """Decode output [Hq, D] (float64) for one sequence.

    ``q_b`` is that sequence's query [Hq, D]; only the heads in ``q_heads``
    (default: all) are computed, the others are left as NaN.
    """
    q_b = as_f64(q_b)
    hq, d = q_b.shape
    hkv = k_cache.shape[1]
    group = hq // hkv
    out = np.full((hq, d), np.nan)
    heads = range(hq) if q_heads is None else q_heads
    if ctx == 0:
        for h in heads:
            out[h] = 0.0
        return out
    K = gather_sequence(k_cache, table_row, ctx, block_size)
    V = gather_sequence(v_cache, table_row, ctx, block_size)
    for h in heads:
        g = h // group
        out[h] = softmax_attention(q_b[h], K[:, g, :], V[:, g, :], scale)
    return out


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, block_size):
    """Paged decode attention for a batch: q [B, Hq, D] -> out [B, Hq, D] float64."""
    B = q.shape[0]
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(B):
        out[b] = decode_sequence(q[b], k_cache, v_cache, block_tables[b],
                                 int(context_lens[b]), scale, block_size)
    return out


def partition_stats(q_b, k_cache, v_cache, table_row, ctx, scale, block_size,
                    partition_size, q_heads=None):
    """Per-partition statistics of one sequence.

    Returns (m, l, o) with shapes [Hq, nparts], [Hq, nparts], [Hq, nparts, D]
    where nparts = ceil(ctx / partition_size) and, for partition p covering
    tokens [p*P, min(ctx, (p+1)*P)):
      m = max score, l = sum exp(score - m), o = sum exp(score - m) v / l.
    Heads outside ``q_heads`` are left as NaN.
    """
    q_b = as_f64(q_b)
    hq, d = q_b.shape
    hkv = k_cache.shape[1]
    group = hq // hkv
    nparts = -(-ctx // partition_size)
    m = np.full((hq, nparts), np.nan)
    l = np.full((hq, nparts), np.nan)
    o = np.full((hq, nparts, d), np.nan)
    if ctx == 0:
        return m, l, o
    K = gather_sequence(k_cache, table_row, ctx, block_size)
    V = gather_sequence(v_cache, table_row, ctx, block_size)
    heads = range(hq) if q_heads is None else q_heads
    for h in heads:
        g = h // group
        for p in range(nparts):
            lo, hi = p * partition_size, min(ctx, (p + 1) * partition_size)
            s = scale * (K[lo:hi, g, :] @ q_b[h])
            m[h, p] = s.max()
            e = np.exp(s - m[h, p])
            l[h, p] = e.sum()
            o[h, p] = (e @ V[lo:hi, g, :]) / l[h, p]
    return m, l, o


def lse_merge(m, l, o):
    """Combine partition statistics (m [n], l [n], o [n, D]) into one output [D]."""
    m = np.asarray(m, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    M = m.max()
    w = l * np.exp(m - M)
    return (w @ o) / w.sum()
