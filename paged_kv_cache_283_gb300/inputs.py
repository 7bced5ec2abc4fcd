"""Seeded synthetic inputs for the paged decode workloads.

This module only draws numbers: context lengths, the order in which the pool's
physical blocks are handed out, and N(0, 1) values rounded to bf16 for q, the
K/V pools and the new tokens' K/V.  It holds none of the method's arithmetic
(no slot or block-table computation, no attention); block tables come from a
block allocator, and both the CUDA path and the CPU oracle consume the same
arrays drawn here.

Shapes follow the Llama 3.1 8B example of "How LLM Inference Serving Works"
(section "What the KV Cache Is, and How Big It Gets": 32 query heads sharing
8 KV heads, head dimension 128, bf16) with blocks of 16 tokens ("Visual
walkthrough", Step 7).  No dataset or trained weights are involved.

Recipe, per decode workload ``idx`` (1..5; the chunked-prefill step,
``chunked_prefill``, states its own):
  rng = numpy.random.default_rng(283 + idx); draws, in this order:
  1. context lengths (or, for the shared-prefix workload, suffix lengths);
  2. the free-block order: a permutation of the pool;
  3. q [B, Hq, D]; 4. k_cache and 5. v_cache [NB, Hkv, bs, D];
  6. key and 7. value of the B new tokens [B, Hkv, D]
  -- all values standard normal in float32, rounded to bf16 (nearest even).
The pool holds ceil(1.25 * blocks needed) blocks except the tiny workload
(8 blocks).  The 32-layer workload draws one base pool and gives layer l the
base pool's blocks in the order of a seeded permutation (seed 283 + 5, l), so
every layer sees different data at the same block-table entries without
drawing 32 pools.
"""
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


@dataclass
class Workload:
    idx: int
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    context_lens: np.ndarray          # int32 [B], new token included
    num_blocks: int
    free_order: np.ndarray            # int32 [NB], permutation of the pool
    scale: float
    layers: int = 1
    partition_size: int = 512
    prefix_len: int = 0               # shared-prefix workload only
    suffix_lens: np.ndarray = None    # shared-prefix workload only
    q: np.ndarray = None              # uint16 [B, Hq, D] bf16 bits
    k_cache: np.ndarray = None        # uint16 [NB, Hkv, bs, D]
    v_cache: np.ndarray = None
    key: np.ndarray = None            # uint16 [B, Hkv, D]: the new tokens
    value: np.ndarray = None
    extra: dict = field(default_factory=dict)

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    def blocks_per_seq(self):
        return -(-self.context_lens.astype(np.int64) // self.block_size)

    @property
    def max_blocks_per_seq(self):
        return int(self.blocks_per_seq().max()) if self.num_seqs else 0


def f32_to_bf16_bits(x):
    """Round float32 values to bf16 (nearest, ties to even); finite inputs only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (r >> np.uint32(16)).astype(np.uint16)


def normal_bf16(rng, shape, chunk=1 << 24):
    """Standard-normal values rounded to bf16, drawn in chunks to bound memory."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = f32_to_bf16_bits(rng.standard_normal(hi - lo, dtype=np.float32))
    return out.reshape(shape)


def _pool_size(need):
    return int(np.ceil(1.25 * need))


def _finish(w, rng, with_data):
    w.free_order = rng.permutation(w.num_blocks).astype(np.int32)
    if with_data:
        B, hq, hkv, d, bs = (w.num_seqs, w.num_q_heads, w.num_kv_heads,
                             w.head_dim, w.block_size)
        w.q = normal_bf16(rng, (B, hq, d))
        w.k_cache = normal_bf16(rng, (w.num_blocks, hkv, bs, d))
        w.v_cache = normal_bf16(rng, (w.num_blocks, hkv, bs, d))
        w.key = normal_bf16(rng, (B, hkv, d))
        w.value = normal_bf16(rng, (B, hkv, d))
    return w


def tiny(with_data=True):
    """2 sequences of 1 and 37 tokens, 4 q / 2 KV heads, head_dim 64, 8 blocks."""
    rng = np.random.default_rng(283 + 1)
    ctx = np.array([1, 37], dtype=np.int32)
    w = Workload(1, "tiny", 2, 4, 2, 64, BLOCK_SIZE, ctx, 8, None,
                 1.0 / np.sqrt(64.0))
    return _finish(w, rng, with_data)


def llama8b_batch64(with_data=True):
    """64 sequences, contexts uniform in [128, 2048], Llama 3.1 8B head shape."""
    rng = np.random.default_rng(283 + 2)
    ctx = rng.integers(128, 2049, size=64).astype(np.int32)
    need = int((-(-ctx.astype(np.int64) // BLOCK_SIZE)).sum())
    w = Workload(2, "llama3.1-8b-shaped decode, batch 64, ctx U[128,2048]",
                 64, 32, 8, 128, BLOCK_SIZE, ctx, _pool_size(need), None,
                 1.0 / np.sqrt(128.0))
    return _finish(w, rng, with_data)


LONG_CONTEXTS = (8192, 16384, 32768, 32768, 65536, 65536, 131072, 131072)


def long_splitk(with_data=True):
    """8 sequences from 8K to 128K tokens, split into 512-token partitions."""
    rng = np.random.default_rng(283 + 3)
    ctx = np.array(LONG_CONTEXTS, dtype=np.int32)
    need = int((ctx // BLOCK_SIZE).sum())
    w = Workload(3, "long-context split-K, batch 8, ctx 8K..128K", 8, 32, 8,
                 128, BLOCK_SIZE, ctx, _pool_size(need), None,
                 1.0 / np.sqrt(128.0), partition_size=512)
    return _finish(w, rng, with_data)


def shared_prefix(with_data=True):
    """128 sequences sharing one 1024-token prefix, private suffixes 16..512."""
    rng = np.random.default_rng(283 + 4)
    suffix = rng.integers(16, 513, size=128).astype(np.int32)
    prefix = 1024
    ctx = (prefix + suffix).astype(np.int32)
    need = prefix // BLOCK_SIZE + int((-(-suffix.astype(np.int64) // BLOCK_SIZE)).sum())
    w = Workload(4, "shared-prefix copy-on-write, batch 128", 128, 32, 8, 128,
                 BLOCK_SIZE, ctx, _pool_size(need), None,
                 1.0 / np.sqrt(128.0), prefix_len=prefix, suffix_lens=suffix)
    return _finish(w, rng, with_data)


def llama8b_32layer_batch256(with_data=True):
    """256 sequences, ctx ~ ceil(Exp(mean 600)) clipped to [1, 4096], 32 layers.

    ``q``, ``key`` and ``value`` are those of layer 0; ``layer_inputs(w, l)``
    gives any layer's.  ``k_cache``/``v_cache`` are the base pool; layer l uses
    ``layer_block_order(w, l)`` as its row order.
    """
    rng = np.random.default_rng(283 + 5)
    ctx = np.clip(np.ceil(rng.exponential(600.0, size=256)), 1, 4096).astype(np.int32)
    need = int((-(-ctx.astype(np.int64) // BLOCK_SIZE)).sum())
    w = Workload(5, "llama3.1-8b-shaped 32-layer decode step, batch 256", 256,
                 32, 8, 128, BLOCK_SIZE, ctx, _pool_size(need), None,
                 1.0 / np.sqrt(128.0), layers=32)
    return _finish(w, rng, with_data)


def layer_block_order(w, layer):
    """Row order of layer ``layer``'s pool over the base pool (32-layer workload)."""
    if layer == 0:
        return np.arange(w.num_blocks, dtype=np.int64)
    rng = np.random.default_rng((283 + 5, layer))
    return rng.permutation(w.num_blocks).astype(np.int64)


def layer_inputs(w, layer):
    """(q, key, value) bf16 bits of one layer of the 32-layer workload."""
    if layer == 0:
        return w.q, w.key, w.value
    rng = np.random.default_rng((283 + 5, layer, 1))
    B, hq, hkv, d = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    return (normal_bf16(rng, (B, hq, d)), normal_bf16(rng, (B, hkv, d)),
            normal_bf16(rng, (B, hkv, d)))


WORKLOADS = {1: tiny, 2: llama8b_batch64, 3: long_splitk, 4: shared_prefix,
             5: llama8b_32layer_batch256}


@dataclass
class PrefillWorkload:
    """A chunked-prefill step: sequence b contributes query_lens[b] new tokens
    at positions context_lens[b] - query_lens[b] .. context_lens[b] - 1."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    context_lens: np.ndarray
    query_lens: np.ndarray
    num_blocks: int
    free_order: np.ndarray
    scale: float
    q: np.ndarray = None        # [T, Hq, D] bf16 bits
    k_cache: np.ndarray = None  # [NB, Hkv, bs, D]
    v_cache: np.ndarray = None


def chunked_prefill(with_data=True, num_seqs=16, chunk=512):
    """An 8192-token step of 16 prefill chunks of 512 tokens (the budget the
    dev.to page's "Chunked prefill" section suggests for throughput on large
    GPUs), each at an earlier context of U{0..224} whole blocks, Llama 3.1 8B
    heads.  rng = default_rng(283 + 6): prior lengths, free-block order, q,
    k_cache, v_cache (N(0, 1) rounded to bf16).  The K/V of the chunk's own
    tokens are part of the pool (written by the cache write before attention)."""
    rng = np.random.default_rng(283 + 6)
    prior = rng.integers(0, 225, size=num_seqs).astype(np.int32) * BLOCK_SIZE
    qlen = np.full(num_seqs, chunk, dtype=np.int32)
    ctx = prior + qlen
    need = int((-(-ctx.astype(np.int64) // BLOCK_SIZE)).sum())
    nb = _pool_size(need)
    w = PrefillWorkload("chunked prefill, 16 x 512-token chunks, prior ctx U{0..3584}", 32, 8,
                        128, BLOCK_SIZE, ctx, qlen, nb, rng.permutation(nb).astype(np.int32),
                        1.0 / np.sqrt(128.0))
    if with_data:
        w.q = normal_bf16(rng, (int(qlen.sum()), 32, 128))
        w.k_cache = normal_bf16(rng, (nb, 8, BLOCK_SIZE, 128))
        w.v_cache = normal_bf16(rng, (nb, 8, BLOCK_SIZE, 128))
    return w


def workload(idx, with_data=True):
    return WORKLOADS[idx](with_data=with_data)


def random_case(seed, num_seqs, context_lens, num_q_heads, num_kv_heads,
                head_dim, num_blocks=None, scale=None):
    """A small ad-hoc workload (edge cases, ragged tails) with the same recipe."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32)
    need = int((-(-ctx.astype(np.int64) // BLOCK_SIZE)).sum())
    nb = num_blocks if num_blocks is not None else max(1, _pool_size(need))
    w = Workload(0, f"case-{seed}", num_seqs, num_q_heads, num_kv_heads,
                 head_dim, BLOCK_SIZE, ctx, nb, None,
                 scale if scale is not None else 1.0 / np.sqrt(head_dim))
    return _finish(w, rng, True)
