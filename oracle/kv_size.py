"""KV-cache size and waste formulas (oracle, test-only).

* ``kv_bytes_per_token``: "How LLM Inference Serving Works" (dev.to),
  section "What the KV Cache Is, and How Big It Gets": two cached vectors (K
  and V) per layer, per KV head, of ``head_dim`` values of ``bytes_per_value``
  bytes each.
* ``kv_total_bytes``: "LLM serving (vLLM, quantized inference): Visual
  walkthrough", Steps 1-5 and the Feynman retelling: the product
  2 * B * S * L * width * p, where the walkthrough's width is d_model for
  multi-head attention; with grouped-query attention the cached width per
  token and layer is kv_heads * head_dim (the dev.to page's form), which is
  what callers pass.
* ``paged_tail_waste`` / ``naive_waste``: Visual walkthrough Steps 6-8 and
  the quick self-check: a paged sequence of S tokens holds ceil(S / bs) whole
  blocks, so ceil(S / bs) * bs - S slots sit empty; a contiguous reservation
  of max_len slots leaves max_len - S empty.
"""


def kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_value):
    """Bytes of K and V cached for one token across all layers."""
    return 2 * layers * kv_heads * head_dim * bytes_per_value


def kv_total_bytes(batch, seq_len, layers, width, bytes_per_value):
    """Bytes of K and V for ``batch`` sequences of ``seq_len`` tokens each."""
    return 2 * batch * seq_len * layers * width * bytes_per_value


def blocks_for_tokens(seq_len, block_size):
    """Whole blocks a paged sequence of ``seq_len`` tokens occupies."""
    return -(-seq_len // block_size)


def paged_tail_waste(seq_len, block_size):
    """Empty slots in the last, partly filled block of a paged sequence."""
    return blocks_for_tokens(seq_len, block_size) * block_size - seq_len


def naive_waste(seq_len, max_len):
    """Empty slots of a contiguous reservation sized to ``max_len`` tokens."""
    return max_len - seq_len
