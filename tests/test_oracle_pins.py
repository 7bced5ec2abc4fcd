"""Pins of the oracle's size / waste formulas and bf16 decoding.

Expected values are the pages' own printed numbers (tests/golden/*.json, each
with its source) or exact IEEE facts; none is produced by the oracle.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import kv_size
from oracle.bf16 import bf16_bits_to_f64

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_bf16_known_patterns():
    bits = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x4000, 0xC040, 0x3F00,
                     0x7F80, 0xFF80, 0x0001, 0x7F7F, 0x3FC0], dtype=np.uint16)
    want = [0.0, -0.0, 1.0, -1.0, 2.0, -3.0, 0.5, math.inf, -math.inf,
            2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, 1.5]
    got = bf16_bits_to_f64(bits)
    for g, w in zip(got, want):
        assert g == w
    assert np.signbit(got[1])
    assert np.isnan(bf16_bits_to_f64(np.array([0x7FC0], dtype=np.uint16))[0])


def test_kv_bytes_per_token_llama():
    g = _gold("kv_cache_sizes.json")
    assert kv_size.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"],
                                      g["bytes_per_value"]) == g["kv_bytes_per_token"]


def test_context_size_table():
    g = _gold("kv_cache_sizes.json")
    per_tok = kv_size.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"],
                                         g["bytes_per_value"])
    for tokens, nbytes in g["context_table"]:
        assert tokens * per_tok == nbytes
        assert kv_size.kv_total_bytes(1, tokens, g["layers"],
                                      g["kv_heads"] * g["head_dim"],
                                      g["bytes_per_value"]) == nbytes


def test_gqa_factor():
    g = _gold("kv_cache_sizes.json")
    gqa = kv_size.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], 2)
    mha = kv_size.kv_bytes_per_token(g["layers"], g["q_heads"], g["head_dim"], 2)
    assert mha == g["gqa_factor"] * gqa


def test_walkthrough_form_matches_per_token_form():
    # Visual walkthrough: width = n_head * d_head = d_model for multi-head
    # attention, so 2*B*S*L*d_model*p equals B*S times the per-token bytes
    # with kv_heads = q_heads.
    g = _gold("kv_cache_sizes.json")
    d_model = g["q_heads"] * g["head_dim"]
    for B, S in [(1, 1), (3, 100), (64, 2048)]:
        assert kv_size.kv_total_bytes(B, S, g["layers"], d_model, 2) == \
            B * S * kv_size.kv_bytes_per_token(g["layers"], g["q_heads"], g["head_dim"], 2)


def test_bytes_per_element_scaling():
    w = _gold("paging_waste.json")["bytes_per_element"]
    base = kv_size.kv_bytes_per_token(32, 8, 128, w["bf16"])
    assert kv_size.kv_bytes_per_token(32, 8, 128, w["int8"]) * 2 == base
    assert kv_size.kv_bytes_per_token(32, 8, 128, w["int4"]) * 4 == base


def test_paged_tail_waste_pins():
    g = _gold("paging_waste.json")
    for S, waste in g["paged_tail_waste"]:
        assert kv_size.paged_tail_waste(S, g["block_size"]) == waste


def test_naive_waste_pins():
    g = _gold("paging_waste.json")
    for S, waste in g["naive_waste"]:
        assert kv_size.naive_waste(S, g["naive_max_len"]) == waste


@pytest.mark.parametrize("bs", [1, 8, 16, 32])
def test_tail_waste_bound_and_exactness(bs):
    for S in range(1, 600):
        w = kv_size.paged_tail_waste(S, bs)
        assert 0 <= w <= bs - 1
        assert (w == 0) == (S % bs == 0)
        # the blocks held are the fewest that fit S tokens
        nb = kv_size.blocks_for_tokens(S, bs)
        assert (nb - 1) * bs < S <= nb * bs
