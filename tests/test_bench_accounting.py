"""The algorithmic bytes and FLOPs the benchmark divides by (its roofline
`achieved` and its `value`), checked against hand-worked cases and brute
force; no GPU needed."""
import numpy as np

import bench


def test_decode_bytes_hand_worked():
    # two sequences of 1 and 37 tokens, 4 q / 2 KV heads, head_dim 64, bf16:
    # K/V 38 tokens x 2 heads x 64 dims x 2 B x 2 (K, V) = 19,456
    # q + out 2 x 2 seqs x 4 heads x 64 x 2 B = 2,048
    # table entries ceil(1/16) + ceil(37/16) = 1 + 3 = 4 -> 16 B, lengths 8 B
    assert bench.decode_bytes([1, 37], 2, 4, 2, 64, 16) == 19456 + 2048 + 16 + 8
    # the same with 1-byte codes: 64 codes + a 4-byte scale per token, head, K or V
    assert bench.decode_bytes([1, 37], 2, 4, 2, 64, 16, "int8") == \
        38 * 2 * (64 + 4) * 2 + 2048 + 16 + 8
    assert bench.decode_bytes([1, 37], 2, 4, 2, 64, 16, "fp8") == \
        bench.decode_bytes([1, 37], 2, 4, 2, 64, 16, "int8")


def test_decode_bytes_llama8b_batch64():
    # 67,794 tokens at the Llama-3.1-8B shape: 4,096 B of K and V per token
    # (8 KV heads x 128 dims x 2 B x 2)
    from paged_kv_cache_283_gb300 import inputs as I
    w = I.llama8b_batch64(with_data=False)
    assert int(w.context_lens.sum()) == 67794
    kv = 67794 * 4096
    qo = 2 * 64 * 32 * 128 * 2
    tables = 4 * int(sum(-(-int(n) // 16) for n in w.context_lens)) + 4 * 64
    assert bench.decode_bytes(w.context_lens, 64, 32, 8, 128, 16) == kv + qo + tables


def test_cache_write_bytes():
    # 64 tokens x 8 KV heads: read K and V (256 B each), write them, read the slots
    assert bench.cache_write_bytes(64, 8, 128) == 2 * 64 * 8 * (256 + 256) + 8 * 64
    assert bench.cache_write_bytes(64, 8, 128, "int8") == 2 * 64 * 8 * (256 + 132) + 8 * 64


def test_prefill_flops_brute_force():
    rng = np.random.default_rng(3)
    for _ in range(20):
        b = int(rng.integers(1, 5))
        n = rng.integers(1, 40, size=b)
        ctx = n + rng.integers(0, 100, size=b)
        hq, d = 4, 8
        brute = 0
        for c, m in zip(ctx.tolist(), n.tolist()):
            for i in range(m):                 # query i of the chunk sits at c - m + i
                p = c - m + i
                brute += 2 * (p + 1) * d * 2 * hq  # QK and PV over keys 0 .. p
        assert bench.prefill_flops(ctx, n, hq, d) == brute


def test_unique_decode_bytes_shared_prefix():
    # the shared-prefix batch: 128 sequences whose first 1024 tokens are one
    # set of 64 blocks; unique K/V bytes count those tokens once, logical
    # bytes once per sequence; q/out and table terms are the same
    from paged_kv_cache_283_gb300 import inputs as I
    w = I.shared_prefix(with_data=False)
    assert w.prefix_len == 1024 and w.num_seqs == 128
    suffix = int(w.context_lens.sum()) - 128 * 1024
    logical = bench.decode_bytes(w.context_lens, 128, 32, 8, 128, 16)
    unique = bench.unique_decode_bytes(w)
    assert logical - unique == 127 * 1024 * 4096
    assert unique == (1024 + suffix) * 4096 + 2 * 128 * 32 * 128 * 2 + \
        4 * int(sum(-(-int(n) // 16) for n in w.context_lens)) + 4 * 128
    # every other workload has nothing shared
    w2 = I.llama8b_batch64(with_data=False)
    assert bench.unique_decode_bytes(w2) == bench.decode_bytes(w2.context_lens, 64, 32, 8, 128, 16)


def test_reference_arm_line_matches_the_gpu_arm_keys():
    # the reference arm (the float64 oracle on the host) prints the GPU arm's
    # metric, unit, direction and workload keys; timed here on the tiny workload
    import argparse
    args = argparse.Namespace(workload=1, steps=1, warmup=0, gpus=1)
    line = bench._reference_timed(args, 2)
    assert line["impl"] == "reference"
    assert (line["metric"], line["unit"], line["higher_is_better"]) == \
        (bench.METRIC, bench.UNIT, True)
    assert line["n_gpus"] == 1 and line["value"] > 0
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["value"] == line["value"]
    for key in ("workload", "batch", "layers", "q_heads", "kv_heads", "head_dim", "block_size",
                "num_blocks", "mean_context", "new_tokens_per_step", "kv_cache"):
        assert key in line["config"], key
    assert line["config"]["batch"] == 2 and line["config"]["sample_seqs"] == 2
