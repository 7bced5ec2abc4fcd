"""The shared-prefix decode step (pa_decode_step_shared_prefix: the prefix's
partitions by the tensor-core prefill kernel over the whole batch, the rest by
the split-K decode with the cache write, then the merge) against the float64
oracle, over block tables whose first blocks are the same for every sequence
(a forked prompt) followed by private blocks: pools bit-exact after the new
tokens' write, outputs within the parity tolerance of the oracle's decode.
Batches from 1 to 128 sequences, prefixes of 256 and 1024 tokens, suffixes
from 1 token to several partitions, KV groups of 2 to 8 heads, the
benchmark's shared-prefix workload; a table not holding the prefix, or a
context not past it, raises PA_DEVERR_PREFIX."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import attention as OA  # noqa: E402
from oracle import cache as OC  # noqa: E402
from paged_kv_cache_283_gb300 import inputs as I  # noqa: E402
from paged_kv_cache_283_gb300 import pa  # noqa: E402

from gpu_helpers import assert_close, bf16_to_f64, dev_bf16, host_bits  # noqa: E402

pytestmark = pytest.mark.gpu


def _shared_case(seed, B, prefix_len, suffix, hq, hkv, d=128):
    """Pools, tables (prefix blocks shared, suffix blocks private), contexts
    prefix_len + suffix[b], the new tokens and their slots (position ctx - 1)."""
    rng = np.random.default_rng(seed)
    pb = prefix_len // 16
    sb = [-(-int(s) // 16) for s in suffix]
    nb = pb + sum(sb) + 7
    perm = rng.permutation(nb).astype(np.int32)
    prefix_ids = perm[:pb]
    cap = pb + max(sb)
    bt = np.full((B, cap), -1, dtype=np.int32)
    at = pb
    for b in range(B):
        bt[b, :pb] = prefix_ids
        bt[b, pb:pb + sb[b]] = perm[at:at + sb[b]]
        at += sb[b]
    ctx = (prefix_len + np.asarray(suffix)).astype(np.int32)
    slots = np.array([bt[b][(c - 1) // 16] * 16 + (c - 1) % 16 for b, c in enumerate(ctx)],
                     dtype=np.int64)
    kc = I.normal_bf16(rng, (nb, hkv, 16, d))
    vc = I.normal_bf16(rng, (nb, hkv, 16, d))
    q = I.normal_bf16(rng, (B, hq, d))
    key = I.normal_bf16(rng, (B, hkv, d))
    val = I.normal_bf16(rng, (B, hkv, d))
    return kc, vc, bt, ctx, slots, q, key, val


def _run(kc, vc, bt, ctx, slots, q, key, val, prefix_len, part, scale, write=True, split=None,
         ordered=False):
    B, hq, d = q.shape
    hkv = kc.shape[1]
    split = split or part
    dk, dv = dev_bf16(kc), dev_bf16(vc)
    qd = dev_bf16(q)
    out = torch.empty_like(qd)
    ws = pa.shared_prefix_workspace(B, hq, d, int(ctx.max()), prefix_len, split, part)
    counters = pa.step_counters(B, hkv)
    kw = {}
    if ordered:
        kw["order"] = torch.from_numpy(pa.shared_prefix_order(
            ctx, prefix_len, part, ws[1].shape[2], split)).cuda()
    if write:
        kw = {"key": dev_bf16(key), "value": dev_bf16(val),
              "slot_mapping": torch.from_numpy(slots).cuda()}
    pa.pa_decode_step_shared_prefix(out, qd, dk, dv, torch.from_numpy(np.maximum(bt, 0)).cuda(),
                                    torch.from_numpy(ctx).cuda(), scale, prefix_len, split, part,
                                    ws, counters, **kw)
    torch.cuda.synchronize()
    assert int(counters.abs().sum().item()) == 0, "arrival counters left nonzero"
    return out, dk, dv


@pytest.mark.parametrize("B,prefix_len,split,part", [(1, 256, 256, 256), (5, 256, 128, 64),
                                                     (33, 1024, 512, 256),
                                                     (128, 1024, 256, 512)])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 8), (16, 8)])
@pytest.mark.parametrize("ordered", [False, True])
def test_shared_prefix_step_matches_oracle(B, prefix_len, split, part, hq, hkv, ordered):
    rng = np.random.default_rng(B * 7 + prefix_len + hq)
    suffix = rng.integers(1, 3 * part, size=B)
    suffix[0] = 1                       # the new token right after the prefix
    if B > 2:
        suffix[1] = part                # a suffix of exactly one partition
        suffix[2] = 17
    kc, vc, bt, ctx, slots, q, key, val = _shared_case(8000 + B + hq, B, prefix_len, suffix, hq,
                                                       hkv)
    scale = 1 / np.sqrt(128)
    pa.pa_clear_device_error()
    out, dk, dv = _run(kc, vc, bt, ctx, slots, q, key, val, prefix_len, part, scale, split=split,
                       ordered=ordered)
    assert pa.pa_get_device_error() == 0
    kc2, vc2 = OC.reshape_and_cache(key, val, kc, vc, slots, 16)
    assert np.array_equal(host_bits(dk), kc2) and np.array_equal(host_bits(dv), vc2)
    ref = OA.decode(q, kc2, vc2, bt, ctx, scale, 16)
    assert_close(bf16_to_f64(out), ref,
                 f"shared prefix B={B} prefix={prefix_len} split={split} part={part} "
                 f"G={hq // hkv} ordered={ordered}")


def test_shared_prefix_step_attention_only():
    suffix = np.array([40, 1, 300, 77])
    kc, vc, bt, ctx, slots, q, key, val = _shared_case(8100, 4, 512, suffix, 32, 8)
    pa.pa_clear_device_error()
    out, dk, dv = _run(kc, vc, bt, ctx, slots, q, key, val, 512, 256, 0.1, write=False)
    assert pa.pa_get_device_error() == 0
    assert np.array_equal(host_bits(dk), kc) and np.array_equal(host_bits(dv), vc)
    assert_close(bf16_to_f64(out), OA.decode(q, kc, vc, bt, ctx, 0.1, 16), "attention only")


@pytest.mark.parametrize("what", ["table", "context"])
def test_shared_prefix_step_refuses_a_sequence_without_the_prefix(what):
    """A table whose prefix block differs from sequence 0's, or a context not
    past the prefix: PA_DEVERR_PREFIX (no fault; that sequence's output is
    not the attention it asked for, the others' are)."""
    suffix = np.array([40, 30, 300, 77])
    kc, vc, bt, ctx, slots, q, key, val = _shared_case(8200, 4, 512, suffix, 32, 8)
    if what == "table":
        bt[2, 5] = bt[2, 32 + 1]        # a private block in place of a prefix block
    else:
        ctx[3] = 512                    # the context ends at the prefix
        slots[3] = -1
    pa.pa_clear_device_error()
    out, _, _ = _run(kc, vc, bt, ctx, slots, q, key, val, 512, 256, 0.1, write=False)
    assert pa.pa_get_device_error() & pa.PA_DEVERR_PREFIX
    pa.pa_clear_device_error()
    good = [0, 1] + ([3] if what == "table" else [2])
    ref = OA.decode(q, kc, vc, bt, ctx, 0.1, 16)
    assert_close(bf16_to_f64(out)[good], ref[good], f"the sequences holding the prefix ({what})")


def test_shared_prefix_benchmark_workload():
    """The benchmark's shared-prefix batch (128 forks of one 1024-token
    prompt, private suffixes), its tables from the library's allocator as the
    benchmark builds them."""
    import bench
    dev = torch.device("cuda", 0)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    st = bench._setup(4, dev, 4 * l2, "bf16", n_replicas=1)
    w = st["w"]
    pool = st["replicas"][0][0]
    kc = host_bits(pool[0])
    vc = host_bits(pool[1])
    lp = bench.step_launch(4, w, "bf16", step="shared-prefix")
    assert lp["shared_prefix"]
    order = torch.from_numpy(lp["order"]).to(dev)
    step, _, outs = bench._attn_fns(st, lp["attn"], lp["partition"], lp["fused"], order,
                                    lp["early_read"], True)
    pa.pa_clear_device_error()
    step(0)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    out = outs[0]
    bt, slots = st["bt_host"], st["slots_host"]
    kc2, vc2 = OC.reshape_and_cache(w.key, w.value, kc, vc, slots, 16)
    assert np.array_equal(host_bits(pool[0]), kc2) and np.array_equal(host_bits(pool[1]), vc2)
    ref = OA.decode(w.q, kc2, vc2, bt, w.context_lens, w.scale, 16)
    assert_close(bf16_to_f64(out), ref, "shared-prefix workload")
