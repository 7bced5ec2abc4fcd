"""pa_splitk_partition_size (host): the split-K partition size chosen for a
decode batch by the launch-time model pa.h states.  The model is restated
here in Python (CTAs in grid order onto the first free slot; per-token,
per-CTA and merge costs; a second merge launch past 16 partitions) and the
library's choice must equal the restatement's on varied batches; plus the
properties any such choice has."""
import ctypes
import heapq

import numpy as np
import pytest

from paged_kv_cache_283_gb300 import pa

CANDIDATES = (256, 384, 512, 640, 768, 1024, 1280, 1536, 1792, 2048, 4096)
# (token µs for bf16, for 1-byte caches, per-CTA µs, merge µs) per dispatch order
COSTS = {False: (0.025, 0.019, 4.0, 2.0), True: (0.022, 0.0167, 7.0, 3.0)}
APART_US, IN_KERNEL_PARTS = 3.0, 16


def _slots(num_sms, group, kind):
    if kind == 0:
        return num_sms * (3 if group <= 4 else 1)
    return num_sms * (4 if group <= 4 else 3)


def _makespan(ctx, hkv, part, slots, token_us, ordered=False):
    nps = [max(0, -(-int(n) // part)) for n in ctx]
    maxp = max([1] + nps)
    apart = maxp > IN_KERNEL_PARTS
    durs = []
    for z in range(maxp):
        for n, np_ in zip(ctx, nps):
            if z >= max(np_, 1):
                continue
            tokens = max(0, min(part, int(n) - z * part))
            cta_us, merge_us = COSTS[ordered][2:]
            durs.append(token_us * tokens + cta_us + (merge_us if (np_ > 1 and not apart) else 0.0))
    if ordered:
        durs.sort(reverse=True)  # stable: equal durations keep their order
    free = [0.0] * slots
    for d in durs:
        for _ in range(hkv):
            t = heapq.heappop(free)
            heapq.heappush(free, t + d)
    return max(free) + (APART_US if apart else 0.0)


def _model_choice(ctx, hq, hkv, d, kind, num_sms, ordered=False):
    slots = _slots(num_sms, hq // hkv, kind)
    token_us = COSTS[ordered][0 if kind == 0 else 1] * d / 128.0
    if not ordered and kind != 0 and len(ctx) * hkv < slots and -(-max(ctx) // 512) <= 65535:
        return 512  # 1-byte caches in grid order with fewer units than slots
    best, best_t = 0, 0.0
    for part in CANDIDATES:
        if -(-max(ctx) // part) > 65535:
            continue
        t = _makespan(ctx, hkv, part, slots, token_us, ordered)
        if best == 0 or t <= best_t + 1e-9:
            best, best_t = part, t
        if part >= max(ctx):
            break
    return best


@pytest.mark.parametrize("seed", range(6))
def test_choice_equals_the_stated_model(seed):
    rng = np.random.default_rng(seed)
    kinds = ["bf16", "int8", "fp8"]
    for _ in range(4):
        b = int(rng.integers(1, 300))
        hkv = int(rng.choice([2, 4, 8]))
        hq = hkv * int(rng.choice([2, 4, 8]))
        d = int(rng.choice([64, 128]))
        kind = int(rng.integers(0, 3))
        sms = int(rng.choice([132, 148, 152]))
        shape = rng.choice(["uniform", "exp", "long"])
        if shape == "uniform":
            ctx = rng.integers(1, 4097, size=b)
        elif shape == "exp":
            ctx = np.clip(np.ceil(rng.exponential(600.0, size=b)), 1, 8192)
        else:
            ctx = rng.integers(1, 131073, size=max(1, b // 30))
        ctx = ctx.astype(np.int32)
        for ordered in (False, True):
            got = pa.splitk_partition_size(ctx, hq, hkv, d, kinds[kind], num_sms=sms,
                                           ordered=ordered)
            assert got == _model_choice(ctx.tolist(), hq, hkv, d, kind, sms, ordered), \
                (b, hq, hkv, d, kind, ordered)


def test_choice_properties():
    # one very long sequence: many partitions are needed to fill the GPU
    assert pa.splitk_partition_size([131072], 32, 8, 128, num_sms=152) <= 1024
    # many short sequences: one partition each is best (no split, no merge)
    ctx = np.full(1024, 200, dtype=np.int32)
    assert pa.splitk_partition_size(ctx, 32, 8, 128, num_sms=152) >= 200
    # every answer is a candidate
    rng = np.random.default_rng(1)
    for _ in range(20):
        ctx = rng.integers(1, 20000, size=int(rng.integers(1, 64))).astype(np.int32)
        assert pa.splitk_partition_size(ctx, 32, 8, 128, num_sms=152) in CANDIDATES


def test_invalid_arguments_return_zero():
    f = pa.lib().pa_splitk_partition_size
    ctx = np.array([100, 200], dtype=np.int32)
    p = ctx.ctypes.data_as(ctypes.c_void_p)
    assert f(None, 2, 32, 8, 128, 0, 152, 0) == 0
    assert f(p, 0, 32, 8, 128, 0, 152, 0) == 0
    assert f(p, 2, 30, 8, 128, 0, 152, 0) == 0   # heads not divisible
    assert f(p, 2, 32, 8, 128, 3, 152, 0) == 0   # unknown cache kind
    assert f(p, 2, 32, 8, 128, 0, 0, 1) == 0
    assert f(p, 2, 32, 8, 128, 0, 152, 1) > 0
    g = pa.lib().pa_splitk_order
    out = np.empty(4, dtype=np.int32)
    q = out.ctypes.data_as(ctypes.c_void_p)
    assert g(p, 2, 512, 2, None) == -1
    assert g(p, 2, 0, 2, q) == -1
    assert g(p, 2, 512, 0, q) == -1
    assert g(p, 40000, 512, 2, q) == -1          # more than 65535 items
    assert g(p, 2, 512, 2, q) == 4


@pytest.mark.parametrize("seed", range(4))
def test_order_is_a_longest_first_permutation(seed):
    """Every item once; tokens per item non-increasing along the order; equal
    token counts in item order (item = part * B + b)."""
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 200))
    ctx = rng.integers(0, 5000, size=b).astype(np.int32)
    ps = int(rng.choice([256, 512, 768, 1024]))
    maxp = int(-(-int(ctx.max()) // ps)) + int(rng.integers(0, 3))
    maxp = max(1, min(maxp, 65535 // b))
    order = pa.splitk_order(ctx, ps, maxp)
    assert sorted(order.tolist()) == list(range(b * maxp))
    tok = [max(0, min(ps, int(ctx[i % b]) - (i // b) * ps)) for i in order]
    for k in range(1, len(order)):
        assert tok[k - 1] > tok[k] or (tok[k - 1] == tok[k] and order[k - 1] < order[k])
