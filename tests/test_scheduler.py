"""Chunked-prefill step planning: the oracle model pinned to the dev.to page's
scenario and hand-worked cases, and the C++ planner bit-exact against it."""
import numpy as np
import pytest

from oracle.scheduler import plan_step


def test_page_scenario_long_prompt_and_streams():
    # "Chunked prefill": a 10,000-token prompt arrives while 60 users stream;
    # with the docs' example budget of 2048, every step keeps all 60 decodes
    # and the prompt advances 1988 tokens per step -> 6 steps (5 x 1988 + 60).
    remaining, steps, seen = 10_000, 0, []
    while remaining:
        dec, (chunk,) = plan_step(2048, 60, [remaining])
        assert dec == 60 and chunk == min(1988, remaining)
        seen.append(chunk)
        remaining -= chunk
        steps += 1
    assert steps == 6 and seen == [1988] * 5 + [60]


def test_hand_worked():
    assert plan_step(8192, 3, [100, 9000, 50]) == (3, [100, 8089, 0])
    assert plan_step(10, 12, [5]) == (10, [0])          # decodes alone exceed the budget
    assert plan_step(0, 0, []) == (0, [])
    assert plan_step(16, 0, [16, 1]) == (0, [16, 0])
    with pytest.raises(ValueError):
        plan_step(-1, 0, [])


def test_invariants_random():
    rng = np.random.default_rng(7)
    for _ in range(500):
        budget = int(rng.integers(0, 5000))
        dec = int(rng.integers(0, 300))
        rem = rng.integers(0, 3000, size=int(rng.integers(0, 8))).tolist()
        d, ch = plan_step(budget, dec, rem)
        assert d == min(dec, budget) and d + sum(ch) <= budget
        assert all(0 <= c <= r for c, r in zip(ch, rem))
        # queue order: a later prefill gets tokens only if every earlier one is whole
        for i, c in enumerate(ch):
            if c > 0:
                assert all(ch[j] == rem[j] for j in range(i))
        if d + sum(ch) < budget:       # budget left over: everything pending fit
            assert d == dec and ch == rem


def test_native_planner_matches_model():
    pa = pytest.importorskip("paged_kv_cache_283_gb300.pa")
    try:
        pa.lib()
    except Exception as e:  # no library in this checkout
        pytest.skip(f"libpa.so not built: {e}")
    rng = np.random.default_rng(8)
    for _ in range(300):
        budget = int(rng.integers(0, 9000))
        dec = int(rng.integers(0, 400))
        rem = rng.integers(0, 5000, size=int(rng.integers(0, 10))).tolist()
        d, ch = pa.pa_plan_step(budget, dec, rem)
        assert (d, ch.tolist()) == plan_step(budget, dec, rem)
    with pytest.raises(pa.PAError):
        pa.pa_plan_step(-1, 0, [])
