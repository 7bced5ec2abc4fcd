"""pa_decode_splitk_noalloc: split-K decode for callers that cannot allocate.

Serving runtimes that reserve all device memory for their own pools, or
threads that must not take an allocation's device synchronisation, cannot
hand the library a cudaMalloc'd workspace.  This entry point keeps the
workspace in a fixed array inside libpa.so.  The test calls it through the C
ABI twice in a row (different inputs and shapes, so the second call runs on
top of the first call's leftover partials) and checks each output against the
regular pa_decode_splitk + pa_splitk_reduce with a caller-allocated
workspace and against the float64 oracle, under the same tolerance the
parity tests use.  It also checks that a call needing more than the built-in
workspace is refused before any launch, and that a context longer than the
caller's max_context_len is reported (PA_DEVERR_CONTEXT_LEN) and only its
first partitions are attended, the rest of the batch unaffected.  The file
sorts last so that a run stopping at the first failure has run every other
test already.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import attention as OA
from paged_kv_cache_283_gb300 import inputs as I
from paged_kv_cache_283_gb300 import pa

from gpu_helpers import assert_close, bf16_to_f64, dev_bf16, model_tables

pytestmark = pytest.mark.gpu


def _dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _regular(q, kc, vc, bt, ctx, scale, max_ctx, partition):
    out = torch.empty_like(q)
    ws = pa.splitk_workspace(q.shape[0], q.shape[1], q.shape[2], max_ctx, partition)
    pa.pa_decode_splitk(*ws, q, kc, vc, bt, ctx, scale, partition_size=partition)
    pa.pa_splitk_reduce(out, *ws, ctx, partition_size=partition)
    return out


def _noalloc_c_abi(q, kc, vc, bt, ctx, scale, max_ctx, partition):
    """Direct C-ABI call with raw device pointers and the current stream."""
    out = torch.empty_like(q)
    B, hq, d = q.shape
    nb, hkv, bs, _ = kc.shape
    st = pa.lib().pa_decode_splitk_noalloc(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
        ctypes.c_void_p(bt.data_ptr()), bt.shape[1], ctypes.c_void_p(ctx.data_ptr()), B, hq,
        hkv, d, bs, nb, float(scale), partition, max_ctx,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pa.PA_OK, pa.lib().pa_status_string(st)
    return out


def _tables(w):
    bt, _ = model_tables(w, step_append=False)
    bt[bt < 0] = 0
    return bt


def _case(w):
    bt = _tables(w)
    return (dev_bf16(w.q), dev_bf16(w.k_cache), dev_bf16(w.v_cache), _dev_i32(bt),
            _dev_i32(w.context_lens), w.scale, int(w.context_lens.max()))


def test_noalloc_matches_regular_split_k_twice_in_a_row():
    pa.pa_clear_device_error()
    first = I.llama8b_batch64()
    second = I.random_case(4242, 5, [1, 700, 16, 1500, 33], 16, 8, 128)
    for w, partition in ((first, 512), (second, 256)):
        q, kc, vc, bt, ctx, scale, max_ctx = _case(w)
        got = _noalloc_c_abi(q, kc, vc, bt, ctx, scale, max_ctx, partition)
        want = _regular(q, kc, vc, bt, ctx, scale, max_ctx, partition)
        torch.cuda.synchronize()
        assert_close(bf16_to_f64(got), bf16_to_f64(want), f"no-alloc vs regular, {w.name}")
        ref = OA.decode(w.q, w.k_cache, w.v_cache, _tables(w), w.context_lens, w.scale, 16)
        assert_close(bf16_to_f64(got), ref, f"no-alloc vs oracle, {w.name}")
    assert pa.pa_get_device_error() == 0


def test_noalloc_context_beyond_max_context_len():
    """max_context_len 512 at partition 256 sizes the built-in workspace for
    two partitions per sequence; a 700-token context raises
    PA_DEVERR_CONTEXT_LEN and attends only its first 512 tokens (the excess
    is dropped); the other sequences are exact."""
    ctx = np.array([100, 700, 512, 1], dtype=np.int32)
    w = I.random_case(4444, len(ctx), ctx, 32, 8, 128)
    q, kc, vc, bt, ctx_d, scale, _ = _case(w)
    pa.pa_clear_device_error()
    got = _noalloc_c_abi(q, kc, vc, bt, ctx_d, scale, 512, 256)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() & pa.PA_DEVERR_CONTEXT_LEN
    pa.pa_clear_device_error()
    seen = np.minimum(ctx, 512)
    ref = OA.decode(w.q, w.k_cache, w.v_cache, _tables(w), seen, w.scale, 16)
    assert_close(bf16_to_f64(got), ref, "no-alloc, one context beyond max_context_len")


def test_noalloc_refuses_more_than_its_workspace():
    w = I.random_case(4343, 2, [40, 20], 32, 8, 128)
    q, kc, vc, bt, ctx, scale, _ = _case(w)
    # B * Hq * ceil(max_ctx / 16) rows of (128 + 2) floats: far beyond 8 MiB
    too_long = 16 * 65535
    out = torch.empty_like(q)
    st = pa.lib().pa_decode_splitk_noalloc(
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
        ctypes.c_void_p(bt.data_ptr()), bt.shape[1], ctypes.c_void_p(ctx.data_ptr()), 2, 32, 8,
        128, 16, kc.shape[0], float(scale), 16, too_long,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pa.PA_ERR_INVALID_ARG
