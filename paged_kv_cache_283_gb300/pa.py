"""Thin ctypes binding of libpa.so (include/pa.h), same names as the C ABI.

Argument marshalling only: every device function here checks the tensors'
device / dtype / contiguity, reads their shapes, and passes ``data_ptr()`` and
the current CUDA stream to the C entry point; all computation happens in the
library's kernels.  A non-OK status raises ``PAError``.  There is no fallback:
if ``libpa.so`` is missing this module raises on first use.

Tensors: bf16 data is passed as ``torch.bfloat16`` tensors; block tables and
context lengths as ``torch.int32``; slot mappings as ``torch.int64``.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED_SHAPE = 2
PA_ERR_OUT_OF_BLOCKS = 3
PA_ERR_CUDA = 4

PA_DEVERR_BLOCK_ID = 0x1
PA_DEVERR_CONTEXT_LEN = 0x2
PA_DEVERR_SLOT = 0x4
PA_DEVERR_WAIT_TIMEOUT = 0x8
PA_DEVERR_ORDER = 0x10
PA_DEVERR_PREFIX = 0x20
PA_STEP_EARLY_READ = 0x1

# Every function include/pa.h declares: name -> (restype, argtypes).
_vp, _i, _u, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_float, ctypes.c_size_t
_i64, _pi32, _pi64, _pint = ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), \
    ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [_i]),
    "pa_last_cuda_error": (ctypes.c_char_p, []),
    "pa_get_device_error": (_i, [ctypes.POINTER(_u)]),
    "pa_clear_device_error": (_i, []),
    "pa_decode_supported": (_i, [_i, _i, _i, _i]),
    "pa_reshape_and_cache": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "pa_copy_blocks": (_i, [_vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _vp]),
    "pa_reshape_and_cache_int8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                       _vp]),
    "pa_decode_int8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                            _f, _vp]),
    "pa_decode_splitk_int8": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i,
                                   _i, _i, _i, _i, _i, _f, _i, _vp]),
    "pa_reshape_and_cache_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                      _vp]),
    "pa_decode_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                           _f, _vp]),
    "pa_decode_splitk_fp8": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i,
                                  _i, _i, _i, _i, _i, _f, _i, _vp]),
    "pa_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _f, _vp]),
    "pa_splitk_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "pa_decode_splitk": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i,
                              _i, _i, _f, _i, _vp]),
    "pa_splitk_reduce": (_i, [_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _vp]),
    "pa_splitk_partition_size": (_i, [_vp, _i, _i, _i, _i, _i, _i, _i]),
    "pa_splitk_order": (_i, [_vp, _i, _i, _i, _vp]),
    "pa_decode_step_shared_prefix": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i,
                                          _i, _i, _i, _i, _i, _f, _i, _i, _i, _vp, _vp, _vp,
                                          _vp, _i, _vp, _vp]),
    "pa_decode_step": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i,
                            _i, _f, _i, _vp, _vp, _vp, _vp, _i, _vp, _i, _vp]),
    "pa_decode_step_int8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i,
                                 _i, _i, _i, _i, _i, _f, _i, _vp, _vp, _vp, _vp, _i, _vp, _i,
                                 _vp]),
    "pa_decode_step_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i,
                                _i, _i, _i, _i, _i, _f, _i, _vp, _vp, _vp, _vp, _i, _vp, _i,
                                _vp]),
    "pa_decode_splitk_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                                      _f, _i, _i, _vp]),
    "pa_prefill_supported": (_i, [_i, _i, _i]),
    "pa_prefill": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i,
                        _f, _vp]),
    "pa_plan_step": (_i, [_i, _i, _vp, _i, _vp, _pint]),
    "pa_alloc_create": (_i, [_i, _i, _vp, ctypes.POINTER(_vp)]),
    "pa_alloc_destroy": (None, [_vp]),
    "pa_alloc_add_seq": (_i, [_vp, _i]),
    "pa_alloc_append_slot": (_i, [_vp, _i, _pi64, _pi32, _pi32]),
    "pa_alloc_append_slots": (_i, [_vp, _vp, _i, _vp, _vp, _vp]),
    "pa_alloc_reserve": (_i, [_vp, _i, _i, _pi32, _pi32]),
    "pa_alloc_fork": (_i, [_vp, _i, _i]),
    "pa_alloc_free_seq": (_i, [_vp, _i]),
    "pa_alloc_block_table": (_i, [_vp, _i, _vp, _i, _pint]),
    "pa_alloc_block_tables": (_i, [_vp, _vp, _i, _vp, _i, _vp]),
    "pa_alloc_seq_len": (_i64, [_vp, _i]),
    "pa_alloc_refcount": (_i, [_vp, _i]),
    "pa_alloc_num_free": (_i, [_vp]),
    "pa_alloc_num_blocks": (_i, [_vp]),
    "pa_alloc_free_list": (_i, [_vp, _vp, _i, _pint]),
    "pa_alloc_tail_waste": (_i, [_vp, _i]),
    "pa_alloc_enable_prefix_cache": (_i, [_vp]),
    "pa_alloc_add_seq_prompt": (_i, [_vp, _i, _vp, _i, _vp, _i, _pint]),
    "pa_alloc_num_evictable": (_i, [_vp]),
    "pa_alloc_evictable_list": (_i, [_vp, _vp, _i, _pint]),
    "pa_prefix_root_hash": (_i, [_vp, _i, _vp]),
    "pa_prefix_block_hash": (_i, [_vp, _vp, _i, _vp]),
}

_lib = None


class PAError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = lib().pa_status_string(status).decode()
        if status == PA_ERR_CUDA:
            msg += ": " + lib().pa_last_cuda_error().decode()
        super().__init__(f"{where}: {msg}")


class OutOfBlocks(PAError):
    pass


def lib():
    """The loaded library (ctypes.CDLL); raises if libpa.so was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m paged_kv_cache_283_gb300.build` (needs nvcc)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status, where):
    if status != PA_OK:
        if status == PA_ERR_OUT_OF_BLOCKS:
            raise OutOfBlocks(status, where)
        raise PAError(status, where)


# --------------------------------------------------------------------------
# device entry points (torch tensors in, launches on the current stream)

def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, dtype, name, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def pa_decode_supported(num_q_heads, num_kv_heads, head_dim, block_size):
    return lib().pa_decode_supported(num_q_heads, num_kv_heads, head_dim, block_size) == PA_OK


def pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, stream=None):
    """key/value [T, Hkv, D] bf16; pools [NB, Hkv, bs, D] bf16; slot_mapping [T] int64."""
    torch = _torch()
    T, hkv, d = key.shape
    nb, hkv2, bs, d2 = k_cache.shape
    if value.shape != key.shape or v_cache.shape != k_cache.shape or (hkv, d) != (hkv2, d2):
        raise ValueError("pa_reshape_and_cache: inconsistent shapes")
    if slot_mapping.shape != (T,):
        raise ValueError("pa_reshape_and_cache: slot_mapping must be [num_tokens]")
    st = lib().pa_reshape_and_cache(
        _dev(key, torch.bfloat16, "key", 3), _dev(value, torch.bfloat16, "value", 3),
        _dev(k_cache, torch.bfloat16, "k_cache", 4), _dev(v_cache, torch.bfloat16, "v_cache", 4),
        _dev(slot_mapping, torch.int64, "slot_mapping", 1), T, hkv, d, bs, nb, _stream(stream))
    _check(st, "pa_reshape_and_cache")


def pa_copy_blocks(k_caches, v_caches, block_mapping, stream=None):
    """Copy-on-write copies: block_mapping [n, 2] int64 (src, dst) on the device;
    k_caches / v_caches: lists of per-layer pools [NB, Hkv, bs, D] bf16."""
    torch = _torch()
    if len(k_caches) != len(v_caches) or not k_caches:
        raise ValueError("pa_copy_blocks: one K and one V pool per layer")
    nb, hkv, bs, d = k_caches[0].shape
    for kc, vc in zip(k_caches, v_caches):
        if kc.shape != k_caches[0].shape or vc.shape != kc.shape:
            raise ValueError("pa_copy_blocks: all pools must have one shape")
    if block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("pa_copy_blocks: block_mapping must be [num_pairs, 2]")
    n = len(k_caches)
    kp = (ctypes.c_void_p * n)(*[_dev(t, torch.bfloat16, "k_cache", 4).value for t in k_caches])
    vp = (ctypes.c_void_p * n)(*[_dev(t, torch.bfloat16, "v_cache", 4).value for t in v_caches])
    st = lib().pa_copy_blocks(kp, vp, n, _dev(block_mapping, torch.int64, "block_mapping", 2),
                              block_mapping.shape[0], hkv, d, bs, nb, _stream(stream))
    _check(st, "pa_copy_blocks")


def _decode_common(q, k_cache, v_cache, block_tables, context_lens):
    torch = _torch()
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if v_cache.shape != k_cache.shape or d != d2:
        raise ValueError("decode: inconsistent q / cache shapes")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("decode: block_tables must be [B, max_blocks], context_lens [B]")
    ptrs = (_dev(q, torch.bfloat16, "q", 3), _dev(k_cache, torch.bfloat16, "k_cache", 4),
            _dev(v_cache, torch.bfloat16, "v_cache", 4),
            _dev(block_tables, torch.int32, "block_tables", 2),
            _dev(context_lens, torch.int32, "context_lens", 1))
    return ptrs, (B, hq, hkv, d, bs, nb, block_tables.shape[1])


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, stream=None):
    """out, q [B, Hq, D] bf16; pools [NB, Hkv, 16, D]; block_tables [B, MB] int32."""
    torch = _torch()
    (pq, pk, pv, pt, pc), (B, hq, hkv, d, bs, nb, mb) = _decode_common(
        q, k_cache, v_cache, block_tables, context_lens)
    if out.shape != q.shape:
        raise ValueError("pa_decode: out must match q")
    st = lib().pa_decode(_dev(out, torch.bfloat16, "out", 3), pq, pk, pv, pt, mb, pc, B, hq, hkv,
                         d, bs, nb, float(scale), _stream(stream))
    _check(st, "pa_decode")


def _int8_pools(k_cache, v_cache, k_scales, v_scales, fp8=False):
    torch = _torch()
    nb, hkv, bs, d = k_cache.shape
    if v_cache.shape != k_cache.shape or k_scales.shape != (nb, hkv, bs) or \
            v_scales.shape != k_scales.shape:
        raise ValueError("1-byte cache: pools [NB, Hkv, bs, D] int8 (INT8) or uint8 (FP8 E4M3 "
                         "codes), scales [NB, Hkv, bs] fp32")
    code = torch.uint8 if fp8 else torch.int8
    return (_dev(k_cache, code, "k_cache", 4), _dev(v_cache, code, "v_cache", 4),
            _dev(k_scales, torch.float32, "k_scales", 3),
            _dev(v_scales, torch.float32, "v_scales", 3)), (nb, hkv, bs, d)


def pa_reshape_and_cache_int8(key, value, k_cache, v_cache, k_scales, v_scales, slot_mapping,
                              stream=None):
    """key/value [T, Hkv, D] bf16 quantised into int8 pools + fp32 scales."""
    torch = _torch()
    T, hkv, d = key.shape
    (pk, pv, pks, pvs), (nb, hkv2, bs, d2) = _int8_pools(k_cache, v_cache, k_scales, v_scales)
    if value.shape != key.shape or (hkv, d) != (hkv2, d2) or slot_mapping.shape != (T,):
        raise ValueError("pa_reshape_and_cache_int8: inconsistent shapes")
    st = lib().pa_reshape_and_cache_int8(
        _dev(key, torch.bfloat16, "key", 3), _dev(value, torch.bfloat16, "value", 3), pk, pv,
        pks, pvs, _dev(slot_mapping, torch.int64, "slot_mapping", 1), T, hkv, d, bs, nb,
        _stream(stream))
    _check(st, "pa_reshape_and_cache_int8")


def _decode_int8_common(q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens,
                        fp8=False):
    torch = _torch()
    B, hq, d = q.shape
    pools, (nb, hkv, bs, d2) = _int8_pools(k_cache, v_cache, k_scales, v_scales, fp8)
    if d != d2 or block_tables.dim() != 2 or block_tables.shape[0] != B or \
            context_lens.shape != (B,):
        raise ValueError("int8 decode: inconsistent shapes")
    return (_dev(q, torch.bfloat16, "q", 3),) + pools + (
        _dev(block_tables, torch.int32, "block_tables", 2),
        _dev(context_lens, torch.int32, "context_lens", 1)), (B, hq, hkv, d, bs, nb,
                                                              block_tables.shape[1])


def pa_decode_int8(out, q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens,
                   scale, stream=None):
    torch = _torch()
    (pq, pk, pv, pks, pvs, pt, pc), (B, hq, hkv, d, bs, nb, mb) = _decode_int8_common(
        q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens)
    if out.shape != q.shape:
        raise ValueError("pa_decode_int8: out must match q")
    st = lib().pa_decode_int8(_dev(out, torch.bfloat16, "out", 3), pq, pk, pv, pks, pvs, pt, mb,
                              pc, B, hq, hkv, d, bs, nb, float(scale), _stream(stream))
    _check(st, "pa_decode_int8")


def pa_decode_splitk_int8(ws_out, ws_m, ws_l, q, k_cache, v_cache, k_scales, v_scales,
                          block_tables, context_lens, scale, partition_size=512, stream=None):
    torch = _torch()
    (pq, pk, pv, pks, pvs, pt, pc), (B, hq, hkv, d, bs, nb, mb) = _decode_int8_common(
        q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens)
    maxp = ws_m.shape[2]
    if ws_out.shape != (B, hq, maxp, d) or ws_l.shape != ws_m.shape or ws_m.shape[:2] != (B, hq):
        raise ValueError("pa_decode_splitk_int8: workspace shapes")
    st = lib().pa_decode_splitk_int8(
        _dev(ws_out, torch.float32, "ws_out", 4), _dev(ws_m, torch.float32, "ws_m", 3),
        _dev(ws_l, torch.float32, "ws_l", 3), maxp, pq, pk, pv, pks, pvs, pt, mb, pc, B, hq, hkv,
        d, bs, nb, float(scale), int(partition_size), _stream(stream))
    _check(st, "pa_decode_splitk_int8")


def pa_splitk_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len, partition_size):
    return int(lib().pa_splitk_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len,
                                               partition_size))


def pa_decode_splitk(ws_out, ws_m, ws_l, q, k_cache, v_cache, block_tables, context_lens, scale,
                     partition_size=512, stream=None):
    """ws_out [B, Hq, P, D] fp32, ws_m / ws_l [B, Hq, P] fp32 (P = max partitions)."""
    torch = _torch()
    (pq, pk, pv, pt, pc), (B, hq, hkv, d, bs, nb, mb) = _decode_common(
        q, k_cache, v_cache, block_tables, context_lens)
    maxp = ws_m.shape[2]
    if ws_out.shape != (B, hq, maxp, d) or ws_l.shape != ws_m.shape or ws_m.shape[:2] != (B, hq):
        raise ValueError("pa_decode_splitk: workspace shapes")
    st = lib().pa_decode_splitk(
        _dev(ws_out, torch.float32, "ws_out", 4), _dev(ws_m, torch.float32, "ws_m", 3),
        _dev(ws_l, torch.float32, "ws_l", 3), maxp, pq, pk, pv, pt, mb, pc, B, hq, hkv, d, bs, nb,
        float(scale), int(partition_size), _stream(stream))
    _check(st, "pa_decode_splitk")


def pa_splitk_reduce(out, ws_out, ws_m, ws_l, context_lens, partition_size=512, stream=None):
    torch = _torch()
    B, hq, maxp, d = ws_out.shape
    if out.shape != (B, hq, d) or ws_m.shape != (B, hq, maxp) or ws_l.shape != ws_m.shape:
        raise ValueError("pa_splitk_reduce: shapes")
    st = lib().pa_splitk_reduce(
        _dev(out, torch.bfloat16, "out", 3), _dev(ws_out, torch.float32, "ws_out", 4),
        _dev(ws_m, torch.float32, "ws_m", 3), _dev(ws_l, torch.float32, "ws_l", 3), maxp,
        _dev(context_lens, torch.int32, "context_lens", 1), B, hq, d, int(partition_size),
        _stream(stream))
    _check(st, "pa_splitk_reduce")


def splitk_workspace(num_seqs, num_q_heads, head_dim, max_context_len, partition_size=512,
                     device="cuda"):
    """Allocates (ws_out, ws_m, ws_l) for pa_decode_splitk with torch."""
    torch = _torch()
    maxp = max(1, -(-int(max_context_len) // int(partition_size)))
    return (torch.empty((num_seqs, num_q_heads, maxp, head_dim), dtype=torch.float32, device=device),
            torch.empty((num_seqs, num_q_heads, maxp), dtype=torch.float32, device=device),
            torch.empty((num_seqs, num_q_heads, maxp), dtype=torch.float32, device=device))


def splitk_partition_size(context_lens, num_q_heads, num_kv_heads, head_dim, kv="bf16",
                          num_sms=None, ordered=False):
    """The split-K partition size pa_splitk_partition_size chooses for a batch
    (context_lens: host int array); ordered: for a launch with the
    longest-first order of splitk_order.  num_sms defaults to the current CUDA
    device's multiprocessor count."""
    import numpy as np
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    if num_sms is None:
        torch = _torch()
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    kind = {"bf16": 0, "int8": 1, "fp8": 2}[kv]
    r = lib().pa_splitk_partition_size(ctx.ctypes.data_as(ctypes.c_void_p), ctx.shape[0],
                                       num_q_heads, num_kv_heads, head_dim, kind, int(num_sms),
                                       1 if ordered else 0)
    if r <= 0:
        raise ValueError("pa_splitk_partition_size: invalid arguments")
    return int(r)


def splitk_order(context_lens, partition_size, max_partitions):
    """Longest-first work order (host numpy int32 [B * max_partitions]) for a
    split-K pa_decode_step; copy it to the device and pass it as ``order``."""
    import numpy as np
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.empty(ctx.shape[0] * int(max_partitions), dtype=np.int32)
    r = lib().pa_splitk_order(ctx.ctypes.data_as(ctypes.c_void_p), ctx.shape[0],
                              int(partition_size), int(max_partitions),
                              out.ctypes.data_as(ctypes.c_void_p))
    if r != out.shape[0]:
        raise ValueError("pa_splitk_order: invalid arguments")
    return out


def step_counters(num_seqs, num_kv_heads, device="cuda"):
    """Zeroed arrival counters [num_seqs * num_kv_heads] for a split-K pa_decode_step."""
    torch = _torch()
    return torch.zeros(num_seqs * num_kv_heads, dtype=torch.int32, device=device)


# Past this many partitions per sequence a split-K pa_decode_step merges in a
# second launch, the items are nearly all full partitions and the
# longest-first order has nothing to balance (long contexts measured slower
# with it: 336.0 vs 328.3 us), so plan_decode_step keeps grid order there.
ORDER_MAX_PARTITIONS = 16


class StepPlan:
    """Launch arguments of a split-K pa_decode_step for one batch's contexts:
    partition_size, max_partitions (the workspace's P) and order (host
    numpy int32 [B * max_partitions], longest first, or None for grid
    order)."""

    def __init__(self, partition_size, max_partitions, order, chosen):
        self.partition_size = int(partition_size)
        self.max_partitions = int(max_partitions)
        self.order = order
        self.chosen = bool(chosen)  # partition size from pa_splitk_partition_size

    def __repr__(self):
        return "StepPlan(partition_size=%d, max_partitions=%d, order=%s)" % (
            self.partition_size, self.max_partitions,
            "grid" if self.order is None else "longest first")


def plan_decode_step(context_lens, num_q_heads, num_kv_heads, head_dim, kv="bf16",
                     num_sms=None, partition_size=None, order="longest",
                     max_context_len=None):
    """Partition size, workspace partitions and work order of a split-K
    pa_decode_step for the host context lengths ``context_lens``.

    partition_size None: pa_splitk_partition_size's choice (for a
    longest-first launch when ``order`` is "longest").  max_context_len (the
    longest context the launch must cover; default: the longest of
    context_lens) sets max_partitions.  order "longest": pa_splitk_order's
    order for those partitions when a sequence has at most
    ORDER_MAX_PARTITIONS of them (and the grid fits); otherwise, or with order
    "grid", None.  Every sequence up to max_context_len tokens stays correct
    under the plan whatever its length; other lengths change only the speed."""
    import numpy as np
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    longest = order == "longest"
    if order not in ("longest", "grid"):
        raise ValueError("plan_decode_step: order is 'longest' or 'grid'")
    chosen = partition_size is None
    if chosen:
        partition_size = splitk_partition_size(ctx, num_q_heads, num_kv_heads, head_dim, kv,
                                               num_sms, ordered=longest)
    mc = int(max_context_len) if max_context_len is not None else (
        int(ctx.max()) if ctx.size else 1)
    maxp = max(1, -(-mc // int(partition_size)))
    arr = None
    if longest and maxp <= ORDER_MAX_PARTITIONS and ctx.shape[0] * maxp <= 65535:
        arr = splitk_order(ctx, partition_size, maxp)
    return StepPlan(partition_size, maxp, arr, chosen)


def recover_step_counters(counters):
    """Re-zeroes a split-K pa_decode_step's arrival counters and clears the
    device error word when it holds PA_DEVERR_ORDER or PA_DEVERR_WAIT_TIMEOUT
    (a launch that raised either can leave a counter nonzero, and the next
    launch with those counters would merge too early).  Reads the error word,
    so it synchronises the device.  Returns the error bits it found."""
    err = pa_get_device_error()
    if err & (PA_DEVERR_ORDER | PA_DEVERR_WAIT_TIMEOUT):
        counters.zero_()
        _torch().cuda.synchronize()
        pa_clear_device_error()
    return err


def _step_args(out, q, k_cache, v_cache, block_tables, context_lens, scale, key, value,
               slot_mapping, partition_size, workspace, counters, k_scales, v_scales,
               order=None, early_read=False):
    """(C function, argument tuple without the stream) for pa_decode_step*."""
    torch = _torch()
    fp8 = k_cache.dtype == torch.uint8
    one = fp8 or k_cache.dtype == torch.int8
    if one:
        if k_scales is None or v_scales is None:
            raise ValueError("pa_decode_step: a 1-byte cache needs k_scales and v_scales")
        (pq, pk, pv, pks, pvs, pt, pc), (B, hq, hkv, d, bs, nb, mb) = _decode_int8_common(
            q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens, fp8)
        pools = (pk, pv, pks, pvs)
    else:
        (pq, pk, pv, pt, pc), (B, hq, hkv, d, bs, nb, mb) = _decode_common(
            q, k_cache, v_cache, block_tables, context_lens)
        pools = (pk, pv)
    if out.shape != q.shape:
        raise ValueError("pa_decode_step: out must match q")
    none = ctypes.c_void_p(None)
    if key is None and value is None and slot_mapping is None:
        kvs = (none, none, none)
    elif key is None or value is None or slot_mapping is None:
        raise ValueError("pa_decode_step: key, value and slot_mapping go together")
    else:
        if key.shape != (B, hkv, d) or value.shape != key.shape or slot_mapping.shape != (B,):
            raise ValueError("pa_decode_step: key / value [B, Hkv, D], slot_mapping [B]")
        kvs = (_dev(key, torch.bfloat16, "key", 3), _dev(value, torch.bfloat16, "value", 3),
               _dev(slot_mapping, torch.int64, "slot_mapping", 1))
    ps = int(partition_size)
    if ps > 0:
        if workspace is None or counters is None:
            raise ValueError("pa_decode_step: split-K needs a workspace and counters")
        ws_o, ws_m, ws_l = workspace
        maxp = ws_m.shape[2]
        if ws_o.shape != (B, hq, maxp, d) or ws_l.shape != ws_m.shape or \
                ws_m.shape[:2] != (B, hq) or counters.shape != (B * hkv,):
            raise ValueError("pa_decode_step: workspace / counters shapes")
        wsa = (_dev(ws_o, torch.float32, "ws_out", 4), _dev(ws_m, torch.float32, "ws_m", 3),
               _dev(ws_l, torch.float32, "ws_l", 3), _dev(counters, torch.int32, "counters", 1),
               maxp)
        if order is not None and order.shape != (B * maxp,):
            raise ValueError("pa_decode_step: order must be [num_seqs * max_partitions]")
    else:
        wsa = (none, none, none, none, 0)
        if order is not None:
            raise ValueError("pa_decode_step: an order needs split-K")
    ordp = (none,) if order is None else (_dev(order, torch.int32, "order", 1),)
    fn = lib().pa_decode_step_fp8 if fp8 else (lib().pa_decode_step_int8 if one
                                                else lib().pa_decode_step)
    args = (_dev(out, torch.bfloat16, "out", 3), pq) + kvs + pools + (
        pt, mb, pc, B, hq, hkv, d, bs, nb, float(scale), ps) + wsa + ordp + (
        PA_STEP_EARLY_READ if early_read else 0,)
    return fn, args


def pa_decode_step(out, q, k_cache, v_cache, block_tables, context_lens, scale, key=None,
                   value=None, slot_mapping=None, partition_size=512, workspace=None,
                   counters=None, k_scales=None, v_scales=None, stream=None, order=None,
                   early_read=False):
    """Cache write of each sequence's new token (key / value [B, Hkv, D] at
    slot_mapping [B], which must be the slot of position context_lens[b] - 1)
    and the decode, in one launch.  partition_size 0: whole-sequence CTAs;
    > 0: split-K merged in the same launch (workspace = splitk_workspace(...),
    counters = step_counters(...)).  The cache dtype picks bf16 / INT8 (int8)
    / FP8 (uint8 codes, with k_scales / v_scales).  order: optional device
    int32 work order (splitk_order) for the split-K CTAs.  early_read: the
    caller's promise that tables, lengths, order and pools are not written by
    the kernel launched just before (PA_STEP_EARLY_READ in pa.h)."""
    fn, args = _step_args(out, q, k_cache, v_cache, block_tables, context_lens, scale, key,
                          value, slot_mapping, partition_size, workspace, counters, k_scales,
                          v_scales, order, early_read)
    _check(fn(*args, _stream(stream)), "pa_decode_step")


def shared_prefix_partitions(max_context_len, prefix_len, prefix_split, partition_size):
    """Workspace partitions a pa_decode_step_shared_prefix call needs for
    contexts of up to max_context_len tokens: the prefix's, then the rest's."""
    rest = max(1, int(max_context_len) - int(prefix_len))
    return int(prefix_len) // int(prefix_split) + -(-rest // int(partition_size))


def shared_prefix_workspace(num_seqs, num_q_heads, head_dim, max_context_len, prefix_len,
                            prefix_split, partition_size, device=None):
    """(ws_out, ws_m, ws_l) for pa_decode_step_shared_prefix."""
    torch = _torch()
    device = device or torch.device("cuda")
    p = shared_prefix_partitions(max_context_len, prefix_len, prefix_split, partition_size)
    return (torch.empty(num_seqs, num_q_heads, p, head_dim, dtype=torch.float32, device=device),
            torch.empty(num_seqs, num_q_heads, p, dtype=torch.float32, device=device),
            torch.empty(num_seqs, num_q_heads, p, dtype=torch.float32, device=device))


def _shared_prefix_args(out, q, k_cache, v_cache, block_tables, context_lens, scale, prefix_len,
                        prefix_split, partition_size, workspace, counters, key, value,
                        slot_mapping, order):
    """Checked and marshalled arguments of pa_decode_step_shared_prefix
    (without the stream)."""
    torch = _torch()
    (pq, pk, pv, pt, pc), (B, hq, hkv, d, bs, nb, mb) = _decode_common(
        q, k_cache, v_cache, block_tables, context_lens)
    if out.shape != q.shape:
        raise ValueError("pa_decode_step_shared_prefix: out must match q")
    none = ctypes.c_void_p(None)
    if key is None and value is None and slot_mapping is None:
        kvs = (none, none, none)
    elif key is None or value is None or slot_mapping is None:
        raise ValueError("pa_decode_step_shared_prefix: key, value and slot_mapping go together")
    else:
        if key.shape != (B, hkv, d) or value.shape != key.shape or slot_mapping.shape != (B,):
            raise ValueError("pa_decode_step_shared_prefix: key / value [B, Hkv, D], "
                             "slot_mapping [B]")
        kvs = (_dev(key, torch.bfloat16, "key", 3), _dev(value, torch.bfloat16, "value", 3),
               _dev(slot_mapping, torch.int64, "slot_mapping", 1))
    ws_o, ws_m, ws_l = workspace
    maxp = ws_m.shape[2]
    if ws_o.shape != (B, hq, maxp, d) or ws_l.shape != ws_m.shape or ws_m.shape[:2] != (B, hq) \
            or counters.shape != (B * hkv,):
        raise ValueError("pa_decode_step_shared_prefix: workspace / counters shapes")
    return (_dev(out, torch.bfloat16, "out", 3), pq) + kvs + (
        pk, pv, pt, mb, pc, B, hq, hkv, d, bs, nb, float(scale), int(prefix_len),
        int(prefix_split), int(partition_size), _dev(ws_o, torch.float32, "ws_out", 4),
        _dev(ws_m, torch.float32, "ws_m", 3), _dev(ws_l, torch.float32, "ws_l", 3),
        _dev(counters, torch.int32, "counters", 1), maxp,
        none if order is None else _dev(order, torch.int32, "order", 1))


def pa_decode_step_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                 prefix_len, prefix_split, partition_size, workspace, counters,
                                 key=None, value=None, slot_mapping=None, stream=None,
                                 order=None):
    """pa_decode_step for a batch whose sequences all hold the same first
    prefix_len tokens (the same blocks as sequence 0) and go past them: the
    prefix in partitions of prefix_split tokens, the whole batch's queries
    against each on the tensor cores (one launch for all of them), and the
    rest by the split-K decode with the cache write (partitions of
    partition_size tokens from the prefix's end), merged in its last CTAs.  bf16 cache; workspace =
    shared_prefix_workspace(...); counters = step_counters(...); order
    (optional): shared_prefix_order(...) on the device."""
    args = _shared_prefix_args(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                               prefix_len, prefix_split, partition_size, workspace, counters, key,
                               value, slot_mapping, order)
    _check(lib().pa_decode_step_shared_prefix(*args, _stream(stream)),
           "pa_decode_step_shared_prefix")


class SharedPrefixStep:
    """One shared-prefix decode step of one layer on fixed device buffers
    (pa_decode_step_shared_prefix), its arguments checked and marshalled
    once; each call is one bare C call.  The buffers' contents may change
    between calls, their shapes and addresses may not."""

    def __init__(self, out, q, k_cache, v_cache, block_tables, context_lens, scale, prefix_len,
                 prefix_split, partition_size, workspace, counters, key=None, value=None,
                 slot_mapping=None, order=None, stream=None):
        self._args = _shared_prefix_args(out, q, k_cache, v_cache, block_tables, context_lens,
                                         scale, prefix_len, prefix_split, partition_size,
                                         workspace, counters, key, value, slot_mapping, order)
        self._stream = None if stream is None else ctypes.c_void_p(stream.cuda_stream)
        self._keep = [out, q, k_cache, v_cache, block_tables, context_lens, workspace, counters,
                      key, value, slot_mapping, order]

    def __call__(self):
        _check(lib().pa_decode_step_shared_prefix(*self._args, self._stream),
               "pa_decode_step_shared_prefix")

    def recover(self):
        """After a launch that raised PA_DEVERR_ORDER or PA_DEVERR_WAIT_TIMEOUT:
        re-zeroes this step's arrival counters and clears the error word
        (recover_step_counters).  Returns the error bits found."""
        return recover_step_counters(self._keep[7])


def shared_prefix_order(context_lens, prefix_len, partition_size, max_partitions,
                        prefix_split):
    """Longest-first work order (host numpy int32) of a shared-prefix step's
    second launch: pa_splitk_order of the lengths past the prefix over the
    partitions past the prefix's."""
    import numpy as np
    rest = np.maximum(np.asarray(context_lens, dtype=np.int64) - int(prefix_len), 0)
    return splitk_order(rest.astype(np.int32), partition_size,
                        int(max_partitions) - int(prefix_len) // int(prefix_split))


def pa_reshape_and_cache_fp8(key, value, k_cache, v_cache, k_scales, v_scales, slot_mapping,
                             stream=None):
    """key/value [T, Hkv, D] bf16 quantised into FP8 (E4M3) pools (uint8 codes) + fp32 scales."""
    torch = _torch()
    T, hkv, d = key.shape
    (pk, pv, pks, pvs), (nb, hkv2, bs, d2) = _int8_pools(k_cache, v_cache, k_scales, v_scales,
                                                         True)
    if value.shape != key.shape or (hkv, d) != (hkv2, d2) or slot_mapping.shape != (T,):
        raise ValueError("pa_reshape_and_cache_fp8: inconsistent shapes")
    st = lib().pa_reshape_and_cache_fp8(
        _dev(key, torch.bfloat16, "key", 3), _dev(value, torch.bfloat16, "value", 3), pk, pv,
        pks, pvs, _dev(slot_mapping, torch.int64, "slot_mapping", 1), T, hkv, d, bs, nb,
        _stream(stream))
    _check(st, "pa_reshape_and_cache_fp8")


def pa_decode_fp8(out, q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens,
                  scale, stream=None):
    torch = _torch()
    (pq, pk, pv, pks, pvs, pt, pc), (B, hq, hkv, d, bs, nb, mb) = _decode_int8_common(
        q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens, True)
    if out.shape != q.shape:
        raise ValueError("pa_decode_fp8: out must match q")
    st = lib().pa_decode_fp8(_dev(out, torch.bfloat16, "out", 3), pq, pk, pv, pks, pvs, pt, mb,
                             pc, B, hq, hkv, d, bs, nb, float(scale), _stream(stream))
    _check(st, "pa_decode_fp8")


def pa_decode_splitk_fp8(ws_out, ws_m, ws_l, q, k_cache, v_cache, k_scales, v_scales,
                         block_tables, context_lens, scale, partition_size=512, stream=None):
    torch = _torch()
    (pq, pk, pv, pks, pvs, pt, pc), (B, hq, hkv, d, bs, nb, mb) = _decode_int8_common(
        q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens, True)
    maxp = ws_m.shape[2]
    if ws_out.shape != (B, hq, maxp, d) or ws_l.shape != ws_m.shape or ws_m.shape[:2] != (B, hq):
        raise ValueError("pa_decode_splitk_fp8: workspace shapes")
    st = lib().pa_decode_splitk_fp8(
        _dev(ws_out, torch.float32, "ws_out", 4), _dev(ws_m, torch.float32, "ws_m", 3),
        _dev(ws_l, torch.float32, "ws_l", 3), maxp, pq, pk, pv, pks, pvs, pt, mb, pc, B, hq, hkv,
        d, bs, nb, float(scale), int(partition_size), _stream(stream))
    _check(st, "pa_decode_splitk_fp8")


def pa_decode_splitk_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                             max_context_len, partition_size=512, stream=None):
    """Split-K decode + merge with the library's built-in workspace.

    For callers that must not allocate device memory: nothing is allocated,
    by this binding or the library.  ``max_context_len`` bounds every context
    length; calls needing more than PA_DECODE_NOALLOC_WORKSPACE_BYTES of
    workspace raise PAError (invalid argument).  Concurrent calls on
    different streams share the workspace and race.
    """
    torch = _torch()
    (pq, pk, pv, pt, pc), (B, hq, hkv, d, bs, nb, mb) = _decode_common(
        q, k_cache, v_cache, block_tables, context_lens)
    if out.shape != q.shape:
        raise ValueError("pa_decode_splitk_noalloc: out must match q")
    st = lib().pa_decode_splitk_noalloc(_dev(out, torch.bfloat16, "out", 3), pq, pk, pv, pt, mb,
                                        pc, B, hq, hkv, d, bs, nb, float(scale),
                                        int(partition_size), int(max_context_len),
                                        _stream(stream))
    _check(st, "pa_decode_splitk_noalloc")


def pa_prefill(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
               max_query_len, scale, stream=None):
    """Causal attention of chunks of new tokens over the paged cache (pa.h).

    q, out [T, Hq, D] bf16; query_start_loc [B + 1] int32 (device);
    max_query_len: host bound on every chunk length.
    """
    torch = _torch()
    T, hq, d = q.shape
    if out.shape != q.shape:
        raise ValueError("pa_prefill: out must match q")
    nb, hkv, bs, d2 = k_cache.shape
    if v_cache.shape != k_cache.shape or d2 != d:
        raise ValueError("pa_prefill: cache shapes")
    B, mb = block_tables.shape
    if context_lens.shape != (B,) or query_start_loc.shape != (B + 1,):
        raise ValueError("pa_prefill: context_lens / query_start_loc shapes")
    st = lib().pa_prefill(_dev(out, torch.bfloat16, "out", 3), _dev(q, torch.bfloat16, "q", 3),
                          _dev(k_cache, torch.bfloat16, "k_cache", 4),
                          _dev(v_cache, torch.bfloat16, "v_cache", 4),
                          _dev(block_tables, torch.int32, "block_tables", 2), mb,
                          _dev(context_lens, torch.int32, "context_lens", 1),
                          _dev(query_start_loc, torch.int32, "query_start_loc", 1),
                          int(max_query_len), B, T, hq, hkv, d, bs, nb, float(scale),
                          _stream(stream))
    _check(st, "pa_prefill")


def pa_plan_step(budget, num_decodes, prefill_remaining):
    """(decodes scheduled, numpy int32 tokens per queued prefill) for one step."""
    import numpy as np
    rem = np.ascontiguousarray(prefill_remaining, dtype=np.int32)
    out = np.zeros_like(rem)
    dec = ctypes.c_int()
    _check(lib().pa_plan_step(int(budget), int(num_decodes),
                              rem.ctypes.data_as(ctypes.c_void_p), int(rem.shape[0]),
                              out.ctypes.data_as(ctypes.c_void_p), ctypes.byref(dec)),
           "pa_plan_step")
    return dec.value, out


class DecodeStep:
    """One decode step of one layer on fixed device buffers: the cache write
    of the batch's new tokens, then paged attention (split-K pass + merge, or
    the whole-sequence kernel).  fused=True (the default) makes it one
    pa_decode_step launch (each slot must then be its sequence's position
    context_lens[b] - 1); fused=False, the separate cache-write, partition
    and merge launches.  With partition_size=None and host_context_lens (a
    host copy of the lengths), the fused step picks its partition size and a
    longest-first work order for those lengths (plan_decode_step), with the
    workspace and order covering max_context_len tokens (default: the block
    tables' capacity, max_blocks_per_seq * block_size); any lengths up to that
    stay correct as they grow from call to call, only the speed may differ.
    After a launch that raised PA_DEVERR_ORDER or PA_DEVERR_WAIT_TIMEOUT,
    call recover() before the next one.

    Every argument is checked and marshalled once, here; each call then makes
    two or three bare C calls, which keeps the host ahead of the GPU when a
    step lasts only tens of microseconds.  The buffers' contents may change
    between calls (that is the point); their shapes and addresses may not.
    The split-K workspace is allocated with torch unless one is passed.
    """

    def __init__(self, key, value, k_cache, v_cache, slot_mapping, q, block_tables,
                 context_lens, out, scale, split=True, partition_size=512,
                 max_context_len=None, workspace=None, stream=None, k_scales=None,
                 v_scales=None, fused=True, counters=None, order=None, early_read=False,
                 host_context_lens=None):
        torch = _torch()
        self.fused = bool(fused)
        if self.fused:
            # one pa_decode_step* launch: write + attention (+ merge)
            self._stream = None if stream is None else ctypes.c_void_p(stream.cuda_stream)
            self.split = bool(split)
            B, hq, d = q.shape
            hkv = k_cache.shape[1]
            if self.split and host_context_lens is not None and partition_size is None:
                # chosen for these contexts (plan_decode_step): the partition
                # size for a longest-first launch, and that order.  The
                # workspace and the order cover the block tables' capacity
                # unless max_context_len says less, so the contexts may grow
                # from call to call up to that capacity.
                kind = ("fp8" if k_cache.dtype == torch.uint8 else
                        "int8" if k_cache.dtype == torch.int8 else "bf16")
                if max_context_len is None:
                    max_context_len = block_tables.shape[1] * k_cache.shape[2]
                plan = plan_decode_step(
                    host_context_lens, hq, hkv, d, kind,
                    torch.cuda.get_device_properties(q.device).multi_processor_count,
                    max_context_len=max_context_len)
                partition_size = plan.partition_size
                if order is None and plan.order is not None:
                    order = torch.from_numpy(plan.order).to(q.device)
            elif partition_size is None:
                partition_size = 512
            self.partition_size = partition_size
            if self.split:
                if workspace is None:
                    mc = (int(max_context_len) if max_context_len is not None
                          else block_tables.shape[1] * k_cache.shape[2])
                    workspace = splitk_workspace(B, hq, d, mc, partition_size, q.device)
                if counters is None:
                    counters = step_counters(B, hkv, q.device)
            self.workspace, self.counters = workspace, counters
            self._fn, self._args = _step_args(
                out, q, k_cache, v_cache, block_tables, context_lens, scale, key, value,
                slot_mapping, partition_size if self.split else 0, workspace, counters,
                k_scales, v_scales, order, early_read)
            self._keep = [key, value, k_cache, v_cache, slot_mapping, q, block_tables,
                          context_lens, out, workspace, counters, k_scales, v_scales, order]
            return
        if partition_size is None:
            partition_size = 512
        T, hkv, d = key.shape
        nb, hkv2, bs, d2 = k_cache.shape
        if value.shape != key.shape or v_cache.shape != k_cache.shape or (hkv, d) != (hkv2, d2):
            raise ValueError("DecodeStep: inconsistent key / cache shapes")
        if slot_mapping.shape != (T,):
            raise ValueError("DecodeStep: slot_mapping must be [num_tokens]")
        self.fp8 = k_cache.dtype == torch.uint8        # FP8 (E4M3) codes
        self.int8 = k_cache.dtype == torch.int8 or self.fp8  # a 1-byte cache with scales
        if self.int8:
            (pq, pk, pv, pks, pvs, pt, pc), (B, hq, _, _, _, _, mb) = _decode_int8_common(
                q, k_cache, v_cache, k_scales, v_scales, block_tables, context_lens, self.fp8)
        else:
            (pq, pk, pv, pt, pc), (B, hq, _, _, _, _, mb) = _decode_common(
                q, k_cache, v_cache, block_tables, context_lens)
        if out.shape != q.shape:
            raise ValueError("DecodeStep: out must match q")
        po = _dev(out, torch.bfloat16, "out", 3)
        self._keep = [key, value, k_cache, v_cache, slot_mapping, q, block_tables, context_lens,
                      out]
        self._stream = None if stream is None else ctypes.c_void_p(stream.cuda_stream)
        kv = (_dev(key, torch.bfloat16, "key", 3), _dev(value, torch.bfloat16, "value", 3))
        sm = _dev(slot_mapping, torch.int64, "slot_mapping", 1)
        if self.int8:
            self._keep += [k_scales, v_scales]
            self._rc = kv + (pk, pv, pks, pvs, sm, T, hkv, d, bs, nb)
        else:
            self._rc = kv + (pk, pv, sm, T, hkv, d, bs, nb)
        kvp = (pk, pv, pks, pvs) if self.int8 else (pk, pv)
        self.split = bool(split)
        if self.split:
            if workspace is None:
                mc = int(max_context_len) if max_context_len is not None else mb * bs
                workspace = splitk_workspace(B, hq, d, mc, partition_size, q.device)
            ws_o, ws_m, ws_l = workspace
            maxp = ws_m.shape[2]
            if ws_o.shape != (B, hq, maxp, d) or ws_l.shape != ws_m.shape:
                raise ValueError("DecodeStep: workspace shapes")
            self._keep += list(workspace)
            self.workspace = workspace
            wo = _dev(ws_o, torch.float32, "ws_out", 4)
            wm = _dev(ws_m, torch.float32, "ws_m", 3)
            wl = _dev(ws_l, torch.float32, "ws_l", 3)
            self._dk = (wo, wm, wl, maxp, pq) + kvp + (pt, mb, pc, B, hq, hkv, d, bs, nb,
                                                      float(scale), int(partition_size))
            self._rd = (po, wo, wm, wl, maxp, pc, B, hq, d, int(partition_size))
        else:
            self._dc = (po, pq) + kvp + (pt, mb, pc, B, hq, hkv, d, bs, nb, float(scale))
        L = lib()
        if self.fp8:
            self._f_write, self._f_split, self._f_whole = (
                L.pa_reshape_and_cache_fp8, L.pa_decode_splitk_fp8, L.pa_decode_fp8)
        elif self.int8:
            self._f_write, self._f_split, self._f_whole = (
                L.pa_reshape_and_cache_int8, L.pa_decode_splitk_int8, L.pa_decode_int8)
        else:
            self._f_write, self._f_split, self._f_whole = (
                L.pa_reshape_and_cache, L.pa_decode_splitk, L.pa_decode)

    def recover(self):
        """Reads the device error word (synchronises); after PA_DEVERR_ORDER
        or PA_DEVERR_WAIT_TIMEOUT re-zeroes this step's arrival counters and
        clears the word.  Returns the error bits found."""
        if self.fused and self.split and self.counters is not None:
            return recover_step_counters(self.counters)
        return pa_get_device_error()

    def __call__(self, stream=None):
        s = self._stream if stream is None and self._stream is not None else _stream(stream)
        if self.fused:
            st = self._fn(*self._args, s)
            if st != PA_OK:
                _check(st, "DecodeStep: pa_decode_step")
            return
        st = self._f_write(*self._rc, s)
        if st != PA_OK:
            _check(st, "DecodeStep: cache write")
        if self.split:
            st = self._f_split(*self._dk, s)
            if st != PA_OK:
                _check(st, "DecodeStep: split-K partition pass")
            st = _lib.pa_splitk_reduce(*self._rd, s)
            if st != PA_OK:
                _check(st, "DecodeStep: pa_splitk_reduce")
        else:
            st = self._f_whole(*self._dc, s)
            if st != PA_OK:
                _check(st, "DecodeStep: decode")


def pa_get_device_error():
    v = ctypes.c_uint(0)
    _check(lib().pa_get_device_error(ctypes.byref(v)), "pa_get_device_error")
    return v.value


def pa_clear_device_error():
    _check(lib().pa_clear_device_error(), "pa_clear_device_error")


# --------------------------------------------------------------------------
# host block allocator (no GPU needed)

class BlockAllocator:
    """Wraps pa_alloc_* (include/pa.h).  numpy arrays in and out."""

    def __init__(self, num_blocks, block_size, initial_free_order=None):
        import numpy as np
        self._np = np
        h = ctypes.c_void_p()
        order = None
        if initial_free_order is not None:
            order = np.ascontiguousarray(initial_free_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("initial_free_order must have num_blocks entries")
        st = lib().pa_alloc_create(num_blocks, block_size,
                                   None if order is None else order.ctypes.data_as(_vp),
                                   ctypes.byref(h))
        _check(st, "pa_alloc_create")
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if getattr(self, "_h", None):
            lib().pa_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq):
        _check(lib().pa_alloc_add_seq(self._h, seq), "pa_alloc_add_seq")

    def append_slot(self, seq):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib().pa_alloc_append_slot(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                          ctypes.byref(dst)), "pa_alloc_append_slot")
        return slot.value, src.value, dst.value

    def append_slots(self, seqs):
        np = self._np
        ids = np.ascontiguousarray(seqs, dtype=np.intc)
        n = ids.shape[0]
        slots = np.empty(n, dtype=np.int64)
        src = np.empty(n, dtype=np.int32)
        dst = np.empty(n, dtype=np.int32)
        _check(lib().pa_alloc_append_slots(self._h, ids.ctypes.data_as(_vp), n,
                                           slots.ctypes.data_as(_vp), src.ctypes.data_as(_vp),
                                           dst.ctypes.data_as(_vp)), "pa_alloc_append_slots")
        return slots, src, dst

    def reserve(self, seq, num_tokens):
        src, dst = ctypes.c_int32(), ctypes.c_int32()
        _check(lib().pa_alloc_reserve(self._h, seq, int(num_tokens), ctypes.byref(src),
                                      ctypes.byref(dst)), "pa_alloc_reserve")
        return src.value, dst.value

    def fork(self, parent, child):
        _check(lib().pa_alloc_fork(self._h, parent, child), "pa_alloc_fork")

    def free_seq(self, seq):
        _check(lib().pa_alloc_free_seq(self._h, seq), "pa_alloc_free_seq")

    def block_table(self, seq):
        np = self._np
        n = ctypes.c_int()
        _check(lib().pa_alloc_block_table(self._h, seq, None, 0, ctypes.byref(n)),
               "pa_alloc_block_table")
        out = np.empty(n.value, dtype=np.int32)
        _check(lib().pa_alloc_block_table(self._h, seq, out.ctypes.data_as(_vp), n.value,
                                          ctypes.byref(n)), "pa_alloc_block_table")
        return out

    def block_tables(self, seqs, max_blocks):
        np = self._np
        ids = np.ascontiguousarray(seqs, dtype=np.intc)
        out = np.empty((ids.shape[0], max_blocks), dtype=np.int32)
        ctx = np.empty(ids.shape[0], dtype=np.int32)
        _check(lib().pa_alloc_block_tables(self._h, ids.ctypes.data_as(_vp), ids.shape[0],
                                           out.ctypes.data_as(_vp), max_blocks,
                                           ctx.ctypes.data_as(_vp)), "pa_alloc_block_tables")
        return out, ctx

    def seq_len(self, seq):
        return int(lib().pa_alloc_seq_len(self._h, seq))

    def refcount(self, blk):
        return int(lib().pa_alloc_refcount(self._h, blk))

    def num_free(self):
        return int(lib().pa_alloc_num_free(self._h))

    def free_list(self):
        np = self._np
        n = ctypes.c_int()
        out = np.empty(self.num_blocks, dtype=np.int32)
        _check(lib().pa_alloc_free_list(self._h, out.ctypes.data_as(_vp), self.num_blocks,
                                        ctypes.byref(n)), "pa_alloc_free_list")
        return out[:n.value]

    def tail_waste(self, seq):
        return int(lib().pa_alloc_tail_waste(self._h, seq))

    # automatic prefix caching
    def enable_prefix_cache(self):
        _check(lib().pa_alloc_enable_prefix_cache(self._h), "pa_alloc_enable_prefix_cache")

    def add_seq_prompt(self, seq, tokens, salt=b""):
        """Registers a sequence with its prompt; returns the number of cached tokens."""
        np = self._np
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        salt = bytes(salt)
        n = ctypes.c_int()
        _check(lib().pa_alloc_add_seq_prompt(self._h, seq, tok.ctypes.data_as(_vp), tok.shape[0],
                                              salt if salt else None, len(salt), ctypes.byref(n)),
               "pa_alloc_add_seq_prompt")
        return n.value

    def num_evictable(self):
        return int(lib().pa_alloc_num_evictable(self._h))

    def evictable_list(self):
        np = self._np
        n = ctypes.c_int()
        out = np.empty(self.num_blocks, dtype=np.int32)
        _check(lib().pa_alloc_evictable_list(self._h, out.ctypes.data_as(_vp), self.num_blocks,
                                             ctypes.byref(n)), "pa_alloc_evictable_list")
        return out[:n.value]


def pa_prefix_root_hash(salt=b""):
    out = (ctypes.c_uint8 * 32)()
    salt = bytes(salt)
    _check(lib().pa_prefix_root_hash(salt if salt else None, len(salt), out), "pa_prefix_root_hash")
    return bytes(out)


def pa_prefix_block_hash(parent, tokens):
    import numpy as np
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    par = (ctypes.c_uint8 * 32)(*bytes(parent))
    out = (ctypes.c_uint8 * 32)()
    _check(lib().pa_prefix_block_hash(par, tok.ctypes.data_as(_vp), tok.shape[0], out),
           "pa_prefix_block_hash")
    return bytes(out)
