"""The C-ABI library loads on a machine without a GPU and exports every
function include/pa.h declares; the binding declares exactly those names.
Host-side argument checks are exercised without touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_cache_283_gb300 import pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(pa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pa.LIB_PATH):
        from paged_kv_cache_283_gb300 import build
        build.build()
    return pa.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["pa_reshape_and_cache", "pa_decode", "pa_decode_splitk", "pa_splitk_reduce",
                 "pa_splitk_workspace_bytes", "pa_alloc_create", "pa_alloc_append_slot",
                 "pa_alloc_fork", "pa_alloc_free_seq", "pa_alloc_block_table"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True,
                        text=True)
    if nm.returncode == 0:
        exported = set(line.split()[-1] for line in nm.stdout.splitlines() if line.strip())
        assert set(declared_functions()) <= exported


def test_binding_covers_exactly_the_header():
    assert sorted(pa.SIGNATURES) == declared_functions()


def test_status_strings(lib):
    for s in range(5):
        assert lib.pa_status_string(s)
    assert b"unknown" in lib.pa_status_string(99)


def test_supported_shapes(lib):
    assert lib.pa_decode_supported(32, 8, 128, 16) == pa.PA_OK
    assert lib.pa_decode_supported(4, 2, 64, 16) == pa.PA_OK
    assert lib.pa_decode_supported(32, 8, 96, 16) == pa.PA_ERR_UNSUPPORTED_SHAPE
    assert lib.pa_decode_supported(32, 8, 128, 32) == pa.PA_ERR_UNSUPPORTED_SHAPE
    assert lib.pa_decode_supported(32, 32, 128, 16) == pa.PA_ERR_UNSUPPORTED_SHAPE
    assert lib.pa_decode_supported(30, 8, 128, 16) == pa.PA_ERR_INVALID_ARG


def test_host_checks_reject_before_any_launch(lib):
    # Null or misaligned pointers and bad sizes are refused on the host, so
    # these calls never reach CUDA.  Every call below fails a host check: none
    # may pass them, since the fake addresses must never reach a kernel.
    fake = ctypes.c_void_p(0x10000)
    mis = ctypes.c_void_p(0x10008)
    st = lib.pa_decode(None, fake, fake, fake, fake, 4, fake, 2, 32, 8, 128, 16, 10, 0.1, None)
    assert st == pa.PA_ERR_INVALID_ARG
    st = lib.pa_decode(fake, mis, fake, fake, fake, 4, fake, 2, 32, 8, 128, 16, 10, 0.1, None)
    assert st == pa.PA_ERR_INVALID_ARG
    st = lib.pa_decode(fake, fake, fake, fake, fake, 4, fake, 2, 32, 8, 96, 16, 10, 0.1, None)
    assert st == pa.PA_ERR_UNSUPPORTED_SHAPE
    st = lib.pa_decode(fake, fake, fake, fake, fake, 0, fake, 2, 32, 8, 128, 16, 10, 0.1, None)
    assert st == pa.PA_ERR_INVALID_ARG
    st = lib.pa_decode(fake, fake, fake, fake, fake, 4, fake, 70000, 32, 8, 128, 16, 10, 0.1, None)
    assert st == pa.PA_ERR_UNSUPPORTED_SHAPE
    st = lib.pa_reshape_and_cache(fake, fake, fake, fake, fake, 3, 8, 100, 16, 10, None)
    assert st == pa.PA_ERR_INVALID_ARG               # head_dim not a multiple of 8
    st = lib.pa_reshape_and_cache(fake, fake, fake, fake, ctypes.c_void_p(0x10004), 3, 8, 128,
                                  16, 10, None)
    assert st == pa.PA_ERR_INVALID_ARG               # int64 slots must be 8-byte aligned
    st = lib.pa_reshape_and_cache(None, None, None, None, None, 0, 8, 128, 16, 10, None)
    assert st == pa.PA_OK                            # nothing to do
    st = lib.pa_decode_splitk(fake, fake, fake, 4, fake, fake, fake, fake, 4, fake, 2, 32, 8,
                              128, 16, 10, 0.1, 100, None)
    assert st == pa.PA_ERR_INVALID_ARG               # partition not a multiple of 16
    st = lib.pa_splitk_reduce(fake, fake, fake, fake, 4, fake, 2, 32, 96, 512, None)
    assert st == pa.PA_ERR_UNSUPPORTED_SHAPE
    # pa_prefill: the kernel takes row maxima of unscaled scores, so scale > 0
    for scale in (0.0, -0.1, float("nan")):
        st = lib.pa_prefill(fake, fake, fake, fake, fake, 4, fake, fake, 8, 2, 16, 32, 8, 128,
                            16, 10, scale, None)
        assert st == pa.PA_ERR_INVALID_ARG
    st = lib.pa_prefill(fake, fake, fake, fake, fake, 4, fake, fake, 8, 2, 16, 32, 8, 64, 16,
                        10, 0.1, None)
    assert st == pa.PA_ERR_UNSUPPORTED_SHAPE         # head_dim 128 only


def test_workspace_bytes(lib):
    # [B, Hq, P, D] + 2 [B, Hq, P] fp32, P = ceil(max_ctx / partition)
    B, hq, d = 8, 32, 128
    P = -(-131072 // 512)
    assert pa.pa_splitk_workspace_bytes(B, hq, d, 131072, 512) == 4 * B * hq * P * (d + 2)
    assert pa.pa_splitk_workspace_bytes(1, 1, 64, 1, 512) == 4 * 66
    assert pa.pa_splitk_workspace_bytes(1, 1, 64, 10, 0) == 0


def test_decode_step_host_checks(lib):
    # pa_decode_step's own checks (write arguments together, split-K
    # workspace and counters, work order, flags); every call fails one of them
    # before any CUDA call, so the fake addresses never reach a kernel.
    f = ctypes.c_void_p(0x10000)

    def call(out=f, key=f, value=f, slots=f, partition=512, ws=f, counters=f, maxp=4,
             order=None, flags=0, num_seqs=2):
        return lib.pa_decode_step(out, f, key, value, slots, f, f, f, 4, f, num_seqs, 32, 8,
                                  128, 16, 10, 0.1, partition, ws, ws, ws, counters, maxp,
                                  order, flags, None)

    assert call(out=None) == pa.PA_ERR_INVALID_ARG
    assert call(value=None) == pa.PA_ERR_INVALID_ARG            # key, value, slots together
    assert call(slots=ctypes.c_void_p(0x10004)) == pa.PA_ERR_INVALID_ARG  # int64 slots aligned
    assert call(partition=-16) == pa.PA_ERR_INVALID_ARG
    assert call(partition=100) == pa.PA_ERR_INVALID_ARG         # not a multiple of 16
    assert call(maxp=0) == pa.PA_ERR_INVALID_ARG
    assert call(counters=None) == pa.PA_ERR_INVALID_ARG         # split-K needs counters
    assert call(ws=None) == pa.PA_ERR_INVALID_ARG               # and a workspace
    assert call(flags=2) == pa.PA_ERR_INVALID_ARG               # unknown flag bit
    assert call(order=f, partition=0) == pa.PA_ERR_INVALID_ARG  # an order needs split-K
    assert call(order=f, num_seqs=300, maxp=300) == pa.PA_ERR_UNSUPPORTED_SHAPE
    assert call(num_seqs=0, out=None) == pa.PA_OK               # nothing to do


def test_shared_prefix_step_host_checks(lib):
    # pa_decode_step_shared_prefix's own checks; each call fails one of them
    # before any CUDA call (fake addresses never reach a kernel)
    f = ctypes.c_void_p(0x10000)

    def call(prefix=512, split=256, part=256, maxp=4, d=128, hkv=8, seqs=2, out=f, counters=f,
             scale=0.1):
        return lib.pa_decode_step_shared_prefix(out, f, None, None, None, f, f, f, 64, f, seqs, 32,
                                                hkv, d, 16, 100, scale, prefix, split, part, f, f,
                                                f, counters, maxp, None, None)

    assert call(prefix=0) == pa.PA_ERR_INVALID_ARG
    assert call(scale=0.0) == pa.PA_ERR_INVALID_ARG         # the prefill kernel: scale > 0
    assert call(scale=-0.1) == pa.PA_ERR_INVALID_ARG
    assert call(prefix=300) == pa.PA_ERR_INVALID_ARG        # not a multiple of the split
    assert call(split=100) == pa.PA_ERR_INVALID_ARG         # not a multiple of the block
    assert call(part=100) == pa.PA_ERR_INVALID_ARG
    assert call(maxp=2) == pa.PA_ERR_INVALID_ARG            # no partition left past the prefix
    assert call(counters=None) == pa.PA_ERR_INVALID_ARG     # the merge needs counters
    assert call(prefix=2048) == pa.PA_ERR_INVALID_ARG       # longer than the tables
    assert call(d=64) == pa.PA_ERR_UNSUPPORTED_SHAPE        # the prefill kernel's shapes only
    assert call(hkv=2) == pa.PA_ERR_UNSUPPORTED_SHAPE       # group of 16
    assert call(out=None) == pa.PA_ERR_INVALID_ARG
    assert call(seqs=0) == pa.PA_OK
