"""Helpers shared by the GPU parity tests: moving seeded inputs to the
device, building block tables on both sides, and the tolerance gate.

Block tables for the oracle side come from the oracle's allocator model and
for the CUDA side from the C++ allocator; the two are asserted identical
before either is used.
"""
import numpy as np
import torch

from oracle.allocator import BlockAllocatorModel
from paged_kv_cache_283_gb300 import pa

# Tolerance on attention outputs versus the float64 oracle: max-abs 2e-2 and
# max-rel 1e-2 (relative error over elements with |ref| > 2e-2), plus a
# normwise 1e-2 per (sequence, head) so that small outputs are checked too.
ATOL = 2e-2
RTOL = 1e-2
NORM_RTOL = 1e-2


def dev_bf16(bits):
    """uint16 bf16 bit patterns (numpy) -> torch.bfloat16 on cuda, same bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to("cuda").view(torch.bfloat16)


def host_bits(t):
    """torch.bfloat16 -> numpy uint16 bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def model_tables(w, step_append=True):
    """(block_tables [B, MB] int32, slots [B] int64) from the oracle's allocator model."""
    m = BlockAllocatorModel(w.num_blocks, w.block_size, w.free_order)
    for b, n in enumerate(w.context_lens.tolist()):
        m.add_seq(b)
        m.reserve(b, n - 1 if step_append else n)
    slots = [x[0] for x in m.append_slots(range(w.num_seqs))] if step_append else []
    mb = max(1, w.max_blocks_per_seq)
    bt = np.full((w.num_seqs, mb), -1, dtype=np.int32)
    for b in range(w.num_seqs):
        t = m.block_table(b)
        bt[b, :len(t)] = t
    return bt, np.array(slots, dtype=np.int64)


def product_tables(w):
    """Same as model_tables, through the C++ allocator."""
    a = pa.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    for b, n in enumerate(w.context_lens.tolist()):
        a.add_seq(b)
        a.reserve(b, n - 1)
    slots, _, _ = a.append_slots(list(range(w.num_seqs)))
    bt, ctx = a.block_tables(list(range(w.num_seqs)), max(1, w.max_blocks_per_seq))
    assert np.array_equal(ctx, w.context_lens)
    return bt, slots


def both_tables(w):
    bt_m, sl_m = model_tables(w)
    bt_p, sl_p = product_tables(w)
    assert np.array_equal(bt_m, bt_p) and np.array_equal(sl_m, sl_p)
    return bt_m, sl_m, bt_p, sl_p


def assert_close(got, ref, what=""):
    """The tolerance gate on [..., D] arrays (float64)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    d = np.abs(got - ref)
    amax = float(d.max()) if d.size else 0.0
    assert amax <= ATOL, f"{what}: max abs err {amax:.3e} > {ATOL}"
    big = np.abs(ref) > ATOL
    if big.any():
        rmax = float((d[big] / np.abs(ref[big])).max())
        assert rmax <= RTOL, f"{what}: max rel err {rmax:.3e} > {RTOL}"
    num = np.linalg.norm((got - ref).reshape(-1, ref.shape[-1]), axis=1)
    den = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=1)
    nz = den > 0
    if nz.any():
        nmax = float((num[nz] / den[nz]).max())
        assert nmax <= NORM_RTOL, f"{what}: normwise rel err {nmax:.3e} > {NORM_RTOL}"
    assert np.all(num[~nz] == 0), f"{what}: nonzero output where the reference is zero"
    return amax


def v_tile_positions(d):
    """[16, d] int array: the byte offset, within one (block, head) tile of a
    1-byte V pool, of token t's code of dim j, as the library's header states:
    L * (d/2) + 16 * ((w // 4) ^ f) + 4 * (w % 4) + y with r = j % 16,
    L = 4 * (r % 8) + (t % 8) // 2, w = 2 * (j // 16) + r // 8,
    y = (t % 2) + 2 * (t // 8), f = (L // 2) % 4 at d = 128, (L // 4) % 2 at 64."""
    t = np.arange(16)[:, None]
    j = np.arange(d)[None, :]
    r = j % 16
    L = 4 * (r % 8) + (t % 8) // 2
    w = 2 * (j // 16) + r // 8
    y = (t % 2) + 2 * (t // 8)
    f = (L // 2) % 4 if d == 128 else (L // 4) % 2
    return L * (d // 2) + 16 * ((w // 4) ^ f) + 4 * (w % 4) + y


def v_pool_stored(v, fp8):
    """The 1-byte V pool as the device stores it, from logical codes
    [NB, Hkv, 16, D] (int8 INT8 codes, or uint8 E4M3 codes): each tile
    transposed by v_tile_positions, INT8 codes offset by 128."""
    v = np.ascontiguousarray(v)
    nb, hkv, bs, d = v.shape
    src = v.reshape(nb, hkv, bs * d).view(np.uint8)
    if not fp8:
        src = src ^ np.uint8(0x80)
    out = np.empty_like(src)
    out[:, :, v_tile_positions(d).reshape(-1)] = src
    out = out.reshape(v.shape)
    return out if fp8 else out.view(np.int8)


def v_pool_logical(v, fp8):
    """Inverse of v_pool_stored: logical codes from the device's V pool bytes."""
    v = np.ascontiguousarray(v)
    nb, hkv, bs, d = v.shape
    out = v.reshape(nb, hkv, bs * d).view(np.uint8)[:, :, v_tile_positions(d).reshape(-1)]
    if not fp8:
        out = out ^ np.uint8(0x80)
    out = out.reshape(v.shape)
    return out if fp8 else out.view(np.int8)
