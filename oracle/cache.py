"""The cache write, restated plainly (oracle, test-only).

Each decode step appends one token's K and V into the request's current block
("How LLM Inference Serving Works", section "Putting It Together: The Life of
a Request in vLLM"); the keys and values are stored once and never recomputed
("What the KV Cache Is, and How Big It Gets").  The position a token lands in
is given by a slot number: slot = physical_block * block_size + offset, and a
negative slot marks a padding token that is not written.  The slot encoding
and the pool layout [num_blocks, Hkv, bs, D] are not stated on the pages; they
are the plainest reading of "a block table maps each logical block to a
physical block" with fixed-size blocks.

This is a bit copy: arrays of raw bf16 bit patterns go in and come out.

``copy_blocks`` is the copy half of copy-on-write ("Sharing comes for free": a
shared block is copied only when one branch needs to write into it): for each
(source, destination) pair the whole destination block takes the source
block's contents, in every layer's K and V pool.
"""
import numpy as np


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, block_size,
                      inplace=False):
    """Write key[t], value[t] ([T, Hkv, D]) at slot_mapping[t] of the pools.

    Returns the (k_cache, v_cache) pair that results; the inputs are copied
    first unless ``inplace`` is set.
    """
    kc = k_cache if inplace else np.array(k_cache, copy=True)
    vc = v_cache if inplace else np.array(v_cache, copy=True)
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        kc[blk, :, off, :] = key[t]
        vc[blk, :, off, :] = value[t]
    return kc, vc


def copy_blocks(k_caches, v_caches, pairs, inplace=False):
    """Copy block src to block dst for every (src, dst) in ``pairs``, in every
    layer's pools; returns the lists of resulting pools."""
    ks = [k if inplace else np.array(k, copy=True) for k in k_caches]
    vs = [v if inplace else np.array(v, copy=True) for v in v_caches]
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        for k, v in zip(ks, vs):
            k[dst] = k[src]
            v[dst] = v[src]
    return ks, vs
