"""CPU oracle for PagedAttention decode: TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct restatement of what the
paged decode path computes, written in numpy float64 (and pure Python for the
block allocator).  It exists so that the tests, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` have
something independent to compare the CUDA path against.  Nothing in the
product package (``paged_kv_cache_283_gb300``) imports it, and it imports
nothing from there: the two sides share no kernels, headers, helpers or
constants.  Only the seeded input generators (``paged_kv_cache_283_gb300.inputs``)
feed both, and those hold none of the method's arithmetic.

Sources (by page title and section):

* "How LLM Inference Serving Works: KV Cache, PagedAttention and Continuous
  Batching" (dev.to) -- sections "What the KV Cache Is, and How Big It Gets",
  "PagedAttention: Virtual Memory for the KV Cache", "Sharing comes for free",
  "Two Phases: Prefill and Decode", "Chunked prefill" and "Putting It
  Together: The Life of a Request in vLLM".
* "LLM serving (vLLM, quantized inference): Visual walkthrough" -- Steps 1-8
  and the quick self-check.

Modules:

* ``bf16``       exact bf16 -> float64 decoding of raw bit patterns.
* ``kv_size``    the KV-cache byte formulas and the paged / naive waste counts.
* ``attention``  block-table gather + dense softmax attention, per-partition
                 statistics and the log-sum-exp merge.
* ``prefill``    causal attention of a chunk of new tokens over the paged
                 cache (chunked prefill; one token = one decode step).
* ``scheduler``  the chunked-prefill step budget (decodes first, then
                 prefill chunks in queue order).
* ``fp8``        the FP8 (E4M3) KV scheme: the format from its definition,
                 per-row quantisation, the FP8 cache write and decode.
* ``quant``      the INT8 KV scheme: per-row quantisation, the INT8 cache
                 write and the INT8 decode.
* ``cache``      the cache write (scatter of new K/V through a slot mapping).
* ``allocator``  a pure-Python block allocator model (FIFO free list,
                 refcounts, fork / copy-on-write, free).

Every function is pinned by a ``-m "not gpu"`` test against values the pages
print, closed forms, library routines or brute force; none is marked
"parity unpinned".
"""
