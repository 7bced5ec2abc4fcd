"""GB300-native PagedAttention decode: KV cache write and paged GQA decode.

The compute path lives in ``libpa.so`` (hand-written CUDA for sm_103a plus a
C++ host block allocator, C ABI declared in ``include/pa.h``).  ``pa`` is its
thin ctypes binding; ``inputs`` draws seeded synthetic workloads.  Importing
this package loads nothing; ``pa`` loads the library on first use and raises
if it is missing.
"""
