"""Oracle for the paged KV-cache hot path — TEST INFRASTRUCTURE.

Plain, slow, obviously-correct CPU implementations of what the GPU path
computes, written from the pages (cited per function):

  attention.py      paged and contiguous decode attention in float64
                    (C loops in pa_oracle.c, loaded through ctypes)
  kvcache.py        address translation, KV append and block copy on raw bits
  block_manager.py  free pool, reference counts, copy-on-write and the
                    parent-chained block hash, as naive Python lists/dicts

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
(``--impl reference``) leg may import or run anything in this package.  The
CUDA library never does, and shares no code with it.

Parity pins: every function here is checked by ``tests/test_oracle_*.py``
against something other than itself (the pages' worked example, closed forms,
library routines, invariants, brute force).  The choice of FNV-1a-64 as the
block hash is this build's own (the pages only fix the parent chaining); the
hash function is pinned to FNV's published test vectors, its use as the block
key is "parity unpinned" beyond the chaining invariants.
"""
