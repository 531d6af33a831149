"""Plain CPU oracle for paged decode attention and its cache-feeding ops.

TEST INFRASTRUCTURE ONLY.  This package is a slow, obviously correct restatement
of what the paged attention path computes, written in NumPy float64 and plain
Python loops.  It exists so that the CUDA path can be checked against something
that shares none of its code.  Only the test suite, the smoke check and the
CPU-baseline leg of the benchmark may import it; the product path never does,
and there is no CPU fallback through it.

Modules
-------
attention   gather through the block table + textbook softmax attention
            (with grouped-query head sharing) and the exact block merge.
cache_ops   slot-mapping scatter (reshape_and_cache) and copy-on-write block
            copy (copy_blocks) on a host copy of the pool.
allocator   reference block manager: LIFO free list, reference counts, fork,
            append with copy-on-write, release.
sizing      KV-cache sizing arithmetic (bytes per token, blocks, tail waste).

Sources (the three web pages this method is described on):
  [P1] "PagedAttention: Virtual Memory for the KV Cache" (int8ai.pages.dev)
  [P2] "PagedAttention in vLLM: scattered memory, exact attention"
       (abhiram1809.github.io)
  [P3] "PagedAttention and KV Memory" (blog.michaelsam94.com)

Every function is pinned by tests under tests/ to values the pages print,
closed forms, invariants or brute force; none is marked "parity unpinned".
"""

from . import allocator, attention, cache_ops, sizing  # noqa: F401
