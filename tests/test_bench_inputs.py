"""Host-side inputs of the bench workloads, pinned to the oracle: the
copy-on-write pairs of the CoW sampling config (16 prompts of 2,003 tokens,
8 samples each, one appended token per sample) that the cache-ops workload
copies come from the C++ block manager; the oracle allocator replaying the
same operations must plan the same pairs, and their number follows from the
pages' rule that each writer of a shared tail block copies it except the
last ("PagedAttention: Virtual Memory for the KV Cache", sections 15-16)."""
import numpy as np
import pytest

api = pytest.importorskip("paged_kv_cache_124_gb300.api")

import bench  # noqa: E402
from oracle.allocator import RefAllocator  # noqa: E402


def test_cow_pairs_match_the_oracle_allocator():
    sc, slots, pairs, nb = bench._cache_ops_inputs(0, 16, api)
    n_prompts, samples = len(sc.ctxs), 8
    ref = RefAllocator(nb, sc.block_size)
    assert ref.set_free_order(list(sc.free_order) + list(range(sc.num_blocks, nb))) == 0
    for s, c in enumerate(sc.ctxs):
        assert ref.allocate(s * samples, c) == 0
        for f in range(1, samples):
            assert ref.fork(s * samples, s * samples + f) == 0
    want = []
    for s in range(n_prompts * samples):
        st, _, src, dst = ref.append_slot(s)
        assert st == 0
        if src >= 0:
            want.append((src, dst))
    assert pairs.tolist() == [list(p) for p in want]
    # 2,003 = 125 * 16 + 3: the tail block is shared by 8 samples; the first 7
    # writers copy it, the 8th writes in place
    assert len(pairs) == n_prompts * (samples - 1) == 112
    srcs = pairs[:, 0].tolist()
    assert len(set(srcs)) == n_prompts and all(srcs.count(x) == samples - 1 for x in set(srcs))
    assert len(set(pairs[:, 1].tolist())) == len(pairs)             # fresh destinations
    assert not set(pairs[:, 1].tolist()) & set(srcs)


def test_prefill_slots_are_the_new_positions_of_each_prompt():
    sc, slots, _, _ = bench._cache_ops_inputs(0, 16, api)
    assert len(slots) == sum(sc.news) == 16 * 2003
    assert len(set(slots.tolist())) == len(slots)                   # one slot per position
    assert slots.min() >= 0 and slots.max() < sc.num_blocks * sc.block_size
