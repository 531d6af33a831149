"""C ABI on the host: the library loads, exports every declared symbol, and
its block manager matches the reference allocator operation by operation.
No GPU needed (the block manager is host code)."""
import ctypes

import numpy as np
import pytest

from oracle import allocator as AL
from _golden import load

api = pytest.importorskip("paged_kv_cache_124_gb300.api")


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(api.library_path())
    names = api.header_functions()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert "sm_103a" in api.version()
    assert api.status_string(api.PA_FAIL_NO_BLOCKS).startswith("no free blocks")


def test_fixed_partition_workspace_size():
    assert api.pa_decode_workspace_size(64, 32, 128, 512, 512) == 0
    n = api.pa_decode_workspace_size(64, 32, 128, 4096, 512)
    parts = 64 * 32 * 8
    al = lambda x: (x + 255) // 256 * 256
    # a 256-byte header (the claim counters), then the maxima, the sums and the value sums
    assert n == 256 + 2 * al(parts * 4) + al(parts * 128 * 4)


def test_prefill_workspace_size():
    """V staging (KV heads x sequences x positions rounded up to 128 x d_head
    x 2 bytes) plus one format byte per 128 positions, each part rounded up
    to 256 bytes."""
    # 16 prompts of 126 blocks of 16 (2,016 positions -> 2,048), 8 KV heads, d 128
    stage = 8 * 16 * 2048 * 128 * 2
    assert api.pa_prefill_workspace_size(16, 126, 16, 8, 128) == stage + 256 * -(-(8 * 16 * 16) // 256)
    # 300 positions -> 384 (3 tiles): 2 x 3 x 384 x 64 x 2 = 294,912 bytes, 18 format bytes -> 256
    assert api.pa_prefill_workspace_size(3, 10, 30, 2, 64) == 294912 + 256
    assert api.pa_prefill_workspace_size(0, 10, 16, 2, 64) == 0
    assert api.pa_prefill_workspace_size(3, 10, 16, 2, -1) == 0


STATUS_MAP = {AL.OK: api.PA_OK, AL.FAIL_NO_BLOCKS: api.PA_FAIL_NO_BLOCKS, AL.ERR_INVALID_ARG: api.PA_ERR_INVALID_ARG,
              AL.ERR_UNKNOWN_SEQ: api.PA_ERR_UNKNOWN_SEQ, AL.ERR_DUPLICATE_SEQ: api.PA_ERR_DUPLICATE_SEQ}


def _same_state(ref, dut, seqs):
    assert dut.free_list() == ref.free_blocks
    assert [dut.ref_count(b) for b in range(ref.num_blocks)] == ref.ref_counts
    for s in seqs:
        if s in ref.block_tables:
            assert dut.block_table(s) == ref.block_tables[s]
            assert dut.seq_len(s) == ref.seq_lengths[s]
        else:
            assert dut.seq_len(s) == -1


@pytest.mark.parametrize("seed,B,NB", [(0, 4, 24), (1, 8, 64), (2, 16, 16), (3, 1, 40)])
def test_block_manager_matches_reference_under_random_ops(seed, B, NB):
    rng = np.random.default_rng(seed)
    ref, dut = AL.RefAllocator(NB, B), api.BlockAllocator(NB, B)
    perm = rng.permutation(NB)
    assert STATUS_MAP[ref.set_free_order(perm)] == dut.set_free_order(perm)
    seqs = list(range(12))
    for _ in range(4000):
        op = int(rng.integers(0, 5))
        s = int(rng.choice(seqs))
        if op == 0:
            n = int(rng.integers(-1, 5 * B))
            assert STATUS_MAP[ref.allocate(s, n)] == dut.allocate(s, n)
        elif op == 1:
            c = int(rng.choice(seqs))
            assert STATUS_MAP[ref.fork(s, c)] == dut.fork(s, c)
        elif op in (2, 3):
            r = ref.append_slot(s)
            d = dut.append_slot(s)
            assert (STATUS_MAP[r[0]],) + tuple(r[1:]) == d
        else:
            assert STATUS_MAP[ref.free(s)] == dut.free(s)
    _same_state(ref, dut, seqs)
    st = dut.stats()
    assert st["num_free"] == ref.num_free() and st["num_cow_copies"] == ref.num_cow_copies


def test_batch_append_matches_sequential_reference():
    rng = np.random.default_rng(9)
    ref, dut = AL.RefAllocator(200, 8), api.BlockAllocator(200, 8)
    for s in range(10):
        n = int(rng.integers(1, 30))
        assert ref.allocate(s, n) == 0 and dut.allocate(s, n) == 0
    for s in range(10, 20):
        assert ref.fork(s - 10, s) == 0 and dut.fork(s - 10, s) == 0
    for _ in range(5):
        batch = [int(x) for x in rng.permutation(20)]
        st, slots, pairs, done = dut.append_slots(batch)
        want_slots, want_pairs = [], []
        for s in batch:
            r = ref.append_slot(s)
            want_slots.append(r[1])
            if r[2] >= 0:
                want_pairs.append([r[2], r[3]])
        assert st == 0 and done == 20 and slots.tolist() == want_slots
        assert pairs.tolist() == want_pairs
    _same_state(ref, dut, list(range(20)))


def test_batch_append_stops_at_exhaustion():
    dut = api.BlockAllocator(3, 4)
    assert dut.allocate(0, 4) == 0 and dut.allocate(1, 4) == 0 and dut.allocate(2, 3) == 0
    st, slots, pairs, done = dut.append_slots([2, 0, 1])
    assert st == api.PA_FAIL_NO_BLOCKS and done == 1 and slots[0] == 2 * 4 + 3
    assert dut.seq_len(0) == 4 and dut.seq_len(2) == 4


def test_traces_through_the_abi():
    tr = load("p1_allocator_traces.json")["fork_trace_35"]
    a = api.BlockAllocator(16, 16)
    order = [b for b in range(16) if b not in (10, 11, 12, 13)] + [13, 12, 11, 10]
    assert a.set_free_order(order) == 0
    assert a.allocate(7, 35) == 0 and a.block_table(7) == tr["prompt_blocks"]
    assert a.fork(7, 8) == 0
    assert a.append_slot(7) == (0, 13 * 16 + 3, 12, 13)
    assert a.append_slot(8) == (0, 12 * 16 + 3, -1, -1)
    assert [a.ref_count(b) for b in (10, 11, 12, 13)] == [2, 2, 1, 1]
    a.free(7)
    assert [a.ref_count(b) for b in (10, 11, 12, 13)] == [1, 1, 1, 0]
    ex = load("p1_allocator_traces.json")["exercise_2"]
    b = api.BlockAllocator(16, 8)
    assert b.allocate(1, 22) == 0 and b.fork(1, 2) == 0
    for _ in range(10):
        assert b.append_slot(1)[0] == 0
    assert b.block_table(1) == ex["table_a"] and b.block_table(2) == ex["table_b"]
    assert [b.ref_count(i) for i in range(5)] == [ex["refs_final"][str(i)] for i in range(5)]
    t3 = load("p1_allocator_traces.json")["verification_suite"]["test3"]
    c = api.BlockAllocator(4, 4)
    assert c.set_free_order(t3["free_list"]) == 0 and c.allocate(0, 6) == 0
    assert c.block_table(0) == t3["table"]
    assert c.slot_mapping(0, 0, 6).tolist() == [2 * 4 + i for i in range(4)] + [0, 1]
    tab, ctx = c.build_tables([0], 3)
    assert tab.tolist() == [[2, 0, -1]] and ctx.tolist() == [6]


def test_argument_errors():
    with pytest.raises(ValueError):
        api.BlockAllocator(0, 16)
    a = api.BlockAllocator(4, 4)
    assert a.allocate(1, 0) == api.PA_ERR_INVALID_ARG
    assert a.fork(5, 6) == api.PA_ERR_UNKNOWN_SEQ
    assert a.set_free_order([0, 1, 2]) == api.PA_ERR_INVALID_ARG
    assert a.set_free_order([0, 1, 2, 2]) == api.PA_ERR_INVALID_ARG
    assert a.allocate(1, 5) == 0
    assert a.set_free_order([0, 1, 2, 3]) == api.PA_ERR_INVALID_ARG
    with pytest.raises(api.PAError):
        a.slot_mapping(1, 3, 5)
    with pytest.raises(KeyError):
        a.block_table(99)
