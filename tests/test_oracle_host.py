"""Pins for the sizing, allocator and cache-op oracles: the pages' worked
traces, exercises and verification suite.  CPU only."""
import numpy as np
import pytest

from oracle import allocator as AL
from oracle import attention as A
from oracle import cache_ops as C
from oracle import sizing as Z
from _golden import load


# --------------------------------------------------------------------------
# Sizing ([P1] sections 1, 8, 10, 11, 23; [P2] section 4; [P3] sizing)
# --------------------------------------------------------------------------

def test_bytes_per_token_and_sequence():
    g = load("p1_sizing.json")
    m = g["model_8b"]
    bpt = Z.kv_bytes_per_token(m["n_layers"], m["n_kv_heads"], m["d_head"], m["elem_bytes"])
    assert bpt == g["bytes_per_token"] == g["kib_per_token"] * 1024
    seq = Z.kv_bytes(m["n_layers"], 4096, m["n_kv_heads"], m["d_head"], m["elem_bytes"])
    assert seq == g["seq_4096_bytes"] == g["seq_4096_mib"] * 1024 * 1024


def test_block_table_footprint():
    t = load("p1_sizing.json")["table"]
    assert Z.blocks_needed(t["tokens"], t["block_size"]) == t["blocks"]
    assert Z.block_table_bytes(t["tokens"], t["block_size"]) == t["bytes"]
    payload = Z.kv_bytes(32, t["tokens"], 8, 128, 2)
    assert payload // t["bytes"] == t["ratio_denominator"] and payload % t["bytes"] == 0


@pytest.mark.parametrize("B", [8, 16, 32])
def test_capacity_decision(B):
    c = load("p1_sizing.json")["capacity"]
    want = c["B%d" % B]
    assert [Z.blocks_needed(s, B) for s in c["lengths"]] == want["per_request_blocks"]
    assert [Z.tail_waste_slots(s, B) for s in c["lengths"]] == want["per_request_waste"]
    plan = Z.capacity_plan(c["lengths"], B, c["pool_slots"])
    assert plan["slots"] == want["slots"] and plan["waste"] == want["waste"]
    assert plan["fits"] == want["fits"] and plan["deficit_slots"] == want["deficit_slots"]
    assert round(100 * plan["waste_frac"], 2) == want["waste_pct"]
    assert plan["slots"] * c["kib_per_slot"] == want["mib"] * 1024
    assert sum(c["lengths"]) == c["useful_tokens"]


def test_index_overhead_ratio():
    c = load("p1_sizing.json")["capacity"]
    e8 = sum(Z.blocks_needed(s, 8) for s in c["lengths"])
    e16 = sum(Z.blocks_needed(s, 16) for s in c["lengths"])
    assert (e8, e16) == (c["table_entries"]["B8"], c["table_entries"]["B16"])
    assert round(e8 / e16, 2) == c["index_overhead_ratio"]


@pytest.mark.parametrize("B", [4, 8])
def test_exercise_1(B):
    e = load("p1_sizing.json")["exercise_1"]
    want = e["B%d" % B]
    assert [Z.blocks_needed(s, B) for s in e["lengths"]] == want["per_request_blocks"]
    assert [Z.tail_waste_slots(s, B) for s in e["lengths"]] == want["per_request_waste"]
    plan = Z.capacity_plan(e["lengths"], B, e["pool_slots"])
    assert (plan["blocks"], plan["slots"], plan["waste"], plan["fits"]) == \
        (want["blocks"], want["slots"], want["waste"], want["fits"])
    assert plan["slots"] * e["kib_per_slot"] == want["mib"] * 1024
    if "waste_frac" in want:
        assert plan["waste_frac"] == want["waste_frac"]


def test_kv_cache_gb_example():
    x = load("p1_sizing.json")["kv_cache_gb_example"]
    # the page's helper counts all attention heads (32, MHA) per token
    gb = Z.kv_bytes(x["n_layers"], x["seq_len"] * x["batch"], x["n_heads"], x["head_dim"],
                    x["bytes_per_elem"]) / 1e9
    assert round(gb) == x["approx_gb"]


def test_tail_waste_bound():
    for B in (1, 4, 8, 16, 32, 64):
        for S in range(1, 200):
            w = Z.tail_waste_slots(S, B)
            assert 0 <= w <= B - 1
            assert (S + w) % B == 0


# --------------------------------------------------------------------------
# Address translation examples ([P1] sections 5, 7; [P2] sections 2, 5; [P3])
# --------------------------------------------------------------------------

def test_translation_examples():
    t = load("translation_examples.json")
    e = t["p1_section7"]
    lb = e["i"] // e["block_size"]
    assert A.translate(e["i"], e["block_size"], list(range(10))) == (lb, e["offset"])
    assert lb == e["logical_block"]
    e = t["p1_section5"]
    for i, phys, off in e["cases"]:
        assert A.translate(i, e["block_size"], e["table"]) == (phys, off)
    e = t["p2_section5"]
    assert A.translate(e["token"], e["block_size"], e["table"]) == (e["physical_block"], e["slot_in_block"])
    for lo, hi, phys in e["logical_ranges"]:
        for i in range(lo, hi + 1):
            assert A.translate(i, e["block_size"], e["table"])[0] == phys
    assert Z.tail_waste_slots(e["n_tokens"], e["block_size"]) == e["unused_tail_slots"]
    e = t["p3_block_table"]
    for i in range(4 * e["block_size"]):
        assert A.translate(i, e["block_size"], e["table"]) == (e["table"][i // 16], i % 16)


def test_os_analogue_slot_arithmetic():
    """frame * page_size + offset ([P2] section 2) is the slot formula used by
    reshape_and_cache: slot 37,768 with 4,096-slot blocks is block 9, offset 904."""
    e = load("translation_examples.json")["p2_section2_os"]
    phys, off = A.translate(e["virtual_address"], e["page_size"], [0, e["frame"]])
    assert (phys, off) == (e["frame"], e["offset"])
    assert phys * e["page_size"] + off == e["physical_address"]
    k = np.zeros((10, 1, e["page_size"], 1), dtype=np.uint16)
    row = np.array([[7]], dtype=np.uint16)
    k2, _ = C.reshape_and_cache(k.copy(), k.copy(), row[None], row[None], [e["physical_address"]], e["page_size"])
    assert k2[e["frame"], 0, e["offset"], 0] == 7 and int(k2.sum()) == 7


# --------------------------------------------------------------------------
# Allocator traces
# --------------------------------------------------------------------------

def _refs(alloc, ids):
    return {str(b): alloc.ref_counts[b] for b in ids}


def test_fork_trace_35_tokens():
    tr = load("p1_allocator_traces.json")["fork_trace_35"]
    B = tr["block_size"]
    alloc = AL.RefAllocator(16, B)
    # make the pool hand out 10, 11, 12, 13 next (blocks leave from the end)
    order = [b for b in range(16) if b not in (10, 11, 12, 13)] + [13, 12, 11, 10]
    assert alloc.set_free_order(order) == AL.OK
    assert alloc.allocate("A", tr["prompt_tokens"]) == AL.OK
    assert alloc.block_tables["A"] == tr["prompt_blocks"]
    assert alloc.fork("A", "B") == AL.OK
    assert _refs(alloc, tr["prompt_blocks"]) == tr["refs_after_fork"]
    st, slot, src, dst = alloc.append_slot("A")
    a = tr["a_append"]
    assert (st, src, dst) == (AL.OK, a["cow_src"], a["cow_dst"])
    assert slot == a["cow_dst"] * B + a["offset"]
    assert a["position"] % B == a["copied_positions"] == a["offset"]
    st, slot, src, dst = alloc.append_slot("B")
    b = tr["b_append"]
    assert (st, src, dst) == (AL.OK, -1, -1) and slot == b["block"] * B + b["offset"]
    assert _refs(alloc, [10, 11, 12, 13]) == tr["refs_after_appends"]
    assert alloc.block_tables["A"] == tr["table_a"] and alloc.block_tables["B"] == tr["table_b"]
    in_use = 16 - alloc.num_free()
    assert in_use == tr["blocks_in_use"] and in_use * B == tr["slots_in_use"]
    shared = [x for x in alloc.block_tables["A"] if x in alloc.block_tables["B"]]
    assert len(shared) * B == tr["shared_prefix_positions"]
    useful = len(shared) * B + sum(alloc.seq_lengths[s] - len(shared) * B for s in "AB")
    assert useful == tr["useful_tokens"] and in_use * B - useful == tr["tail_waste"]
    assert sum(Z.blocks_needed(alloc.seq_lengths[s], B) for s in "AB") == tr["blocks_without_sharing"]
    alloc.free("A")
    assert _refs(alloc, [10, 11, 12, 13]) == tr["refs_after_free_a"]
    assert alloc.free_blocks[-1] == 13


def test_exercise_2_trace():
    ex = load("p1_allocator_traces.json")["exercise_2"]
    B = ex["block_size"]
    alloc = AL.RefAllocator(16, B)
    assert alloc.allocate("A", ex["seq_a_tokens"]) == AL.OK
    assert alloc.block_tables["A"] == ex["initial_blocks"]
    assert alloc.fork("A", "B") == AL.OK
    assert _refs(alloc, ex["initial_blocks"]) == ex["refs_after_fork"]
    events = {e["token"]: e for e in ex["events"]}
    for _ in range(ex["appends_a"]):
        pos = alloc.seq_lengths["A"]
        st, slot, src, dst = alloc.append_slot("A")
        assert st == AL.OK
        e = events.get(pos)
        if e and "cow_src" in e:
            assert (src, dst) == (e["cow_src"], e["cow_dst"]) and slot == dst * B + e["offset"]
        elif e and "new_block" in e:
            assert src == -1 and slot == e["new_block"] * B + e["offset"]
        elif e:
            assert src == -1 and slot == e["block"] * B + e["offset"]
        else:
            assert src == -1
    assert alloc.block_tables["A"] == ex["table_a"] and alloc.block_tables["B"] == ex["table_b"]
    assert (alloc.seq_lengths["A"], alloc.seq_lengths["B"]) == (ex["len_a"], ex["len_b"])
    assert _refs(alloc, range(5)) == ex["refs_final"]
    in_use = 16 - alloc.num_free()
    assert in_use == ex["blocks_in_use"] and in_use * B == ex["slots_in_use"]
    shared = set(alloc.block_tables["A"]) & set(alloc.block_tables["B"])
    payload = len(shared) * B + (ex["len_b"] - len(shared) * B) + (ex["len_a"] - len(shared) * B)
    assert payload == ex["payload_positions"]
    assert in_use * B - payload == ex["tail_waste"]


def test_verification_suite_1_4_5():
    vs = load("p1_allocator_traces.json")["verification_suite"]
    t1 = vs["test1"]
    alloc = AL.RefAllocator(t1["num_blocks"], t1["block_size"])
    for i, L in enumerate(t1["lengths"]):
        assert alloc.allocate(i, L) == AL.OK
    slots = sum(len(alloc.block_tables[i]) for i in range(4)) * t1["block_size"]
    assert slots == t1["slots"] and slots - sum(t1["lengths"]) == t1["waste"]
    assert alloc.num_free() == 0
    t4 = vs["test4"]
    tiny = AL.RefAllocator(t4["num_blocks"], t4["block_size"])
    assert tiny.allocate("seq", t4["prompt_tokens"]) == AL.OK
    before = (list(tiny.free_blocks), list(tiny.ref_counts), list(tiny.block_tables["seq"]))
    assert tiny.append_slot("seq")[0] == AL.FAIL_NO_BLOCKS
    assert tiny.seq_lengths["seq"] == t4["len_after"]
    assert len(tiny.block_tables["seq"]) == t4["blocks_after"]
    assert (list(tiny.free_blocks), list(tiny.ref_counts), list(tiny.block_tables["seq"])) == before


def test_verification_suite_2_and_5_with_payload():
    """[P1] section 20 tests 2 and 5 with the payload moved by the cache ops."""
    vs = load("p1_allocator_traces.json")["verification_suite"]
    t2 = vs["test2"]
    B = t2["block_size"]
    alloc = AL.RefAllocator(t2["num_blocks"], B)
    kc = np.zeros((t2["num_blocks"], 1, B, 1))
    vc = np.zeros((t2["num_blocks"], 1, B, 1))
    prompt = [(float(i), float(10 * i)) for i in range(t2["prompt_tokens"])]
    assert alloc.allocate("A", len(prompt)) == AL.OK
    slots = [alloc.slot_of("A", i) for i in range(len(prompt))]
    kc, vc = C.reshape_and_cache(kc, vc, np.array([[[k]] for k, _ in prompt]),
                                 np.array([[[v]] for _, v in prompt]), slots, B)
    assert alloc.fork("A", "B") == AL.OK
    for seq, (k, v) in (("A", t2["a_append"]), ("B", t2["b_append"])):
        st, slot, src, dst = alloc.append_slot(seq)
        assert st == AL.OK
        if src >= 0:
            (kc,), (vc,) = C.copy_blocks([kc], [vc], [[src, dst]])
        kc, vc = C.reshape_and_cache(kc, vc, np.array([[[k]]]), np.array([[[v]]]), [slot], B)
    ti = t2["tail_index"]
    tail_a, tail_b = alloc.block_tables["A"][ti], alloc.block_tables["B"][ti]
    assert tail_a != tail_b
    off = t2["tail_offset_of_append"]
    assert (kc[tail_a, 0, off, 0], vc[tail_a, 0, off, 0]) == tuple(t2["a_append"])
    assert (kc[tail_b, 0, off, 0], vc[tail_b, 0, off, 0]) == tuple(t2["b_append"])
    p = t2["a_tail_slot0_is_prompt_position"]
    assert (kc[tail_a, 0, 0, 0], vc[tail_a, 0, 0, 0]) == prompt[p]
    # test 5: releasing both returns the whole pool
    alloc.free("A")
    alloc.free("B")
    t5 = vs["test5"]
    assert alloc.num_free() == t5["free_after_release"] and all(r == 0 for r in alloc.ref_counts)


def test_release_order_is_table_order():
    """[P1] section 20's teaching allocator: the free list starts as the
    block ids in reverse, allocation takes from its end, and freeing a
    sequence appends its blocks in table order.  Derived by hand for a pool
    of 8 blocks of 4 slots: A (10 tokens) takes 0, 1, 2; after A is freed
    the list ends ..., 3, 0, 1, 2, so B (4 tokens) takes 2 and C (8 tokens)
    takes 1, then 0."""
    al = AL.RefAllocator(8, 4)
    assert al.allocate("A", 10) == AL.OK
    assert al.block_tables["A"] == [0, 1, 2]
    assert al.free("A") == AL.OK
    assert al.free_blocks == [7, 6, 5, 4, 3, 0, 1, 2]
    assert al.allocate("B", 4) == AL.OK and al.block_tables["B"] == [2]
    assert al.allocate("C", 8) == AL.OK and al.block_tables["C"] == [1, 0]


def test_allocator_argument_errors_and_transactional_failures():
    with pytest.raises(ValueError):
        AL.RefAllocator(0, 4)
    with pytest.raises(ValueError):
        AL.RefAllocator(4, 0)
    a = AL.RefAllocator(3, 4)
    assert a.allocate("x", 0) == AL.ERR_INVALID_ARG
    assert a.allocate("x", 13) == AL.FAIL_NO_BLOCKS and a.num_free() == 3 and not a.block_tables
    assert a.allocate("x", 5) == AL.OK
    assert a.allocate("x", 1) == AL.ERR_DUPLICATE_SEQ
    assert a.fork("nope", "y") == AL.ERR_UNKNOWN_SEQ
    assert a.fork("x", "x") == AL.ERR_DUPLICATE_SEQ
    assert a.append_slot("nope")[0] == AL.ERR_UNKNOWN_SEQ
    assert a.free("nope") == AL.OK
    assert a.set_free_order([0, 1, 2]) == AL.ERR_INVALID_ARG      # blocks in use
    # shared tail with an empty pool: the CoW append fails and nothing changes
    assert a.fork("x", "y") == AL.OK
    assert a.allocate("z", 4) == AL.OK and a.num_free() == 0
    snap = (list(a.free_blocks), list(a.ref_counts), {k: list(v) for k, v in a.block_tables.items()},
            dict(a.seq_lengths))
    assert a.append_slot("x")[0] == AL.FAIL_NO_BLOCKS
    assert snap == (list(a.free_blocks), list(a.ref_counts),
                    {k: list(v) for k, v in a.block_tables.items()}, dict(a.seq_lengths))


def test_refcount_conservation_under_random_churn():
    """Every block's count equals the number of tables holding it; free blocks
    are exactly those with count 0; no block is both free and referenced."""
    rng = np.random.default_rng(5)
    a = AL.RefAllocator(64, 4)
    live = []
    nxt = 0
    for _ in range(3000):
        op = rng.integers(0, 4)
        if op == 0 or not live:
            if a.allocate(nxt, int(rng.integers(1, 20))) == AL.OK:
                live.append(nxt)
            nxt += 1
        elif op == 1:
            if a.fork(live[int(rng.integers(len(live)))], nxt) == AL.OK:
                live.append(nxt)
            nxt += 1
        elif op == 2:
            a.append_slot(live[int(rng.integers(len(live)))])
        else:
            a.free(live.pop(int(rng.integers(len(live)))))
        counts = [0] * 64
        for t in a.block_tables.values():
            for b in t:
                counts[b] += 1
        assert counts == a.ref_counts
        assert sorted(a.free_blocks) == [b for b in range(64) if counts[b] == 0]
        for s, t in a.block_tables.items():
            assert len(t) == Z.blocks_needed(a.seq_lengths[s], 4)


# --------------------------------------------------------------------------
# Cache ops
# --------------------------------------------------------------------------

def test_reshape_and_cache_writes_only_its_slots():
    rng = np.random.default_rng(6)
    NB, H, B, D = 6, 2, 4, 3
    k = rng.integers(0, 1 << 16, size=(NB, H, B, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(NB, H, B, D), dtype=np.uint16)
    kn = rng.integers(0, 1 << 16, size=(4, H, D), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, size=(4, H, D), dtype=np.uint16)
    # a negative slot is skipped (reading O7); written, -1 would land on
    # block 5, offset 3, which no other token writes
    slots = [5, -1, 22, 0]
    k2, v2 = C.reshape_and_cache(k.copy(), v.copy(), kn, vn, slots, B)
    touched = np.zeros((NB, B), dtype=bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(s, B)
        touched[blk, off] = True
        assert np.array_equal(k2[blk, :, off], kn[t]) and np.array_equal(v2[blk, :, off], vn[t])
    mask = ~touched[:, None, :, None].repeat(H, 1).repeat(D, 3)
    assert np.array_equal(k2[mask], k[mask]) and np.array_equal(v2[mask], v[mask])


def test_swap_blocks_moves_whole_blocks():
    """[P1] section 19, item 4: a swapped block moves whole, K and V, from
    one pool to the other; each pair names (source block, destination
    block), the other blocks are untouched, and swapping back into other
    blocks restores the payload."""
    rng = np.random.default_rng(9)
    dev_k = rng.integers(0, 1 << 16, size=(6, 2, 4, 3), dtype=np.uint16)
    dev_v = rng.integers(0, 1 << 16, size=(6, 2, 4, 3), dtype=np.uint16)
    host_k = np.zeros((4, 2, 4, 3), dtype=np.uint16)
    host_v = np.zeros((4, 2, 4, 3), dtype=np.uint16)
    C.swap_blocks(host_k, host_v, dev_k, dev_v, [(5, 0), (2, 3)])
    assert np.array_equal(host_k[0], dev_k[5]) and np.array_equal(host_v[0], dev_v[5])
    assert np.array_equal(host_k[3], dev_k[2]) and np.array_equal(host_v[3], dev_v[2])
    assert not host_k[1:3].any() and not host_v[1:3].any()
    back_k = np.zeros_like(dev_k)
    back_v = np.zeros_like(dev_v)
    C.swap_blocks(back_k, back_v, host_k, host_v, [(0, 1), (3, 4)])
    assert np.array_equal(back_k[1], dev_k[5]) and np.array_equal(back_v[4], dev_v[2])
    assert not back_k[[0, 2, 3, 5]].any() and not back_v[[0, 2, 3, 5]].any()


def test_copy_blocks_cow_trace_payload():
    """[P1] section 16: after the copy, block 13 holds positions 32..34 of the
    shared tail; the other blocks are untouched, in every layer."""
    rng = np.random.default_rng(8)
    layers = [rng.integers(0, 1 << 16, size=(16, 2, 16, 4), dtype=np.uint16) for _ in range(3)]
    vlayers = [rng.integers(0, 1 << 16, size=(16, 2, 16, 4), dtype=np.uint16) for _ in range(3)]
    k2, v2 = C.copy_blocks([x.copy() for x in layers], [x.copy() for x in vlayers], [[12, 13]])
    for l in range(3):
        assert np.array_equal(k2[l][13, :, :3], layers[l][12, :, :3])
        assert np.array_equal(k2[l][13], layers[l][12]) and np.array_equal(v2[l][13], vlayers[l][12])
        others = [b for b in range(16) if b != 13]
        assert np.array_equal(k2[l][others], layers[l][others])
