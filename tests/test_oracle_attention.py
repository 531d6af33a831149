"""Pins for the attention oracle: page-printed worked examples, closed forms,
invariants and brute force.  CPU only."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from _golden import ev, ev_all, load


# --------------------------------------------------------------------------
# bf16 decoding (format definition: 1 sign, 8 exponent, 7 fraction bits)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xBF80, -1.0), (0x4000, 2.0), (0x3FC0, 1.5),
    (0x3E00, 0.125), (0x0000, 0.0), (0x0001, 2.0 ** -133),
    (0x0080, 2.0 ** -126), (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),
    (0x7F80, math.inf), (0xFF80, -math.inf),
])
def test_bf16_decode_known_patterns(bits, value):
    assert A.bf16_to_f64(np.array([bits], dtype=np.uint16))[0] == value


def test_bf16_decode_nan_and_negative_zero():
    x = A.bf16_to_f64(np.array([0x7FC0, 0x8000], dtype=np.uint16))
    assert math.isnan(x[0])
    assert x[1] == 0.0 and math.copysign(1.0, x[1]) == -1.0


def test_bf16_decode_matches_torch_on_all_finite_patterns():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = A.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


# --------------------------------------------------------------------------
# Worked example of [P2] sections 10 and 11
# --------------------------------------------------------------------------

@pytest.fixture(scope="module")
def worked():
    g = load("p2_worked_attention.json")
    return {
        "g": g,
        "q": np.array(ev_all(g["q"])),
        "K": np.array(ev_all(g["K"])),
        "V": np.array(ev_all(g["V"])),
        "scale": ev(g["scale"]),
    }


def test_worked_example_scores_weights_output(worked):
    g, q, K, V, scale = worked["g"], worked["q"], worked["K"], worked["V"], worked["scale"]
    scores = scale * (K @ q)
    np.testing.assert_allclose(scores, ev_all(g["scores"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(np.exp(scores), g["exp_scores"], rtol=1e-14)
    o = A.softmax_attention(q, K, V, scale)
    np.testing.assert_allclose(o, g["o"], rtol=1e-14)


def test_worked_example_through_scattered_pages(worked):
    """Same example with two tokens per page, stored in physical pages 9 and 2
    of a pool whose other pages hold NaN; the block table restores order."""
    g, q, K, V, scale = worked["g"], worked["q"], worked["K"], worked["V"], worked["scale"]
    B = g["paging"]["tokens_per_page"]
    pages = g["paging"]["physical_pages"]
    k_cache = np.full((10, 1, B, 2), np.nan)
    v_cache = np.full((10, 1, B, 2), np.nan)
    for lb, phys in enumerate(pages):
        k_cache[phys, 0] = K[lb * B:(lb + 1) * B]
        v_cache[phys, 0] = V[lb * B:(lb + 1) * B]
    out = A.paged_decode(q.reshape(1, 1, 2), k_cache, v_cache,
                         np.array([pages]), np.array([4]), scale, B)
    np.testing.assert_allclose(out[0, 0], g["o"], rtol=1e-14)


def test_worked_example_page_sums(worked):
    g, q, K, V, scale = worked["g"], worked["q"], worked["K"], worked["V"], worked["scale"]
    s = scale * (K @ q)
    N_a, Z_a = A.page_sums(s[:2], V[:2])
    N_b, Z_b = A.page_sums(s[2:], V[2:])
    np.testing.assert_allclose(N_a, g["page_A"]["N"], rtol=1e-14)
    np.testing.assert_allclose(Z_a, g["page_A"]["Z"], rtol=1e-14)
    np.testing.assert_allclose(N_b, g["page_B"]["N"], rtol=1e-14)
    np.testing.assert_allclose(Z_b, g["page_B"]["Z"], rtol=1e-14)
    np.testing.assert_allclose((N_a + N_b) / (Z_a + Z_b), g["o"], rtol=1e-14)


def test_worked_example_stable_merge(worked):
    g, q, K, V, scale = worked["g"], worked["q"], worked["K"], worked["V"], worked["scale"]
    s = scale * (K @ q)
    sa = A.block_summary(s[:2], V[:2])
    sb = A.block_summary(s[2:], V[2:])
    for got, want in ((sa, g["stable_A"]), (sb, g["stable_B"])):
        assert got[0] == pytest.approx(ev(want["m"]), abs=1e-15)
        assert got[1] == pytest.approx(want["z"], rel=1e-14)
        np.testing.assert_allclose(got[2], want["u"], rtol=1e-14)
    m, z, u = A.merge_summaries([sa, sb])
    assert m == pytest.approx(ev(g["merged"]["m"]), abs=1e-15)
    assert z == pytest.approx(g["merged"]["z"], rel=1e-14)
    np.testing.assert_allclose(u, g["merged"]["u"], rtol=1e-14)
    np.testing.assert_allclose(u / z, g["o"], rtol=1e-14)
    # partition_summaries with two positions per partition is the same split
    parts = A.partition_summaries(q, K, V, scale, 2)
    for got, want in zip(parts, (sa, sb)):
        assert got[0] == want[0] and got[1] == want[1]
        np.testing.assert_array_equal(got[2], want[2])


def test_merge_of_any_split_equals_single_pass():
    rng = np.random.default_rng(7)
    for trial in range(20):
        n = int(rng.integers(1, 300))
        d = int(rng.integers(1, 9))
        q = rng.normal(size=d)
        K = rng.normal(size=(n, d)) * 3
        V = rng.normal(size=(n, d))
        ref = A.softmax_attention(q, K, V, 0.7)
        p = int(rng.integers(1, n + 1))
        m, z, u = A.merge_summaries(A.partition_summaries(q, K, V, 0.7, p))
        np.testing.assert_allclose(u / z, ref, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------
# Closed forms and special cases
# --------------------------------------------------------------------------

def test_single_position_returns_its_value_row():
    rng = np.random.default_rng(1)
    q, K, V = rng.normal(size=4), rng.normal(size=(1, 4)), rng.normal(size=(1, 4))
    np.testing.assert_array_equal(A.softmax_attention(q, K, V, 0.5), V[0])


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    K = np.tile(rng.normal(size=(1, 8)), (37, 1))
    V = rng.normal(size=(37, 8))
    o = A.softmax_attention(rng.normal(size=8), K, V, 0.3)
    np.testing.assert_allclose(o, V.mean(axis=0), rtol=1e-13, atol=1e-15)


def test_two_positions_closed_form():
    """o = v0 + sigmoid(s1 - s0) * (v1 - v0) for two cached positions."""
    rng = np.random.default_rng(3)
    for _ in range(10):
        q, K, V = rng.normal(size=6), rng.normal(size=(2, 6)), rng.normal(size=(2, 6))
        s = 0.4 * (K @ q)
        w1 = 1.0 / (1.0 + math.exp(-(s[1] - s[0])))
        np.testing.assert_allclose(A.softmax_attention(q, K, V, 0.4),
                                   V[0] + w1 * (V[1] - V[0]), rtol=1e-13, atol=1e-15)


def test_large_scores_do_not_overflow_and_shift_invariance():
    rng = np.random.default_rng(4)
    q, K, V = rng.normal(size=4), rng.normal(size=(50, 4)), rng.normal(size=(50, 4))
    base = A.softmax_attention(q, K, V, 1.0)
    # adding c * q / |q|^2 to every key adds the constant c to every score
    c = 5000.0
    shifted = A.softmax_attention(q, K + c * q / (q @ q), V, 1.0)
    assert np.all(np.isfinite(shifted))
    np.testing.assert_allclose(shifted, base, rtol=1e-9, atol=1e-12)


def test_dominant_score_gives_its_value_row():
    """One score 1,000 above all others ([P2] section 11: subtracting the
    maximum keeps every exponential at most 1): each other weight is
    exp(-1000), which is 0 in float64, so the output is exactly that value
    row.  Exponentials of the raw or minimum-shifted scores overflow."""
    rng = np.random.default_rng(5)
    K = np.zeros((6, 3))
    K[4, 0] = 1000.0
    V = rng.normal(size=(6, 3))
    o = A.softmax_attention(np.array([1.0, 0.0, 0.0]), K, V, 1.0)
    assert np.array_equal(o, V[4])


def test_zero_context_gives_zero_row():
    q = np.ones((1, 2, 4))
    kc = np.ones((2, 1, 4, 4))
    out = A.paged_decode(q, kc, kc, np.array([[0, 1]]), np.array([0]), 1.0, 4)
    assert np.array_equal(out, np.zeros_like(out))


# --------------------------------------------------------------------------
# Paging invariants ([P1] section 20 test 3; [P2] sections 10 and 12)
# --------------------------------------------------------------------------

def _random_paged_problem(rng, S, Hq, Hkv, D, B, lens, extra_blocks=5, junk=np.nan):
    nblk = [-(-l // B) for l in lens]
    NB = sum(nblk) + extra_blocks
    perm = rng.permutation(NB)
    MB = max(nblk)
    tables = np.full((S, MB), -1, dtype=np.int64)
    k_cache = np.full((NB, Hkv, B, D), junk)
    v_cache = np.full((NB, Hkv, B, D), junk)
    K_dense = np.zeros((S, Hkv, max(lens), D))
    V_dense = np.zeros((S, Hkv, max(lens), D))
    pos = 0
    for s, L in enumerate(lens):
        K_dense[s, :, :L] = rng.normal(size=(Hkv, L, D))
        V_dense[s, :, :L] = rng.normal(size=(Hkv, L, D))
        for lb in range(nblk[s]):
            phys = int(perm[pos])
            pos += 1
            tables[s, lb] = phys
            n = min(B, L - lb * B)
            k_cache[phys, :, :n] = K_dense[s, :, lb * B: lb * B + n]
            v_cache[phys, :, :n] = V_dense[s, :, lb * B: lb * B + n]
    q = rng.normal(size=(S, Hq, D))
    return q, k_cache, v_cache, tables, np.array(lens), K_dense, V_dense


@pytest.mark.parametrize("B", [1, 4, 16])
def test_paged_equals_dense_with_junk_tails(B):
    rng = np.random.default_rng(10 + B)
    lens = [1, 5, 16, 17, 40]
    q, kc, vc, tab, ctx, Kd, Vd = _random_paged_problem(rng, 5, 6, 3, 8, B, lens)
    paged = A.paged_decode(q, kc, vc, tab, ctx, 0.35, B)
    dense = A.dense_decode(q, Kd, Vd, ctx, 0.35)
    assert np.all(np.isfinite(paged))
    np.testing.assert_allclose(paged, dense, rtol=1e-13, atol=1e-15)


def test_output_invariant_under_physical_placement():
    rng = np.random.default_rng(20)
    lens = [9, 33, 64]
    q, kc, vc, tab, ctx, _, _ = _random_paged_problem(rng, 3, 4, 2, 4, 8, lens)
    ref = A.paged_decode(q, kc, vc, tab, ctx, 0.5, 8)
    NB = kc.shape[0]
    for _ in range(5):
        perm = rng.permutation(NB)          # block p moves to perm[p]
        kc2 = np.empty_like(kc)
        vc2 = np.empty_like(vc)
        kc2[perm] = kc
        vc2[perm] = vc
        tab2 = np.where(tab >= 0, perm[np.maximum(tab, 0)], -1)
        np.testing.assert_array_equal(A.paged_decode(q, kc2, vc2, tab2, ctx, 0.5, 8), ref)


def test_p1_verification_test3_paged_vs_dense():
    """[P1] section 20, test 3: free list forced to [1, 3, 0, 2] gives table
    [2, 0]; junk in the two masked tail slots; paged equals dense."""
    from oracle.allocator import RefAllocator
    t3 = load("p1_allocator_traces.json")["verification_suite"]["test3"]
    alloc = RefAllocator(t3["num_blocks"], t3["block_size"])
    alloc.set_free_order(t3["free_list"])
    kv = t3["kv"]
    assert alloc.allocate("eval_seq", len(kv)) == 0
    assert alloc.block_tables["eval_seq"] == t3["table"]
    B = t3["block_size"]
    kc = np.zeros((t3["num_blocks"], 1, B, 1))
    vc = np.zeros((t3["num_blocks"], 1, B, 1))
    for i, (k, v) in enumerate(kv):
        blk, off = divmod(alloc.slot_of("eval_seq", i), B)
        kc[blk, 0, off, 0] = k
        vc[blk, 0, off, 0] = v
    tail = alloc.block_tables["eval_seq"][1]
    for off, (k, v) in t3["junk"].items():
        kc[tail, 0, int(off), 0] = k
        vc[tail, 0, int(off), 0] = v
    q = np.array([[[t3["q"]]]])
    paged = A.paged_decode(q, kc, vc, np.array([alloc.block_tables["eval_seq"]]),
                           np.array([len(kv)]), t3["scale"], B)[0, 0, 0]
    dense_scores = [t3["q"] * k * t3["scale"] for k, _ in kv]
    mx = max(dense_scores)
    e = [math.exp(x - mx) for x in dense_scores]
    dense = sum(w / sum(e) * v for w, (_, v) in zip(e, kv))
    assert math.isclose(paged, dense, rel_tol=t3["rel_tol"])


def test_gqa_contiguous_group_mapping():
    """Each KV head's values are a distinct constant; query head g must read
    KV head g // G (reading: contiguous groups), so its output is exactly
    that constant."""
    rng = np.random.default_rng(30)
    for Hq, Hkv in ((8, 2), (8, 1), (4, 4), (6, 3)):
        G = Hq // Hkv
        B, D, L = 4, 3, 10
        kc = rng.normal(size=(5, Hkv, B, D))
        vc = np.zeros((5, Hkv, B, D))
        for h in range(Hkv):
            vc[:, h] = 10.0 + h
        q = rng.normal(size=(1, Hq, D))
        out = A.paged_decode(q, kc, vc, np.array([[3, 0, 4]]), np.array([L]), 0.5, B)
        for g in range(Hq):
            np.testing.assert_allclose(out[0, g], 10.0 + g // G, rtol=1e-14)


def test_gqa_equals_replicated_mha():
    """GQA over Hkv heads equals MHA over Hq heads with each KV head repeated
    G times (contiguously)."""
    rng = np.random.default_rng(31)
    Hq, Hkv, B, D = 8, 2, 4, 5
    q, kc, vc, tab, ctx, _, _ = _random_paged_problem(rng, 2, Hq, Hkv, D, B, [7, 13])
    gqa = A.paged_decode(q, kc, vc, tab, ctx, 0.3, B)
    mha = A.paged_decode(q, np.repeat(kc, Hq // Hkv, axis=1), np.repeat(vc, Hq // Hkv, axis=1),
                         tab, ctx, 0.3, B)
    np.testing.assert_array_equal(gqa, mha)


def _brute_force(q, kc, vc, tables, ctx, scale, B):
    """Pure-Python loops, no NumPy arithmetic."""
    S, Hq, D = q.shape
    Hkv = kc.shape[1]
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(S)]
    for s in range(S):
        for g in range(Hq):
            h = g * Hkv // Hq
            sc = []
            for i in range(int(ctx[s])):
                blk = int(tables[s][i // B])
                sc.append(scale * sum(float(q[s, g, d]) * float(kc[blk, h, i % B, d]) for d in range(D)))
            mx = max(sc)
            w = [math.exp(x - mx) for x in sc]
            tot = sum(w)
            for d in range(D):
                out[s][g][d] = sum(w[i] * float(vc[int(tables[s][i // B]), h, i % B, d])
                                   for i in range(len(w))) / tot
    return np.array(out)


def test_brute_force_tiny():
    rng = np.random.default_rng(40)
    q, kc, vc, tab, ctx, _, _ = _random_paged_problem(rng, 3, 4, 2, 3, 2, [1, 4, 7])
    np.testing.assert_allclose(A.paged_decode(q, kc, vc, tab, ctx, 0.6, 2),
                               _brute_force(q, kc, vc, tab, ctx, 0.6, 2), rtol=1e-12, atol=1e-14)


def test_exhaustive_placements_of_three_blocks():
    import itertools
    rng = np.random.default_rng(41)
    B, D, L = 2, 3, 5                         # 3 logical blocks, last one partial
    K = rng.normal(size=(L, D))
    V = rng.normal(size=(L, D))
    q = rng.normal(size=(1, 1, D))
    ref = A.softmax_attention(q[0, 0], K, V, 0.8)
    for table in itertools.permutations(range(4), 3):
        kc = np.full((4, 1, B, D), np.nan)
        vc = np.full((4, 1, B, D), np.nan)
        for i in range(L):
            kc[table[i // B], 0, i % B] = K[i]
            vc[table[i // B], 0, i % B] = V[i]
        out = A.paged_decode(q, kc, vc, np.array([table]), np.array([L]), 0.8, B)
        np.testing.assert_array_equal(out[0, 0], ref)
