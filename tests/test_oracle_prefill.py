"""Pins for the prefill oracle (causal attention of many new positions).

It is tied to the already pinned decode oracle and to the definition by
reductions and invariants: one new token is a decode step; the first token of
a prompt sees only itself; a query never depends on later positions; a
prompt split into chunks gives the same rows as one pass; pure-Python brute
force on tiny cases; GQA equals replicated MHA.  CPU only."""
import math

import numpy as np
import pytest

from oracle import attention as A
from test_oracle_attention import _random_paged_problem


def _prefill_problem(rng, Hq, Hkv, D, B, lens, news, junk=np.nan):
    """A paged cache holding `lens` positions per sequence and queries for
    the last `news[s]` positions of each."""
    S = len(lens)
    _, kc, vc, tab, ctx, Kd, Vd = _random_paged_problem(rng, S, Hq, Hkv, D, B, lens, junk=junk)
    qs = np.concatenate([[0], np.cumsum(news)]).astype(np.int64)
    q = rng.normal(size=(int(qs[-1]), Hq, D))
    return q, kc, vc, tab, qs, ctx, Kd, Vd


def _brute_force_prefill(q, kc, vc, tables, qs, ctx, scale, B):
    """Pure-Python loops over rows, heads and visible positions."""
    T, Hq, D = q.shape
    Hkv = kc.shape[1]
    out = np.zeros((T, Hq, D))
    for s in range(len(ctx)):
        n = int(qs[s + 1] - qs[s])
        for i in range(n):
            p = int(ctx[s]) - n + i
            for g in range(Hq):
                h = g * Hkv // Hq
                sc = []
                for j in range(p + 1):
                    blk = int(tables[s][j // B])
                    sc.append(scale * sum(float(q[qs[s] + i, g, d]) * float(kc[blk, h, j % B, d]) for d in range(D)))
                mx = max(sc)
                w = [math.exp(x - mx) for x in sc]
                tot = sum(w)
                for d in range(D):
                    out[qs[s] + i, g, d] = sum(w[j] * float(vc[int(tables[s][j // B]), h, j % B, d])
                                               for j in range(p + 1)) / tot
    return out


def test_brute_force_tiny_prefill():
    rng = np.random.default_rng(50)
    q, kc, vc, tab, qs, ctx, _, _ = _prefill_problem(rng, 4, 2, 3, 2, [1, 5, 7], [1, 5, 3])
    np.testing.assert_allclose(A.paged_prefill(q, kc, vc, tab, qs, ctx, 0.7, 2),
                               _brute_force_prefill(q, kc, vc, tab, qs, ctx, 0.7, 2), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("B", [1, 4, 16])
def test_one_new_token_is_a_decode_step(B):
    rng = np.random.default_rng(51 + B)
    lens = [1, 5, 16, 17, 40]
    q, kc, vc, tab, qs, ctx, _, _ = _prefill_problem(rng, 6, 3, 8, B, lens, [1] * 5)
    np.testing.assert_array_equal(A.paged_prefill(q, kc, vc, tab, qs, ctx, 0.35, B),
                                  A.paged_decode(q, kc, vc, tab, ctx, 0.35, B))


def test_first_prompt_token_sees_only_itself():
    rng = np.random.default_rng(52)
    q, kc, vc, tab, qs, ctx, _, Vd = _prefill_problem(rng, 4, 4, 8, 4, [9, 3], [9, 3])
    out = A.paged_prefill(q, kc, vc, tab, qs, ctx, 0.5, 4)
    for s in range(2):
        for g in range(4):
            np.testing.assert_array_equal(out[qs[s], g], Vd[s, g, 0])


def test_causal_later_positions_do_not_matter():
    rng = np.random.default_rng(53)
    B, L = 4, 13
    q, kc, vc, tab, qs, ctx, _, _ = _prefill_problem(rng, 2, 1, 5, B, [L], [L])
    full = A.paged_prefill(q, kc, vc, tab, qs, ctx, 0.5, B)
    for p in range(L - 1):
        k2, v2 = kc.copy(), vc.copy()
        for j in range(p + 1, L):            # poison every later position
            blk = int(tab[0, j // B])
            k2[blk, :, j % B] = np.nan
            v2[blk, :, j % B] = np.nan
        got = A.paged_prefill(q, k2, v2, tab, qs, ctx, 0.5, B)
        np.testing.assert_array_equal(got[:p + 1], full[:p + 1])
        assert np.isnan(got[p + 1:]).all()


def test_last_row_equals_attention_over_the_whole_context():
    rng = np.random.default_rng(54)
    q, kc, vc, tab, qs, ctx, Kd, Vd = _prefill_problem(rng, 4, 2, 6, 4, [23, 8], [7, 8])
    out = A.paged_prefill(q, kc, vc, tab, qs, ctx, 0.4, 4)
    last = q[[qs[1] - 1, qs[2] - 1]]
    np.testing.assert_allclose(out[[qs[1] - 1, qs[2] - 1]], A.dense_decode(last, Kd, Vd, ctx, 0.4),
                               rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("cut", [1, 5, 11])
def test_chunked_prefill_equals_one_pass(cut):
    rng = np.random.default_rng(55)
    B, L = 4, 17
    q, kc, vc, tab, qs, ctx, _, _ = _prefill_problem(rng, 4, 2, 6, B, [L], [L])
    whole = A.paged_prefill(q, kc, vc, tab, qs, ctx, 0.45, B)
    # the same prompt in two chunks: [0, cut) with context cut, then [cut, L)
    first = A.paged_prefill(q[:cut], kc, vc, tab, np.array([0, cut]), np.array([cut]), 0.45, B)
    second = A.paged_prefill(q[cut:], kc, vc, tab, np.array([0, L - cut]), np.array([L]), 0.45, B)
    np.testing.assert_array_equal(np.concatenate([first, second]), whole)


def test_gqa_prefill_equals_replicated_mha():
    rng = np.random.default_rng(56)
    B = 4
    q, kc, vc, tab, qs, ctx, _, _ = _prefill_problem(rng, 6, 2, 5, B, [9, 6], [4, 6])
    gqa = A.paged_prefill(q, kc, vc, tab, qs, ctx, 0.5, B)
    rep = np.repeat(kc, 3, axis=1), np.repeat(vc, 3, axis=1)
    mha = A.paged_prefill(q, rep[0], rep[1], tab, qs, ctx, 0.5, B)
    np.testing.assert_array_equal(gqa, mha)


def test_rows_outside_every_sequence_stay_zero():
    rng = np.random.default_rng(57)
    q, kc, vc, tab, qs, ctx, _, _ = _prefill_problem(rng, 2, 1, 4, 4, [5], [3])
    q = np.concatenate([q, rng.normal(size=(2, 2, 4))])
    out = A.paged_prefill(q, kc, vc, tab, qs, ctx, 0.5, 4)
    assert (out[3:] == 0).all() and np.isfinite(out[:3]).all()
