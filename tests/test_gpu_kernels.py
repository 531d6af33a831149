"""GPU parity of each kernel against the oracle on seeded inputs, through the
C ABI (ctypes binding).  Cache writes and copies are compared bit for bit;
attention within the tolerance of _gpu_util."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import cache_ops as C
from _golden import ev, load
from _gpu_util import assert_attention_close, from_bits, out_to_f64, to_bits

pytestmark = pytest.mark.gpu

api = pytest.importorskip("paged_kv_cache_124_gb300.api")
NAN16 = 0x7FC1


def _rand_bits(rng, shape):
    return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)


def _bf16_bits_normal(rng, shape):
    x = torch.from_numpy(rng.standard_normal(size=shape).astype(np.float32)).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# reshape_and_cache / copy_blocks: bit-exact, whole pool
# --------------------------------------------------------------------------

# 8,193 and 10,003 tokens: calls of prefill size
@pytest.mark.parametrize("D,B,Hkv,T", [(64, 16, 2, 5), (128, 8, 8, 300), (128, 32, 4, 77), (64, 8, 1, 1),
                                       (128, 16, 8, 8193), (64, 8, 2, 10003)])
def test_reshape_and_cache_bit_exact(D, B, Hkv, T):
    rng = np.random.default_rng(D + B + T)
    NB = max(40, -(-T // B) + 10)
    kc = _rand_bits(rng, (NB, Hkv, B, D))          # every bit pattern, NaNs included
    vc = _rand_bits(rng, (NB, Hkv, B, D))
    k = _rand_bits(rng, (T, Hkv, D))
    v = _rand_bits(rng, (T, Hkv, D))
    slots = rng.permutation(NB * B)[:T].astype(np.int64)
    slots[rng.random(T) < 0.2] = -1                # padding tokens
    kd, vd = from_bits(kc), from_bits(vc)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_reshape_and_cache(kd, vd, from_bits(k), from_bits(v), torch.from_numpy(slots).cuda(), status=st)
    C.reshape_and_cache(kc, vc, k, v, slots, B)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(kd), kc) and np.array_equal(to_bits(vd), vc)
    assert st.item() == 0


def test_reshape_and_cache_out_of_range_slot_is_skipped_and_flagged():
    rng = np.random.default_rng(3)
    NB, Hkv, B, D = 4, 2, 8, 64
    kc = _rand_bits(rng, (NB, Hkv, B, D))
    kd, vd = from_bits(kc), from_bits(kc)
    k = from_bits(_rand_bits(rng, (2, Hkv, D)))
    slots = torch.tensor([NB * B, 5], dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_reshape_and_cache(kd, vd, k, k, slots, status=st)
    C.reshape_and_cache(kc, kc.copy(), to_bits(k), to_bits(k), [-1, 5], B)
    torch.cuda.synchronize()
    assert st.item() == api.PA_DEV_BAD_SLOT
    assert np.array_equal(to_bits(kd), kc)


def test_reshape_and_cache_bad_slot_in_a_shared_block_skips_only_that_token():
    """A bad slot and a padding token among thousands of good ones are
    skipped alone."""
    rng = np.random.default_rng(5)
    NB, Hkv, B, D, T = 700, 2, 16, 64, 8195
    kc = _rand_bits(rng, (NB, Hkv, B, D))
    vc = _rand_bits(rng, (NB, Hkv, B, D))
    k = _rand_bits(rng, (T, Hkv, D))
    v = _rand_bits(rng, (T, Hkv, D))
    slots = rng.permutation(NB * B)[:T].astype(np.int64)
    slots[4101] = NB * B + 7                       # outside the pool
    slots[4102] = -1                               # padding
    kd, vd = from_bits(kc), from_bits(vc)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_reshape_and_cache(kd, vd, from_bits(k), from_bits(v), torch.from_numpy(slots).cuda(), status=st)
    want = slots.copy()
    want[4101] = -1
    C.reshape_and_cache(kc, vc, k, v, want, B)
    torch.cuda.synchronize()
    assert st.item() == api.PA_DEV_BAD_SLOT
    assert np.array_equal(to_bits(kd), kc) and np.array_equal(to_bits(vd), vc)


def test_reshape_and_cache_empty_is_noop():
    kd = torch.zeros(2, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    e = torch.zeros(0, 1, 64, dtype=torch.bfloat16, device="cuda")
    assert api.pa_reshape_and_cache(kd, kd, e, e, torch.zeros(0, dtype=torch.int64, device="cuda")) == 0


@pytest.mark.parametrize("L,D,B,Hkv,P", [(1, 128, 16, 8, 112), (3, 64, 8, 2, 5), (70, 64, 32, 1, 3)])
def test_copy_blocks_bit_exact(L, D, B, Hkv, P):
    rng = np.random.default_rng(L * 7 + P)
    NB = 2 * P + 4
    ks = [_rand_bits(rng, (NB, Hkv, B, D)) for _ in range(L)]
    vs = [_rand_bits(rng, (NB, Hkv, B, D)) for _ in range(L)]
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:P], perm[P:2 * P]], axis=1).astype(np.int32)   # distinct dsts, no chains
    kd = [from_bits(x) for x in ks]
    vd = [from_bits(x) for x in vs]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_copy_blocks(kd, vd, torch.from_numpy(pairs).cuda(), status=st)
    C.copy_blocks(ks, vs, pairs)
    torch.cuda.synchronize()
    for l in range(L):
        assert np.array_equal(to_bits(kd[l]), ks[l]) and np.array_equal(to_bits(vd[l]), vs[l])
    assert st.item() == 0


def test_copy_blocks_bad_ids_are_skipped_and_flagged():
    rng = np.random.default_rng(4)
    kc = _rand_bits(rng, (4, 1, 8, 64))
    kd = from_bits(kc)
    vd = from_bits(kc)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pairs = torch.tensor([[0, 4], [-1, 2], [1, 3]], dtype=torch.int32, device="cuda")
    api.pa_copy_blocks([kd], [vd], pairs, status=st)
    C.copy_blocks([kc], [kc.copy()], [[1, 3]])
    torch.cuda.synchronize()
    assert st.item() == api.PA_DEV_BAD_BLOCK_ID
    assert np.array_equal(to_bits(kd), kc)


# --------------------------------------------------------------------------
# decode attention
# --------------------------------------------------------------------------

def _paged_problem(rng, lens, Hq, Hkv, D, B, extra=7, junk="nan"):
    nblk = [max(1, -(-L // B)) for L in lens]
    NB = sum(nblk) + extra
    perm = rng.permutation(NB)
    MB = max(nblk)
    tables = np.full((len(lens), MB), -1, dtype=np.int32)
    pos = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[pos:pos + n]
        pos += n
    kc = _bf16_bits_normal(rng, (NB, Hkv, B, D))
    vc = _bf16_bits_normal(rng, (NB, Hkv, B, D))
    # slots past each context hold junk that must never reach the output
    for s, L in enumerate(lens):
        for i in range(L, nblk[s] * B):
            blk, off = tables[s, i // B], i % B
            val = NAN16 if junk == "nan" else (0x7F80 if (i % 2) else 0x447A)   # inf / 1000
            kc[blk, :, off] = val
            vc[blk, :, off] = val
    q = _bf16_bits_normal(rng, (len(lens), Hq, D))
    return q, kc, vc, tables, np.array(lens, dtype=np.int32)


def _run_decode(q, kc, vc, tables, lens, B, scale, Hq, Hkv, D, out_dtype, P=0, max_ctx=None, status=None):
    S = q.shape[0]
    max_ctx = int(max(lens.max(), 1)) if max_ctx is None else max_ctx
    out = torch.empty(S, Hq, D, dtype=out_dtype, device="cuda")
    ws = api.decode_workspace(S, Hq, D, max_ctx, P)
    api.pa_decode(out, from_bits(q), from_bits(kc), from_bits(vc), torch.from_numpy(tables).cuda(),
                  torch.from_numpy(lens).cuda(), B, scale, Hq, Hkv, D, max_ctx, partition_size=P,
                  workspace=ws, status=status)
    torch.cuda.synchronize()
    return out


CASES = [
    # D, Hq, Hkv, B, lens, partition
    (64, 4, 2, 16, [2, 16, 17, 38], 0),
    (128, 32, 8, 16, [1, 17, 100, 513, 1000, 64, 65], 0),
    (128, 32, 8, 16, [1, 17, 100, 513, 1000, 64, 65], 64),
    (128, 8, 8, 8, [3, 250, 129, 8], 128),
    (128, 16, 8, 32, [31, 32, 33, 700], 64),
    (64, 16, 1, 8, [5, 300, 77], 64),
    (128, 16, 2, 16, [40, 200], 64),
    (128, 64, 4, 32, [90, 1], 0),
    (64, 8, 4, 32, [1024 + 7, 15], 256),
]


@pytest.mark.parametrize("D,Hq,Hkv,B,lens,P", CASES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_matches_oracle(D, Hq, Hkv, B, lens, P, out_dtype):
    rng = np.random.default_rng(sum(lens) + D + Hq + B + P)
    q, kc, vc, tables, ctx = _paged_problem(rng, lens, Hq, Hkv, D, B)
    scale = 1.0 / math.sqrt(D)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _run_decode(q, kc, vc, tables, ctx, B, scale, Hq, Hkv, D, out_dtype, P, status=st)
    ref = A.paged_decode(q, kc, vc, tables, ctx, scale, B)
    assert_attention_close(out_to_f64(out), ref, out_dtype == torch.float32, "decode %r" % ((D, Hq, Hkv, B, lens, P),))
    assert st.item() == 0


def test_decode_ignores_infinite_junk_in_tail_slots():
    rng = np.random.default_rng(11)
    lens = [5, 19, 33]
    q, kc, vc, tables, ctx = _paged_problem(rng, lens, 8, 2, 128, 16, junk="inf")
    out = _run_decode(q, kc, vc, tables, ctx, 16, 0.125, 8, 2, 128, torch.float32)
    assert_attention_close(out_to_f64(out), A.paged_decode(q, kc, vc, tables, ctx, 0.125, 16), True)


def test_decode_invariant_under_physical_placement():
    rng = np.random.default_rng(12)
    lens = [300, 47]
    q, kc, vc, tables, ctx = _paged_problem(rng, lens, 8, 2, 128, 16)
    ref = out_to_f64(_run_decode(q, kc, vc, tables, ctx, 16, 0.1, 8, 2, 128, torch.float32))
    perm = rng.permutation(kc.shape[0])
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    tab2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    got = out_to_f64(_run_decode(q, kc2, vc2, tab2, ctx, 16, 0.1, 8, 2, 128, torch.float32))
    assert np.array_equal(got, ref)      # same positions, same order: same bits


def test_decode_single_position_returns_value_row_exactly():
    rng = np.random.default_rng(13)
    q, kc, vc, tables, ctx = _paged_problem(rng, [1, 1, 1], 8, 8, 64, 8)
    out = _run_decode(q, kc, vc, tables, ctx, 8, 0.3, 8, 8, 64, torch.bfloat16)
    want = np.stack([vc[tables[s, 0], :, 0, :] for s in range(3)])
    assert np.array_equal(to_bits(out), want)


def test_decode_zero_context_writes_zeros_and_bad_metadata_is_flagged():
    rng = np.random.default_rng(14)
    q, kc, vc, tables, ctx = _paged_problem(rng, [0, 20, 40], 8, 2, 128, 16)
    out = _run_decode(q, kc, vc, tables, ctx, 16, 0.1, 8, 2, 128, torch.float32)
    assert torch.count_nonzero(out[0]).item() == 0
    assert_attention_close(out_to_f64(out)[1:], A.paged_decode(q, kc, vc, tables, ctx, 0.1, 16)[1:], True)
    # a table entry outside the pool and a context above the stated maximum
    tables2 = tables.copy()
    tables2[1, 0] = kc.shape[0] + 5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _run_decode(q, kc, vc, tables2, ctx, 16, 0.1, 8, 2, 128, torch.float32, status=st)
    assert st.item() & api.PA_DEV_BAD_BLOCK_ID
    st.zero_()
    _run_decode(q, kc, vc, tables, ctx, 16, 0.1, 8, 2, 128, torch.float32, max_ctx=32, status=st)
    assert st.item() & api.PA_DEV_BAD_CONTEXT


def test_decode_host_argument_errors():
    d = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(2, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    tb = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    cl = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(api.PAError) as e:
        api.pa_decode(d, d, kc, kc, tb, cl, 16, 0.1, 4, 2, 64, 16, partition_size=96)
    assert e.value.status == api.PA_ERR_INVALID_ARG
    tb256 = torch.zeros(1, 256, dtype=torch.int32, device="cuda")   # room for 4096 positions
    with pytest.raises(api.PAError) as e:
        api.pa_decode(d, d, kc, kc, tb256, cl, 16, 0.1, 4, 2, 64, 4096, partition_size=64)
    assert e.value.status == api.PA_ERR_WORKSPACE
    q3 = torch.zeros(1, 6, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.PAError) as e:
        api.pa_decode(q3, q3, kc, kc, tb, cl, 16, 0.1, 6, 2, 64, 16)
    assert e.value.status == api.PA_ERR_UNSUPPORTED


def test_split_partials_match_oracle_partition_summaries():
    """The workspace statistics of a split sequence are the (m, z, u) of
    each partition (second page, section 11)."""
    rng = np.random.default_rng(15)
    D, Hq, Hkv, B, P = 128, 8, 2, 16, 64
    lens = [200, 130]
    q, kc, vc, tables, ctx = _paged_problem(rng, lens, Hq, Hkv, D, B)
    S, max_ctx = len(lens), 200
    out = torch.empty(S, Hq, D, dtype=torch.float32, device="cuda")
    ws = api.decode_workspace(S, Hq, D, max_ctx, P)
    api.pa_decode(out, from_bits(q), from_bits(kc), from_bits(vc), torch.from_numpy(tables).cuda(),
                  torch.from_numpy(ctx).cuda(), B, 0.09, Hq, Hkv, D, max_ctx, partition_size=P, workspace=ws)
    torch.cuda.synchronize()
    NP = -(-max_ctx // P)
    n = S * Hq * NP
    al = lambda x: (x + 255) // 256 * 256
    w = ws.cpu().numpy()
    assert not w[:8].any()               # the claim counters in the 256-byte header are left at zero
    w = w[256:]
    pm = w[:4 * n].view(np.float32).reshape(S, Hq, NP)
    ps = w[al(4 * n):al(4 * n) + 4 * n].view(np.float32).reshape(S, Hq, NP)
    pa_ = w[2 * al(4 * n):2 * al(4 * n) + 4 * n * D].view(np.float32).reshape(S, Hq, NP, D)
    for s, L in enumerate(lens):
        K, V = A.gather_kv(kc, vc, tables[s], L, B)
        qs = A.bf16_to_f64(q[s])
        for g in range(Hq):
            parts = A.partition_summaries(qs[g], K[g // (Hq // Hkv)], V[g // (Hq // Hkv)], 0.09, P)
            for p, (m, z, u) in enumerate(parts):
                assert abs(pm[s, g, p] - m) < 1e-4
                assert abs(ps[s, g, p] - z) <= 1e-4 * z
                np.testing.assert_allclose(pa_[s, g, p], u, rtol=1e-4, atol=1e-4 * z)


def test_lse_merge_worked_example():
    """Second page, section 11: page A (m = ln 2, z = 1.5, u = [0.5, 2]) and
    page B (m = ln 4, z = 1.75, u = [4.25, 4.75]) merge to o = [1.8, 2.3]."""
    g = load("p2_worked_attention.json")
    pm = torch.tensor([[[ev(g["stable_A"]["m"]), ev(g["stable_B"]["m"])]]], dtype=torch.float32, device="cuda")
    ps = torch.tensor([[[g["stable_A"]["z"], g["stable_B"]["z"]]]], dtype=torch.float32, device="cuda")
    pu = torch.tensor([[[g["stable_A"]["u"], g["stable_B"]["u"]]]], dtype=torch.float32, device="cuda")
    ctx = torch.tensor([4], dtype=torch.int32, device="cuda")
    out = torch.empty(1, 1, 2, dtype=torch.float32, device="cuda")
    api.pa_lse_merge(out, pm, ps, pu, ctx, g["paging"]["tokens_per_page"])
    torch.cuda.synchronize()
    np.testing.assert_allclose(out.cpu().numpy()[0, 0], g["o"], rtol=1e-6)


def test_lse_merge_random_against_oracle_merge():
    rng = np.random.default_rng(16)
    S, Hq, NP, D = 3, 4, 6, 64
    pm = rng.normal(size=(S, Hq, NP)) * 5
    ps = rng.uniform(0.5, 20, size=(S, Hq, NP))
    pu = rng.normal(size=(S, Hq, NP, D)) * 3
    ctx = np.array([6 * 10, 25, 0], dtype=np.int32)            # 6, 3 and 0 partitions of 10
    out = torch.empty(S, Hq, D, dtype=torch.float32, device="cuda")
    f = lambda a: torch.from_numpy(a.astype(np.float32)).cuda()
    api.pa_lse_merge(out, f(pm), f(ps), f(pu), torch.from_numpy(ctx).cuda(), 10)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for s, npart in enumerate([6, 3, 0]):
        for h in range(Hq):
            if npart == 0:
                assert np.all(got[s, h] == 0)
                continue
            summ = [(float(np.float32(pm[s, h, p])), float(np.float32(ps[s, h, p])), pu[s, h, p].astype(np.float32))
                    for p in range(npart)]
            m, z, u = A.merge_summaries(summ)
            np.testing.assert_allclose(got[s, h], u / z, rtol=1e-5, atol=1e-6)


def test_bounded_wait_runs_out_and_the_gpu_stays_usable():
    """A wait on a barrier that nothing arrives on gives up after its probe
    limit and flags PA_DEV_WAIT_TIMEOUT; no fault, no hang, and the next
    kernels run normally."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_check_bounded_wait(status, max_probes=20000)
    torch.cuda.synchronize()
    assert status.item() == api.PA_DEV_WAIT_TIMEOUT
    # the context is still usable: a decode right after matches the oracle
    rng = np.random.default_rng(9)
    D, B, Hq, Hkv = 64, 16, 4, 2
    ctx = np.array([37, 5], dtype=np.int32)
    NB = 8
    kc = _bf16_bits_normal(rng, (NB, Hkv, B, D))
    vc = _bf16_bits_normal(rng, (NB, Hkv, B, D))
    tab = np.array([[3, 0, 6], [5, -1, -1]], dtype=np.int32)
    qb = _bf16_bits_normal(rng, (2, Hq, D))
    out = torch.empty((2, Hq, D), dtype=torch.float32, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = api.decode_workspace(2, Hq, D, 37, 0)
    api.pa_decode(out, from_bits(qb), from_bits(kc), from_bits(vc), torch.from_numpy(tab).cuda(),
                  torch.from_numpy(ctx).cuda(), B, 1 / math.sqrt(D), Hq, Hkv, D, 37, workspace=ws, status=st2)
    torch.cuda.synchronize()
    assert st2.item() == 0
    want = A.paged_decode(qb, kc, vc, tab, ctx, 1 / math.sqrt(D), B)
    assert_attention_close(out_to_f64(out), want, True, "after a timed-out wait")


# --------------------------------------------------------------------------
# maximum sizes
# --------------------------------------------------------------------------

def test_decode_262144_position_context_256_partitions():
    """One sequence of 2^18 positions: 256 partitions of the library default
    size, merged by the log-sum-exp kernel."""
    rng = np.random.default_rng(21)
    L = 1 << 18
    q, kc, vc, tables, ctx = _paged_problem(rng, [L], 8, 2, 128, 16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _run_decode(q, kc, vc, tables, ctx, 16, 1 / math.sqrt(128), 8, 2, 128, torch.float32, status=st)
    assert st.item() == 0
    ref = A.paged_decode(q, kc, vc, tables, ctx, 1 / math.sqrt(128), 16)
    assert_attention_close(out_to_f64(out), ref, True, "2^18 positions")


def test_decode_8192_short_sequences():
    """A batch of 8,192 sequences of 1 to 64 positions (grid of 8,192 x heads
    blocks, single-partition path)."""
    rng = np.random.default_rng(22)
    lens = rng.integers(1, 65, size=8192).tolist()
    q, kc, vc, tables, ctx = _paged_problem(rng, lens, 8, 2, 64, 16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _run_decode(q, kc, vc, tables, ctx, 16, 0.125, 8, 2, 64, torch.bfloat16, status=st)
    assert st.item() == 0
    ref = A.paged_decode(q, kc, vc, tables, ctx, 0.125, 16)
    assert_attention_close(out_to_f64(out), ref, False, "8192 sequences")
