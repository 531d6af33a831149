"""GPU parity of pa_prefill (causal paged prefill on the tensor cores)
against the oracle's paged_prefill, element by element, on seeded inputs:
whole prompts, later chunks over a cached prefix, single new tokens, GQA
group sizes 1 to 8, d_head 64 and 128, block sizes 8 to 32, bf16 and fp32
outputs, NaN-filled pools (junk past every context), random placement."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from _gpu_util import assert_attention_close, from_bits, out_to_f64, to_bits

pytestmark = pytest.mark.gpu

api = pytest.importorskip("paged_kv_cache_124_gb300.api")
from paged_kv_cache_124_gb300 import inputs as I  # noqa: E402


def _problem(seed, Hq, Hkv, D, B, ctxs, news, extra_blocks=7, extra_rows=0):
    S = len(ctxs)
    nblk = [-(-c // B) for c in ctxs]
    NB = sum(nblk) + extra_blocks
    perm = I.permutation(NB, seed)
    MB = max(nblk + [1]) + 2
    tables = np.full((S, MB), -1, dtype=np.int32)
    kb = np.full((NB, Hkv, B, D), I.NAN_BF16_BITS, dtype=np.uint16)
    vb = kb.copy()
    pos = 0
    for s, c in enumerate(ctxs):
        k = to_bits(I.bf16_normal((Hkv, c, D), seed * 1000 + 2 * s))
        v = to_bits(I.bf16_normal((Hkv, c, D), seed * 1000 + 2 * s + 1))
        for lb in range(nblk[s]):
            phys = int(perm[pos])
            pos += 1
            tables[s, lb] = phys
            m = min(B, c - lb * B)
            kb[phys, :, :m] = k[:, lb * B:lb * B + m]
            vb[phys, :, :m] = v[:, lb * B:lb * B + m]
    qs = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    T = int(qs[-1]) + extra_rows
    qb = to_bits(I.bf16_normal((T, Hq, D), seed * 1000 + 999))
    return qb, kb, vb, tables, qs, np.array(ctxs, dtype=np.int32)


def _run(qb, kb, vb, tables, qs, ctx, B, Hq, Hkv, D, out_dtype, max_q=None, fill=None):
    dev = lambda a: torch.from_numpy(a).cuda()
    out = torch.full((qb.shape[0], Hq, D), float("nan") if fill is None else fill, dtype=out_dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mq = int(np.diff(qs).max()) if max_q is None else max_q
    api.pa_prefill(out, from_bits(qb), from_bits(kb), from_bits(vb), dev(tables), dev(qs), dev(ctx), mq, B,
                   1.0 / math.sqrt(D), Hq, Hkv, D, status=status)
    torch.cuda.synchronize()
    return out, int(status.item())


CASES = [
    # name, Hq, Hkv, D, B, ctxs, news
    ("g2_d64_b16_ragged", 4, 2, 64, 16, [1, 15, 16, 17, 40, 130], [1, 15, 16, 17, 7, 130]),
    ("g4_d128_b16_8b", 32, 8, 128, 16, [300, 1000, 129, 257], [300, 129, 1, 33]),
    ("g1_d128_b32_mha", 8, 8, 128, 32, [200, 500], [200, 64]),
    ("g8_d128_b8", 32, 4, 128, 8, [100, 77, 260], [100, 20, 3]),
    ("g4_d64_b32_chunks", 16, 4, 64, 32, [1024, 513], [256, 513]),
]


@pytest.mark.parametrize("name,Hq,Hkv,D,B,ctxs,news", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_prefill_matches_oracle(name, Hq, Hkv, D, B, ctxs, news, out_dtype):
    qb, kb, vb, tab, qs, ctx = _problem(3, Hq, Hkv, D, B, ctxs, news)
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(D), B)
    got, status = _run(qb, kb, vb, tab, qs, ctx, B, Hq, Hkv, D, out_dtype)
    assert status == 0
    assert_attention_close(out_to_f64(got), want, out_dtype == torch.float32, name)


def test_prefill_uncovered_rows_and_empty_sequences_untouched():
    # a sequence with no new tokens in the middle, and two rows past the last sequence
    qb, kb, vb, tab, qs, ctx = _problem(4, 8, 2, 128, 16, [50, 30, 90], [50, 0, 17], extra_rows=2)
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(128), 16)
    got, status = _run(qb, kb, vb, tab, qs, ctx, 16, 8, 2, 128, torch.float32, fill=-7.0)
    assert status == 0
    g = out_to_f64(got)
    assert (g[67:] == -7.0).all()
    assert_attention_close(g[:67], want[:67], True, "covered rows")


def test_prefill_equals_decode_for_single_tokens():
    """n = 1 for every sequence is a decode step: both kernels agree with the
    oracle, and with each other within the two tolerances."""
    ctxs = [1, 17, 300, 1024]
    qb, kb, vb, tab, qs, ctx = _problem(5, 32, 8, 128, 16, ctxs, [1] * 4)
    got, status = _run(qb, kb, vb, tab, qs, ctx, 16, 32, 8, 128, torch.float32)
    assert status == 0
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(128), 16)
    assert_attention_close(out_to_f64(got), want, True, "n=1")
    np.testing.assert_array_equal(want, A.paged_decode(qb, kb, vb, tab, ctx, 1.0 / math.sqrt(128), 16))


def test_prefill_chunked_equals_whole_prompt():
    """The last chunk of a prompt computed alone over the cached prefix gives
    the rows of the whole-prompt pass (same kernel, same tiles of keys)."""
    L, cut = 700, 300
    qb, kb, vb, tab, qs, ctx = _problem(6, 32, 8, 128, 16, [L], [L])
    whole, st1 = _run(qb, kb, vb, tab, qs, ctx, 16, 32, 8, 128, torch.float32)
    part, st2 = _run(qb[cut:], kb, vb, tab, np.array([0, L - cut], np.int32), ctx, 16, 32, 8, 128, torch.float32)
    assert st1 == st2 == 0
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(128), 16)
    assert_attention_close(out_to_f64(part), want[cut:], True, "chunk")
    assert_attention_close(out_to_f64(whole), want, True, "whole")


def test_prefill_row_maxima_growing_across_tiles():
    """Rows whose maximum score keeps growing: every q row shares a component
    along d = 0, and the first key of every later 128-key tile is a spike
    along it, so a row's maximum grows by about 5 to 9 (natural log) per tile,
    around the kernel's bound of 2^8 on a weight.  O is then rescaled in
    tensor memory for some rows and tiles and not for others (checked on the
    inputs below), and the output still matches the oracle."""
    Hq, Hkv, D, B, L = 16, 4, 128, 16, 600
    G = Hq // Hkv
    qb, kb, vb, tab, qs, ctx = _problem(9, Hq, Hkv, D, B, [L], [L])
    scale = 1.0 / math.sqrt(D)
    q = from_bits(qb, "cpu").float()
    q[:, :, 0] += 4.0
    qb = to_bits(q.to(torch.bfloat16))
    k = from_bits(kb, "cpu").float()
    for t in range(1, -(-L // 128)):
        blk, off = tab[0, (128 * t) // B], (128 * t) % B
        k[blk, :, off, :] = 0.0
        k[blk, :, off, 0] = 7.0 * t / (4.0 * scale)
    kb = to_bits(k.to(torch.bfloat16))
    # the inputs reach both sides of the bound: simulate the kernel's rule (the
    # running maximum moves only when a tile's maximum exceeds it by more than
    # 8 in log2 units) on the rows that see more than one tile
    qf = from_bits(qb, "cpu").double().numpy()
    kf = from_bits(kb, "cpu").double().numpy()
    kseq = np.stack([kf[tab[0, j // B], :, j % B, :] for j in range(L)], axis=1)     # [Hkv][L][D]
    c = scale / math.log(2.0)
    moved = still = 0
    for i in range(128, L, 7):
        for g in range(0, Hq, 3):
            s = (kseq[g // G, :i + 1] @ qf[i, g]) * c
            m_used = s[:128].max()
            n = 0
            for t in range(1, i // 128 + 1):
                mt = s[128 * t:128 * (t + 1)].max()
                if mt > m_used + 8.0:
                    m_used, n = mt, n + 1
            moved += n > 0
            still += n == 0
    assert moved > 0 and still > 0, (moved, still)
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, scale, B)
    for out_dtype in (torch.float32, torch.bfloat16):
        got, status = _run(qb, kb, vb, tab, qs, ctx, B, Hq, Hkv, D, out_dtype)
        assert status == 0
        assert_attention_close(out_to_f64(got), want, out_dtype == torch.float32, "growing maxima")


def test_prefill_weights_finer_than_bf16():
    """Rows whose softmax weights bf16 cannot carry: 64 two-position
    sequences, key 0 all zeros and key 1 with one component c, so row 1's
    weights are 1 and e^c (relative to the maximum) with V rows -4 and +4.
    The values of c are the bf16 numbers in [-4, 0) whose e^c lies farthest
    from a bf16 number (checked below: weights rounded to bf16 would move
    these outputs by up to ~7e-3, past the 2e-3 bound).  The kernel carries
    each weight in fp16 (a relative 2^-11, moving these outputs by at most
    ~5e-4), so the fp32 outputs stay within 2e-3."""
    S, Hq, Hkv, D, B = 64, 1, 1, 64, 16
    cand = torch.arange(-4.0, 0.0, 2.0 ** -9, dtype=torch.float64).to(torch.bfloat16).unique()
    cand = cand[cand < 0].double()
    p = torch.exp(cand)
    p_bf16 = p.float().to(torch.bfloat16).double()
    moved = (p_bf16 - p).abs() * 8.0 / (1.0 + p) ** 2        # |d o / d p| = |V1 - V0| / (1 + p)^2
    c = cand[torch.argsort(moved, descending=True)[:S]]
    assert float(moved.max()) > 5e-3
    qb, kb, vb, tab, qs, ctx = _problem(15, Hq, Hkv, D, B, [2] * S, [2] * S)
    q = torch.zeros((2 * S, Hq, D))
    q[:, :, 0] = math.sqrt(D)                              # scale * q . k = k[0]
    kf = torch.zeros((kb.shape[0], Hkv, B, D))
    vf = torch.full((kb.shape[0], Hkv, B, D), float("nan"))
    for s_ in range(S):
        blk = tab[s_, 0]
        kf[blk, :, 1, 0] = float(c[s_])
        vf[blk, :, 0, :] = -4.0
        vf[blk, :, 1, :] = 4.0
    qb, kb, vb = to_bits(q.to(torch.bfloat16)), to_bits(kf.to(torch.bfloat16)), to_bits(vf.to(torch.bfloat16))
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(D), B)
    # what bf16-rounded weights (normalised by the unrounded sum) would give
    p_row = torch.exp(c)
    bf_row = (-4.0 + 4.0 * p_row.float().to(torch.bfloat16).double()) / (1.0 + p_row)
    assert np.abs(bf_row.numpy() - want[1::2, 0, 0]).max() > 2e-3
    got, status = _run(qb, kb, vb, tab, qs, ctx, B, Hq, Hkv, D, torch.float32)
    assert status == 0
    assert_attention_close(out_to_f64(got), want, True, "weights finer than bf16")


def _set_v(vb, tab, B, s, pos, cols, val):
    """V of sequence s, position pos, columns cols, every KV head, to val (bf16)."""
    blk, off = tab[s, pos // B], pos % B
    vb[blk, :, off, cols] = to_bits(torch.tensor(float(val)).to(torch.bfloat16).reshape(1))[0]


def test_prefill_values_beyond_fp16_range():
    """The value products run in fp16 where V allows it: a 128-position V
    tile whose values are all of magnitude below 2^16 (and finite) goes as
    fp16, exactly for magnitudes down to 2^-14; a tile holding 2^16 or more
    stays bf16 and its weights go as bf16 hi + lo terms.  Here tiles of
    both kinds alternate in the same rows: spikes of +-2^17 in columns 0
    and 1 at one position of the odd tiles (and of each sequence's last,
    ragged tile, whose rows past the context hold NaN), and +-65280 (the
    largest bf16 below 2^16) and 2^-20 in columns 2 to 4 of the even
    tiles.  Columns 5 and up hold ordinary values and meet the fp32 bound;
    the large columns meet the element rule (2e-3 + 1e-2 relative)."""
    Hq, Hkv, D, B = 16, 4, 128, 16
    ctxs, news = [700, 300, 129], [700, 172, 129]
    qb, kb, vb, tab, qs, ctx = _problem(21, Hq, Hkv, D, B, ctxs, news)
    for s_, c in enumerate(ctxs):
        last = (c - 1) // 128
        for t in range(last + 1):
            pos = min(128 * t + 5 + 11 * s_, c - 1)
            if t % 2 == 1 or t == last:
                _set_v(vb, tab, B, s_, pos, 0, 2.0 ** 17)
                _set_v(vb, tab, B, s_, pos, 1, -3.0 * 2.0 ** 16)
            else:
                _set_v(vb, tab, B, s_, pos, 2, 65280.0)
                _set_v(vb, tab, B, s_, pos + 1, 3, -65280.0)
                _set_v(vb, tab, B, s_, pos, 4, 2.0 ** -20)
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(D), B)
    got, status = _run(qb, kb, vb, tab, qs, ctx, B, Hq, Hkv, D, torch.float32)
    assert status == 0
    g = out_to_f64(got)
    assert_attention_close(g[:, :, 5:], want[:, :, 5:], True, "ordinary columns")
    assert_attention_close(g[:, :, :5], want[:, :, :5], False, "large columns")


def test_prefill_all_values_beyond_fp16_range():
    """Every V value scaled by 2^17 (so every tile stays bf16, with bf16
    hi + lo weights): attention is linear in V and the scaling is exact, so
    the output over 2^17 must meet the fp32 bound against the oracle on the
    unscaled values."""
    Hq, Hkv, D, B = 8, 2, 64, 16
    ctxs, news = [400, 260], [400, 100]
    qb, kb, vb, tab, qs, ctx = _problem(22, Hq, Hkv, D, B, ctxs, news)
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(D), B)
    vs = (from_bits(vb, "cpu").float() * 2.0 ** 17).to(torch.bfloat16)       # exact; NaN junk stays NaN
    got, status = _run(qb, kb, to_bits(vs), tab, qs, ctx, B, Hq, Hkv, D, torch.float32)
    assert status == 0
    assert_attention_close(out_to_f64(got) / 2.0 ** 17, want, True, "V x 2^17")


@pytest.mark.parametrize("Hq,Hkv,D", [(128, 2, 64), (128, 1, 128), (64, 1, 64)], ids=["g64_d64", "g128_d128", "g64_one_kv"])
def test_prefill_largest_groups(Hq, Hkv, D):
    """Group sizes 64 and 128 (the largest the call takes): a 128-row Q tile
    then holds 2 tokens or 1 token of all the group's heads."""
    ctxs, news = [70, 33, 129], [70, 5, 40]
    qb, kb, vb, tab, qs, ctx = _problem(11, Hq, Hkv, D, 16, ctxs, news)
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(D), 16)
    for out_dtype in (torch.float32, torch.bfloat16):
        got, status = _run(qb, kb, vb, tab, qs, ctx, 16, Hq, Hkv, D, out_dtype)
        assert status == 0
        assert_attention_close(out_to_f64(got), want, out_dtype == torch.float32, "G=%d" % (Hq // Hkv))


def test_prefill_device_flags():
    qb, kb, vb, tab, qs, ctx = _problem(7, 8, 2, 64, 16, [40, 20], [40, 20])
    bad_ctx = ctx.copy()
    bad_ctx[1] = 10                                 # fewer positions than new tokens
    got, status = _run(qb, kb, vb, tab, qs, bad_ctx, 16, 8, 2, 64, torch.float32, fill=-3.0)
    assert status & api.PA_DEV_BAD_CONTEXT
    assert (out_to_f64(got)[40:] == -3.0).all()
    want = A.paged_prefill(qb, kb, vb, tab, qs[:2], ctx[:1], 1.0 / 8.0, 16)
    assert_attention_close(out_to_f64(got)[:40], want[:40], True, "good sequence")
    bad_tab = tab.copy()
    bad_tab[0, 1] = kb.shape[0] + 5                 # outside the pool
    _, status = _run(qb, kb, vb, bad_tab, qs, ctx, 16, 8, 2, 64, torch.float32)
    assert status & api.PA_DEV_BAD_BLOCK_ID


def test_prefill_host_errors():
    qb, kb, vb, tab, qs, ctx = _problem(8, 6, 2, 64, 16, [20], [20])
    with pytest.raises(api.PAError) as e:         # G = 3 does not divide 128
        _run(qb, kb, vb, tab, qs, ctx, 16, 6, 2, 64, torch.float32)
    assert e.value.status == api.PA_ERR_UNSUPPORTED
    qb, kb, vb, tab, qs, ctx = _problem(8, 8, 2, 64, 16, [20], [20])
    q, k, v = from_bits(qb), from_bits(kb), from_bits(vb)
    dev = lambda a: torch.from_numpy(a).cuda()
    out = torch.full(q.shape, -1.0, dtype=torch.float32, device="cuda")
    # nothing to compute: returns at once and writes nothing
    api.pa_prefill(out, q, k, v, dev(tab), dev(qs), dev(ctx), 0, 16, 0.125, 8, 2, 64)
    torch.cuda.synchronize()
    assert (out == -1.0).all()
    with pytest.raises(api.PAError) as e:         # misaligned q
        flat = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device="cuda")
        q_mis = flat[1:1 + q.numel()].view(q.shape)
        api.pa_prefill(out, q_mis, k, v, dev(tab), dev(qs), dev(ctx), 20, 16, 0.125, 8, 2, 64)
    assert e.value.status == api.PA_ERR_MISALIGNED
    need = api.pa_prefill_workspace_size(1, tab.shape[1], 16, 2, 64)
    small = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.PAError) as e:         # workspace too small
        api.pa_prefill(out, q, k, v, dev(tab), dev(qs), dev(ctx), 20, 16, 0.125, 8, 2, 64, workspace=small)
    assert e.value.status == api.PA_ERR_WORKSPACE
    assert (out == -1.0).all()


def test_prefill_workspace_reused_across_calls():
    """One caller workspace for calls of different shapes in a row (each call
    restages V over whatever the last one left): every result equals the
    call with a fresh workspace, bit for bit, and the oracle."""
    D, B = 64, 16
    problems = [(31, 8, 2, [300, 90], [300, 40]), (32, 16, 4, [129, 700, 5], [129, 260, 5]),
                (33, 8, 2, [1000], [17])]
    ws = torch.empty(max(api.pa_prefill_workspace_size(len(c), -(-max(c) // B) + 2, B, hkv, D)
                         for _, _, hkv, c, _ in problems), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)                                   # junk format bytes and values
    for seed, Hq, Hkv, ctxs, news in problems:
        qb, kb, vb, tab, qs, ctx = _problem(seed, Hq, Hkv, D, B, ctxs, news)
        fresh, st0 = _run(qb, kb, vb, tab, qs, ctx, B, Hq, Hkv, D, torch.float32)
        dev = lambda a: torch.from_numpy(a).cuda()
        out = torch.full((qb.shape[0], Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        api.pa_prefill(out, from_bits(qb), from_bits(kb), from_bits(vb), dev(tab), dev(qs), dev(ctx), max(news), B,
                       1.0 / math.sqrt(D), Hq, Hkv, D, status=status, workspace=ws)
        torch.cuda.synchronize()
        assert st0 == 0 and int(status.item()) == 0
        assert torch.equal(out.view(torch.int32), fresh.view(torch.int32)), "seed %d" % seed
        want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(D), B)
        assert_attention_close(out_to_f64(out), want, True, "reused workspace")


def test_prefill_work_claiming_orders_agree():
    """Several work items per thread block: the items claimed from the shared
    counters (default), from a caller's pair, and in the fixed round-robin
    order give identical bits, match the oracle, and leave the counters zero."""
    rng = np.random.default_rng(11)
    news = [int(x) for x in rng.integers(65, 400, size=24)]
    ctxs = [n + int(p) for n, p in zip(news, rng.integers(0, 600, size=24))]
    qb, kb, vb, tab, qs, ctx = _problem(12, 16, 4, 64, 16, ctxs, news)
    dev = lambda a: torch.from_numpy(a).cuda()
    args = (from_bits(qb), from_bits(kb), from_bits(vb), dev(tab), dev(qs), dev(ctx), max(news), 16, 0.125, 16, 4, 64)
    outs = []
    mine = torch.zeros(2, dtype=torch.int32, device="cuda")
    for counters in (None, mine, False, mine):
        out = torch.full((qb.shape[0], 16, 64), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        api.pa_prefill(out, *args, status=status, counters=counters)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append(out.cpu())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert mine.cpu().tolist() == [0, 0]
    assert api.prefill_counters("cuda").cpu().tolist() == [0, 0]
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 0.125, 16)
    assert_attention_close(out_to_f64(outs[0]), want, True, "claimed items")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_prefill_output_16_and_32_byte_aligned_agree(out_dtype):
    """Rows are written with 32-byte stores when out is 32-byte aligned and
    with 16-byte stores otherwise: the same bits either way."""
    Hq, Hkv, D, B = 16, 4, 128, 16
    qb, kb, vb, tab, qs, ctx = _problem(13, Hq, Hkv, D, B, [300, 170], [300, 90])
    dev = lambda a: torch.from_numpy(a).cuda()
    T = qb.shape[0]
    outs = []
    for shift in (0, 16 // torch.tensor([], dtype=out_dtype).element_size()):
        flat = torch.full((T * Hq * D + 64,), float("nan"), dtype=out_dtype, device="cuda")
        base = (-flat.data_ptr() // flat.element_size()) % (32 // flat.element_size())   # 32-byte aligned start
        out = flat[base + shift: base + shift + T * Hq * D].view(T, Hq, D)
        assert (out.data_ptr() % 32 == 0) == (shift == 0)
        api.pa_prefill(out, from_bits(qb), from_bits(kb), from_bits(vb), dev(tab), dev(qs), dev(ctx), 300, B,
                       1.0 / math.sqrt(D), Hq, Hkv, D)
        torch.cuda.synchronize()
        outs.append(out.clone())
    assert torch.equal(outs[0].view(torch.int8), outs[1].view(torch.int8))
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(D), B)
    assert_attention_close(out_to_f64(outs[0]), want, out_dtype == torch.float32, "aligned")


def _bench_metadata(sc):
    """Tables and slots from the C++ block manager in the seeded free order,
    as the prefill bench builds them."""
    alloc = api.BlockAllocator(sc.num_blocks, sc.block_size)
    assert alloc.set_free_order(sc.free_order) == 0
    for s, c in enumerate(sc.ctxs):
        assert alloc.allocate(s, c) == 0
    seqs = list(range(len(sc.ctxs)))
    tables, ctx = alloc.build_tables(seqs, max(len(alloc.block_table(s)) for s in seqs))
    slots = np.concatenate([alloc.slot_mapping(s, c - n, n) for s, (c, n) in enumerate(zip(sc.ctxs, sc.news))])
    return tables, ctx, slots


@pytest.mark.parametrize("workload", ["prefill_prompts", "chunked_prefill"])
def test_prefill_full_size_bench_workload_sampled_rows(workload):
    """The bench's full-size workloads (16 prompts of 2,003 tokens; 8 chunks of
    512 over 2K-8K contexts), written with reshape_and_cache and attended with
    the bench's call (bf16 output, shared work-claim counters): windows of
    rows at the start, the middle and the end of sequences against the oracle,
    which computes a window as the same sequence cut after its last row."""
    sc = getattr(I, workload)(0, 16)
    dev = torch.device("cuda")
    tables, ctx, slots = _bench_metadata(sc)
    kc, vc = I.prefill_pool(sc, dev)
    q = I.prefill_q(sc, dev)
    k_new, v_new = I.prefill_new_kv(sc, dev)
    api.pa_reshape_and_cache(kc, vc, k_new, v_new, torch.from_numpy(slots).to(dev))
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    api.pa_prefill(out, q, kc, vc, torch.from_numpy(tables).to(dev), torch.from_numpy(sc.query_start).to(dev),
                   torch.from_numpy(ctx).to(dev), max(sc.news), sc.block_size, sc.scale, sc.n_q_heads,
                   sc.n_kv_heads, sc.d_head, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kb, vb, qb, got = to_bits(kc), to_bits(vc), to_bits(q), out_to_f64(out)
    S = len(sc.ctxs)
    for s in (0, S // 2, S - 1):
        C, n, q0 = int(sc.ctxs[s]), int(sc.news[s]), int(sc.query_start[s])
        for i0 in sorted({0, n // 2 - 16, n - 32}):
            i1 = min(n, i0 + 32)
            rows = slice(q0 + i0, q0 + i1)
            want = A.paged_prefill(qb[rows], kb, vb, tables[s:s + 1], np.array([0, i1 - i0], np.int32),
                                           np.array([C - n + i1], np.int32), sc.scale, sc.block_size)
            assert_attention_close(got[rows], want, False, "%s seq %d rows %d..%d" % (workload, s, i0, i1))


def test_prefill_32768_token_prompt_windows():
    """One prompt of 32,768 tokens (512 work items per KV head, keys up to
    32,768 per row): windows of rows at the start, the middle and the end."""
    Hq, Hkv, D, B, L = 8, 2, 128, 16, 32768
    qb, kb, vb, tab, qs, ctx = _problem(14, Hq, Hkv, D, B, [L], [L])
    out, status = _run(qb, kb, vb, tab, qs, ctx, B, Hq, Hkv, D, torch.bfloat16)
    assert status == 0
    got = out_to_f64(out)
    for i0 in (0, L // 2 - 16, L - 32):
        i1 = i0 + 32
        want = A.paged_prefill(qb[i0:i1], kb, vb, tab, np.array([0, 32], np.int32),
                                       np.array([i1], np.int32), 1.0 / math.sqrt(D), B)
        assert_attention_close(got[i0:i1], want, False, "rows %d..%d" % (i0, i1))


def test_prefill_captured_in_a_cuda_graph_equals_eager():
    """pa_prefill is a chain of programmatic dependent launches (the V
    staging, then the prefill kernel); captured in a CUDA graph and replayed
    twice (the work-claim counters come back to zero after each call), it
    must give the eager call's output bit for bit."""
    Hq, Hkv, D, B = 16, 4, 128, 16
    ctxs, news = [700, 300], [500, 300]
    qb, kb, vb, tab, qs, ctx = _problem(41, Hq, Hkv, D, B, ctxs, news)
    dev = lambda a: torch.from_numpy(a).cuda()
    args = (from_bits(qb), from_bits(kb), from_bits(vb), dev(tab), dev(qs), dev(ctx), max(news), B,
            1 / math.sqrt(D), Hq, Hkv, D)
    ws = api.prefill_workspace(len(ctxs), tab.shape[1], B, Hkv, D)
    cnt = torch.zeros(2, dtype=torch.int32, device="cuda")
    eager = torch.full((qb.shape[0], Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    api.pa_prefill(eager, *args, workspace=ws, counters=cnt)
    torch.cuda.synchronize()
    out = torch.full_like(eager, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        api.pa_prefill(out, *args, workspace=ws, counters=cnt, stream=s)      # warm-up off the default stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        api.pa_prefill(out, *args, workspace=ws, counters=cnt, stream=torch.cuda.current_stream())
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), eager.view(torch.int32))
        out.fill_(float("nan"))
    assert int(cnt.abs().sum().item()) == 0
