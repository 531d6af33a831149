"""GPU parity of pa_prefill_fp8 (causal paged prefill over E4M3 caches)
against the oracle's paged_prefill over the dequantised caches ("PagedAttention
in vLLM: scattered memory, exact attention", section 11: paging is exact at a
given KV precision), within the attention tolerance: whole prompts, chunks
over a cached prefix, GQA group sizes 1 to 8, block sizes 8 to 32, NaN codes
in every unused slot, random placement, q rows of very different magnitude.
With power-of-two scales the call must equal, bit for bit, pa_prefill over
bf16 caches holding the dequantised values (every step then agrees exactly:
the scales only move exponents)."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import quant as Q
from _gpu_util import assert_attention_close, from_bits, out_to_f64, to_bits

pytestmark = pytest.mark.gpu

api = pytest.importorskip("paged_kv_cache_124_gb300.api")
from paged_kv_cache_124_gb300 import inputs as I  # noqa: E402

D = 128


def _problem(seed, Hq, Hkv, B, ctxs, news, k_scale, v_scale, q_mult=None):
    S = len(ctxs)
    nblk = [-(-c // B) for c in ctxs]
    NB = sum(nblk) + 5
    perm = I.permutation(NB, seed)
    tables = np.full((S, max(nblk) + 1), -1, dtype=np.int32)
    kc = np.full((NB, Hkv, B, D), Q.NAN_CODE, dtype=np.uint8)      # NaN code in every unused slot
    vc = kc.copy()
    pos = 0
    for s, c in enumerate(ctxs):
        kx = I.bf16_normal((Hkv, c, D), seed * 100 + 2 * s).float().numpy()
        vx = I.bf16_normal((Hkv, c, D), seed * 100 + 2 * s + 1).float().numpy()
        kq, vq = Q.quantize(kx, k_scale), Q.quantize(vx, v_scale)
        for lb in range(nblk[s]):
            phys = int(perm[pos])
            pos += 1
            tables[s, lb] = phys
            m = min(B, c - lb * B)
            kc[phys, :, :m] = kq[:, lb * B:lb * B + m]
            vc[phys, :, :m] = vq[:, lb * B:lb * B + m]
    qs = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    q = I.bf16_normal((int(qs[-1]), Hq, D), seed * 100 + 99)
    if q_mult is not None:
        q = (q.float() * torch.tensor(q_mult, dtype=torch.float32)[None, :, None]).to(torch.bfloat16)
    return to_bits(q), kc, vc, tables, qs, np.array(ctxs, dtype=np.int32)


def _run(qb, kc, vc, tables, qs, ctx, B, Hq, Hkv, ks, vs, out_dtype, workspace=None):
    dev = lambda a: torch.from_numpy(a).cuda()
    q = from_bits(qb)
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_prefill_fp8(out, q, dev(kc), dev(vc), dev(tables), dev(qs), dev(ctx), int(np.diff(qs).max()), B,
                       1 / math.sqrt(D), ks, vs, Hq, Hkv, D, status=st, workspace=workspace)
    torch.cuda.synchronize()
    return out, int(st.item())


CASES = [
    # name, Hq, Hkv, B, ctxs, news
    ("g4_b16_prompts", 32, 8, 16, [300, 1000, 129], [300, 1000, 129]),
    ("g4_b16_chunks", 16, 4, 16, [1500, 700, 257], [200, 64, 1]),
    ("g1_b32", 8, 8, 32, [200, 500], [200, 64]),
    ("g8_b8", 32, 4, 8, [100, 77, 260], [100, 20, 3]),
    ("g2_b16_ragged", 4, 2, 16, [1, 15, 16, 17, 40], [1, 15, 16, 17, 7]),
]


@pytest.mark.parametrize("name,Hq,Hkv,B,ctxs,news", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_prefill_fp8_matches_oracle(name, Hq, Hkv, B, ctxs, news, out_dtype):
    ks, vs = 4.0 / 448, 3.0 / 448
    qb, kc, vc, tab, qs, ctx = _problem(5, Hq, Hkv, B, ctxs, news, ks, vs)
    want = A.paged_prefill(qb, Q.dequantize(kc, ks), Q.dequantize(vc, vs), tab, qs, ctx, 1 / math.sqrt(D), B)
    got, st = _run(qb, kc, vc, tab, qs, ctx, B, Hq, Hkv, ks, vs, out_dtype)
    assert st == 0
    assert_attention_close(out_to_f64(got), want, out_dtype == torch.float32, name)


def test_prefill_fp8_query_heads_of_very_different_magnitude():
    """q heads of very different magnitude (1e-6 up to 1e4) against the
    staged bf16 K: the K scale is applied to the scores, not to q."""
    Hq, Hkv = 8, 2
    mult = [1e-3, 1.0, 37.0, 2.0 ** -20, 1e4, 0.5, 3.0, 1e-6]
    qb, kc, vc, tab, qs, ctx = _problem(6, Hq, Hkv, 16, [700, 300], [700, 41], 0.01, 0.02, q_mult=mult)
    want = A.paged_prefill(qb, Q.dequantize(kc, 0.01), Q.dequantize(vc, 0.02), tab, qs, ctx, 1 / math.sqrt(D), 16)
    got, st = _run(qb, kc, vc, tab, qs, ctx, 16, Hq, Hkv, 0.01, 0.02, torch.float32)
    assert st == 0
    assert_attention_close(out_to_f64(got), want, True, "magnitudes")


@pytest.mark.parametrize("ks,vs", [(2.0 ** -6, 2.0 ** -7), (1.0, 4.0)])
def test_prefill_fp8_equals_bf16_prefill_with_power_of_two_scales(ks, vs):
    """With power-of-two scales every dequantised value is exact in bf16, and
    each step of the FP8 call equals the bf16 call's: the K scale (on the
    scores) and the V scale (on the output) only move exponents.  Outputs
    must be equal bit for bit (fp32 and bf16)."""
    Hq, Hkv, B = 16, 4, 16
    mult = [1.0, 3e3, 1e-3, 0.25] * 4
    qb, kc, vc, tab, qs, ctx = _problem(7, Hq, Hkv, B, [900, 333, 64], [500, 333, 10], ks, vs, q_mult=mult)
    kd = torch.from_numpy(Q.dequantize(kc, ks)).float().to(torch.bfloat16)
    vd = torch.from_numpy(Q.dequantize(vc, vs)).float().to(torch.bfloat16)
    assert np.array_equal(kd.float().numpy()[np.isfinite(Q.dequantize(kc, ks))],
                          Q.dequantize(kc, ks)[np.isfinite(Q.dequantize(kc, ks))])
    dev = lambda a: torch.from_numpy(a).cuda()
    for out_dtype in (torch.float32, torch.bfloat16):
        got, st = _run(qb, kc, vc, tab, qs, ctx, B, Hq, Hkv, ks, vs, out_dtype)
        ref = torch.full(got.shape, float("nan"), dtype=out_dtype, device="cuda")
        st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        api.pa_prefill(ref, from_bits(qb), kd.cuda(), vd.cuda(), dev(tab), dev(qs), dev(ctx), int(np.diff(qs).max()),
                       B, 1 / math.sqrt(D), Hq, Hkv, D, status=st2)
        torch.cuda.synchronize()
        assert st == 0 and int(st2.item()) == 0
        bits = (lambda t: t.view(torch.int32)) if out_dtype == torch.float32 else (lambda t: t.view(torch.int16))
        assert torch.equal(bits(got), bits(ref)), out_dtype


def test_prefill_fp8_full_size_chunks_sampled_rows():
    """The chunked-prefill bench workload's shape (8 chunks of 512 over long
    prefixes, 32/8 heads), FP8: sampled rows of every sequence against the
    oracle."""
    rng = np.random.default_rng(8)
    ctxs = [int(x) for x in rng.integers(2048, 4096, size=4)]
    news = [512] * 4
    Hq, Hkv, B, ks, vs = 32, 8, 16, 4.0 / 448, 3.0 / 448
    qb, kc, vc, tab, qs, ctx = _problem(8, Hq, Hkv, B, ctxs, news, ks, vs)
    got, st = _run(qb, kc, vc, tab, qs, ctx, B, Hq, Hkv, ks, vs, torch.float32)
    assert st == 0
    g = out_to_f64(got)
    kd, vd = Q.dequantize(kc, ks), Q.dequantize(vc, vs)
    for s_ in range(len(ctxs)):
        rows = sorted(set([0, 1, 255, 511] + [int(x) for x in rng.integers(0, 512, size=4)]))
        for r in rows:
            # the oracle on one new position: a one-row "chunk" at its place
            p = ctxs[s_] - news[s_] + r
            one_qs = np.array([0, 1], dtype=np.int32)
            want = A.paged_prefill(qb[qs[s_] + r:qs[s_] + r + 1], kd, vd, tab[s_:s_ + 1], one_qs,
                                   np.array([p + 1], dtype=np.int32), 1 / math.sqrt(D), B)
            assert_attention_close(g[qs[s_] + r:qs[s_] + r + 1], want, True, "seq %d row %d" % (s_, r))


def test_prefill_fp8_errors_and_flags():
    Hq, Hkv, B = 8, 2, 16
    qb, kc, vc, tab, qs, ctx = _problem(9, Hq, Hkv, B, [40, 20], [40, 20], 0.01, 0.01)
    dev = lambda a: torch.from_numpy(a).cuda()
    q = from_bits(qb)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(api.PAError) as e:                 # scales must be finite and > 0
        api.pa_prefill_fp8(out, q, dev(kc), dev(vc), dev(tab), dev(qs), dev(ctx), 40, B, 0.1, 0.0, 0.01, Hq, Hkv, D)
    assert e.value.status == api.PA_ERR_INVALID_ARG
    small = torch.empty(100, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.PAError) as e:
        api.pa_prefill_fp8(out, q, dev(kc), dev(vc), dev(tab), dev(qs), dev(ctx), 40, B, 0.1, 0.01, 0.01, Hq, Hkv, D,
                           workspace=small)
    assert e.value.status == api.PA_ERR_WORKSPACE
    q64 = torch.zeros(q.shape[0], Hq, 64, dtype=torch.bfloat16, device="cuda")
    k64 = torch.zeros(kc.shape[:3] + (64,), dtype=torch.uint8, device="cuda")
    with pytest.raises(api.PAError) as e:                 # d_head 128 only
        api.pa_prefill_fp8(q64.float(), q64, k64, k64, dev(tab), dev(qs), dev(ctx), 40, B, 0.1, 0.01, 0.01, Hq, Hkv,
                           64)
    assert e.value.status == api.PA_ERR_UNSUPPORTED
    bad = tab.copy()
    bad[0, 1] = kc.shape[0] + 3                           # outside the pool
    _, st = _run(qb, kc, vc, bad, qs, ctx, B, Hq, Hkv, 0.01, 0.01, torch.float32)
    assert st & api.PA_DEV_BAD_BLOCK_ID


def test_prefill_fp8_captured_in_a_cuda_graph_equals_eager():
    """The FP8 call (K and V staging, then the prefill kernel) captured in a
    CUDA graph and replayed twice gives the eager call's output bit for bit."""
    Hq, Hkv, B, ks, vs = 16, 4, 16, 4.0 / 448, 3.0 / 448
    qb, kc, vc, tab, qs, ctx = _problem(10, Hq, Hkv, B, [600, 257], [600, 100], ks, vs)
    dev = lambda a: torch.from_numpy(a).cuda()
    args = (from_bits(qb), dev(kc), dev(vc), dev(tab), dev(qs), dev(ctx), 600, B, 1 / math.sqrt(D), ks, vs, Hq, Hkv, D)
    ws = api.prefill_fp8_workspace(2, tab.shape[1], B, Hkv, D)
    cnt = torch.zeros(2, dtype=torch.int32, device="cuda")
    eager = torch.full((qb.shape[0], Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    api.pa_prefill_fp8(eager, *args, workspace=ws, counters=cnt)
    torch.cuda.synchronize()
    out = torch.full_like(eager, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        api.pa_prefill_fp8(out, *args, workspace=ws, counters=cnt, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        api.pa_prefill_fp8(out, *args, workspace=ws, counters=cnt, stream=torch.cuda.current_stream())
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), eager.view(torch.int32))
