"""GPU parity of the FP8 (E4M3) KV path: pa_reshape_and_cache_fp8 writes the
oracle's codes bit for bit; pa_decode_fp8 matches the oracle's paged
attention over the dequantised cache ("PagedAttention in vLLM: scattered
memory, exact attention", section 11: paging is exact at a given KV
precision) within the decode tolerance, with NaN codes in every unused slot,
random placement, split partitions, block sizes 8 to 32 and q heads of very
different magnitudes."""
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


def _fp8_problem(seed, Hq, Hkv, B, ctxs, k_scale, v_scale, q_mult=None):
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
    q = I.bf16_normal((S, Hq, D), seed * 100 + 99)
    if q_mult is not None:
        q = (q.float() * torch.tensor(q_mult, dtype=torch.float32)[None, :, None]).to(torch.bfloat16)
    return to_bits(q), kc, vc, tables, np.array(ctxs, dtype=np.int32)


def _decode_fp8(qb, kc, vc, tables, ctx, B, Hq, Hkv, k_scale, v_scale, out_dtype, partition=0):
    dev = lambda a: torch.from_numpy(a).cuda()
    q = from_bits(qb)
    out = torch.empty(q.shape, dtype=out_dtype, device="cuda")
    max_ctx = int(ctx.max())
    ws = api.decode_workspace(q.shape[0], Hq, D, max_ctx, partition)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_decode_fp8(out, q, dev(kc), dev(vc), dev(tables), dev(ctx), B, 1 / math.sqrt(D), k_scale, v_scale, Hq,
                      Hkv, D, max_ctx, partition_size=partition, workspace=ws, status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


CASES = [
    ("tiny_g2_b16", 4, 2, 16, [1, 15, 16, 37], 0),
    ("g4_b16_batch", 32, 8, 16, [512, 777, 1024, 1500, 2048, 4096], 0),
    ("g4_odd_kv_heads", 12, 3, 16, [300, 1100, 17], 0),              # G = 4, one KV head per block
    ("g4_two_kv_heads_b8", 8, 2, 8, [1, 8, 9, 2000], 0),
    ("g4_b8_split", 32, 8, 8, [3000, 257, 64], 256),
    ("g4_b32_split", 32, 8, 32, [5000, 100], 512),
    ("g8_b16", 32, 4, 16, [900, 33], 0),
]


@pytest.mark.parametrize("name,Hq,Hkv,B,ctxs,P", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_fp8_matches_oracle(name, Hq, Hkv, B, ctxs, P, out_dtype):
    ks, vs = 4.0 / 448, 3.0 / 448
    qb, kc, vc, tab, ctx = _fp8_problem(5, Hq, Hkv, B, ctxs, ks, vs)
    want = A.paged_decode(qb, Q.dequantize(kc, ks), Q.dequantize(vc, vs), tab, ctx, 1 / math.sqrt(D), B)
    got, st = _decode_fp8(qb, kc, vc, tab, ctx, B, Hq, Hkv, ks, vs, out_dtype, P)
    assert st == 0
    assert_attention_close(out_to_f64(got), want, out_dtype == torch.float32, name)


def test_decode_fp8_heads_of_very_different_magnitude():
    """Each q head is scaled by its own power of two before the f16 product."""
    Hq, Hkv = 8, 2
    mult = [1e-3, 1.0, 37.0, 2.0 ** -20, 1e4, 0.5, 3.0, 1e-6]
    qb, kc, vc, tab, ctx = _fp8_problem(6, Hq, Hkv, 16, [700, 41], 0.01, 0.02, q_mult=mult)
    want = A.paged_decode(qb, Q.dequantize(kc, 0.01), Q.dequantize(vc, 0.02), tab, ctx, 1 / math.sqrt(D), 16)
    got, st = _decode_fp8(qb, kc, vc, tab, ctx, 16, Hq, Hkv, 0.01, 0.02, torch.float32)
    assert st == 0
    assert_attention_close(out_to_f64(got), want, True, "magnitudes")


@pytest.mark.parametrize("B,P", [(16, 256), (8, 512), (32, 0)])
def test_decode_fp8_two_head_blocks_equal_one_head_blocks(B, P):
    """With G = 4 and an even KV head count a thread block covers two KV
    heads (8 query heads).  Each head's products only add exact zeros for the
    other head's columns, so at the same partition size the result must equal,
    bit for bit, decoding each KV head alone (G = 4 with a single KV head takes
    one head per block)."""
    Hq, Hkv, ks, vs = 16, 4, 0.01, 0.02
    ctxs = [1, 700, 2049, 64]
    qb, kc, vc, tab, ctx = _fp8_problem(9, Hq, Hkv, B, ctxs, ks, vs)
    part = P or 768
    both, st = _decode_fp8(qb, kc, vc, tab, ctx, B, Hq, Hkv, ks, vs, torch.float32, part)
    assert st == 0
    for h in range(Hkv):
        one, st = _decode_fp8(np.ascontiguousarray(qb[:, 4 * h:4 * h + 4]), np.ascontiguousarray(kc[:, h:h + 1]),
                              np.ascontiguousarray(vc[:, h:h + 1]), tab, ctx, B, 4, 1, ks, vs, torch.float32, part)
        assert st == 0
        assert torch.equal(one, both[:, 4 * h:4 * h + 4]), "KV head %d" % h


@pytest.mark.parametrize("scale", [4.0 / 448, 0.001])
def test_reshape_and_cache_fp8_bit_exact(scale):
    """Codes equal the oracle's quantisation; with the small scale many
    inputs saturate at +-448."""
    T, Hkv, B, NB = 37, 8, 16, 12
    k = I.bf16_normal((T, Hkv, D), 7)
    v = I.bf16_normal((T, Hkv, D), 8)
    slots = I.permutation(NB * B, 9)[:T].astype(np.int64)
    slots[5] = -1                                        # padding token: nothing written
    kc = torch.full((NB, Hkv, B, D), 0xAB, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_reshape_and_cache_fp8(kc, vc, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), scale, 2 * scale,
                                 status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    want_k = np.full((NB, Hkv, B, D), 0xAB, dtype=np.uint8)
    want_v = want_k.copy()
    kq, vq = Q.quantize(k.float().numpy(), scale), Q.quantize(v.float().numpy(), 2 * scale)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        want_k[s // B, :, s % B] = kq[t]
        want_v[s // B, :, s % B] = vq[t]
    assert np.array_equal(kc.cpu().numpy(), want_k)
    assert np.array_equal(vc.cpu().numpy(), want_v)


def test_fp8_write_then_decode_end_to_end():
    B, Hq, Hkv = 16, 32, 8
    ctxs = [300, 1200, 45]
    NB = sum(-(-c // B) for c in ctxs) + 3
    alloc = api.BlockAllocator(NB, B)
    assert alloc.set_free_order(I.permutation(NB, 3)) == 0
    kc = torch.full((NB, Hkv, B, D), Q.NAN_CODE, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    ks, vs = 0.02, 0.015
    kd = np.zeros((NB, Hkv, B, D))
    vd = np.zeros((NB, Hkv, B, D))
    for s, c in enumerate(ctxs):
        assert alloc.allocate(s, c) == 0
        k = I.bf16_normal((c, Hkv, D), 40 + s)
        v = I.bf16_normal((c, Hkv, D), 50 + s)
        slots = alloc.slot_mapping(s, 0, c)
        api.pa_reshape_and_cache_fp8(kc, vc, k.cuda(), v.cuda(), torch.from_numpy(slots).cuda(), ks, vs)
        kq, vq = Q.quantize(k.float().numpy(), ks), Q.quantize(v.float().numpy(), vs)
        for i, sl in enumerate(slots):
            kd[sl // B, :, sl % B] = Q.e4m3_to_f64(kq[i]) * float(np.float32(ks))
            vd[sl // B, :, sl % B] = Q.e4m3_to_f64(vq[i]) * float(np.float32(vs))
    tables, ctx = alloc.build_tables(list(range(3)), max(len(alloc.block_table(s)) for s in range(3)))
    qb = to_bits(I.bf16_normal((3, Hq, D), 77))
    want = A.paged_decode(qb, kd, vd, tables, ctx, 1 / math.sqrt(D), B)
    got, st = _decode_fp8(qb, kc.cpu().numpy(), vc.cpu().numpy(), tables, ctx, B, Hq, Hkv, ks, vs, torch.float32)
    assert st == 0
    assert_attention_close(out_to_f64(got), want, True, "write+decode")


def test_fp8_argument_errors():
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.uint8, device="cuda")
    q = torch.zeros((1, 4, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    tab = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    ctx = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(api.PAError) as e:
        api.pa_decode_fp8(out, q, kc, kc, tab, ctx, 16, 0.125, 1.0, 1.0, 4, 2, 64, 1)
    assert e.value.status == api.PA_ERR_UNSUPPORTED
    kc = torch.zeros((4, 2, 16, 128), dtype=torch.uint8, device="cuda")
    q = torch.zeros((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(api.PAError) as e:
        api.pa_decode_fp8(out, q, kc, kc, tab, ctx, 16, 0.125, 0.0, 1.0, 4, 2, 128, 1)
    assert e.value.status == api.PA_ERR_INVALID_ARG
    with pytest.raises(api.PAError):
        api.pa_reshape_and_cache_fp8(kc, kc, torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda"),
                                     torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda"),
                                     torch.zeros(1, dtype=torch.int64, device="cuda"), -1.0, 1.0)


# --------------------------------------------------------------------------
# copy-on-write and swapping of FP8 pools: bit copies of one-byte codes
# --------------------------------------------------------------------------

@pytest.mark.parametrize("L,B,Hkv,Dh,P", [(1, 16, 8, 128, 7), (3, 8, 2, 64, 20), (2, 32, 4, 128, 1)])
def test_copy_blocks_fp8_bit_exact(L, B, Hkv, Dh, P):
    from oracle import cache_ops as C
    rng = np.random.default_rng(L * 13 + P)
    NB = 2 * P + 5
    ks = [rng.integers(0, 256, size=(NB, Hkv, B, Dh), dtype=np.uint8) for _ in range(L)]   # NaN codes included
    vs = [rng.integers(0, 256, size=(NB, Hkv, B, Dh), dtype=np.uint8) for _ in range(L)]
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:P], perm[P:2 * P]], axis=1).astype(np.int32)
    kd = [torch.from_numpy(x).cuda() for x in ks]
    vd = [torch.from_numpy(x).cuda() for x in vs]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_copy_blocks(kd, vd, torch.from_numpy(pairs).cuda(), status=st)
    C.copy_blocks(ks, vs, pairs)
    torch.cuda.synchronize()
    for l in range(L):
        assert np.array_equal(kd[l].cpu().numpy(), ks[l]) and np.array_equal(vd[l].cpu().numpy(), vs[l])
    assert st.item() == 0


def test_swap_blocks_fp8_round_trip_bit_exact():
    from oracle import cache_ops as C
    rng = np.random.default_rng(21)
    L, NB, HNB, Hkv, B, Dh = 2, 30, 12, 4, 16, 128
    dk = [rng.integers(0, 256, size=(NB, Hkv, B, Dh), dtype=np.uint8) for _ in range(L)]
    dv = [rng.integers(0, 256, size=(NB, Hkv, B, Dh), dtype=np.uint8) for _ in range(L)]
    hk = [np.zeros((HNB, Hkv, B, Dh), dtype=np.uint8) for _ in range(L)]
    hv = [np.zeros((HNB, Hkv, B, Dh), dtype=np.uint8) for _ in range(L)]
    out_pairs = np.stack([rng.permutation(NB)[:HNB], rng.permutation(HNB)], axis=1).astype(np.int32)
    gk, gv = [torch.from_numpy(x).cuda() for x in dk], [torch.from_numpy(x).cuda() for x in dv]
    pk, pv = [torch.from_numpy(x).pin_memory() for x in hk], [torch.from_numpy(x).pin_memory() for x in hv]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # device -> pinned host, then back into other device blocks
    api.pa_swap_blocks(pk, pv, gk, gv, torch.from_numpy(out_pairs).cuda(), status=st)
    for l in range(L):
        C.swap_blocks(hk[l], hv[l], dk[l], dv[l], out_pairs.tolist())
    torch.cuda.synchronize()
    for l in range(L):
        assert np.array_equal(pk[l].numpy(), hk[l]) and np.array_equal(pv[l].numpy(), hv[l])
    in_pairs = np.stack([np.arange(HNB), rng.permutation(NB)[:HNB]], axis=1).astype(np.int32)
    api.pa_swap_blocks(gk, gv, pk, pv, torch.from_numpy(in_pairs).pin_memory(), status=st)
    for l in range(L):
        C.swap_blocks(dk[l], dv[l], hk[l], hv[l], in_pairs.tolist())
    torch.cuda.synchronize()
    for l in range(L):
        assert np.array_equal(gk[l].cpu().numpy(), dk[l]) and np.array_equal(gv[l].cpu().numpy(), dv[l])
    assert st.item() == 0


def test_fp8_copy_and_swap_reject_mixed_element_types():
    k8 = [torch.zeros((4, 2, 16, 64), dtype=torch.uint8, device="cuda")]
    kb = [torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device="cuda")]
    pairs = torch.tensor([[0, 1]], dtype=torch.int32, device="cuda")
    with pytest.raises(TypeError):
        api.pa_copy_blocks(k8, kb, pairs)
    with pytest.raises(TypeError):
        api.pa_swap_blocks(kb, kb, k8, k8, pairs)


def test_decode_fp8_full_size_batch_sampled_sequences():
    """The bench's FP8 decode: the 64-sequence 8B-shaped batch quantised as
    the bench does it, decoded in one call with the library's default
    partitions; four sequences checked against the oracle over the
    dequantised codes (each gathered into a compact pool of its own blocks)."""
    from paged_kv_cache_124_gb300.runner import ScenarioRunner
    sc = I.batch64_8b(0)
    run = ScenarioRunner(sc, device="cuda", data_device="cpu").replay()
    tables, ctx, max_ctx = run.decode_metadata()
    kc, vc = run.k_caches[0], run.v_caches[0]
    ks = float(kc.float().nan_to_num(0.0).abs().amax()) / 448.0
    vs = float(vc.float().nan_to_num(0.0).abs().amax()) / 448.0
    k8 = (kc.float() / ks).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (vc.float() / vs).to(torch.float8_e4m3fn).view(torch.uint8)
    S = len(sc.decode_seqs)
    q = I.decode_q(sc.seed, 0, S, sc.n_q_heads, sc.d_head).cuda()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = api.decode_workspace(S, sc.n_q_heads, sc.d_head, max_ctx, 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_decode_fp8(out, q, k8, v8, tables, ctx, sc.block_size, sc.scale, ks, vs, sc.n_q_heads, sc.n_kv_heads,
                      sc.d_head, max_ctx, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    got, qb = out_to_f64(out), to_bits(q)
    tab_h, ctx_h = tables.cpu().numpy(), ctx.cpu().numpy()
    for s in (0, 17, 42, S - 1):
        nb = -(-int(ctx_h[s]) // sc.block_size)
        blocks = torch.from_numpy(tab_h[s, :nb].astype(np.int64)).cuda()
        kq, vq = k8.index_select(0, blocks).cpu().numpy(), v8.index_select(0, blocks).cpu().numpy()
        want = A.paged_decode(qb[s:s + 1], Q.dequantize(kq, ks), Q.dequantize(vq, vs),
                              np.arange(nb, dtype=np.int32)[None, :], ctx_h[s:s + 1], sc.scale, sc.block_size)
        assert_attention_close(got[s:s + 1], want, True, "batch64 fp8 seq %d" % s)
