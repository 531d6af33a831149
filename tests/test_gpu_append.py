"""pa_decode_append / pa_decode_append_fp8: a decode step's cache write and
attention in one call.  Writing each sequence's new token (position
context_lens[s] - 1) into the cache and attending to it must give, bit for
bit, the output, the cache and the status of pa_reshape_and_cache (or its FP8
form) followed by pa_decode: the same rows land in the same slots and the
same kernels read them.  Pools start with NaN junk, so a stale slot that the
fused call failed to replace would show."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from _gpu_util import assert_attention_close, out_to_f64, to_bits

pytestmark = pytest.mark.gpu

api = pytest.importorskip("paged_kv_cache_124_gb300.api")
from paged_kv_cache_124_gb300 import inputs as I  # noqa: E402


def _problem(seed, Hq, Hkv, D, B, ctxs, fp8=False):
    """Pools with every slot before each sequence's last position filled, the
    last position's slot (and everything unused) NaN junk; the new rows, q,
    tables and the slots of the last positions."""
    rng = np.random.default_rng(seed)
    S = len(ctxs)
    nblk = [-(-c // B) for c in ctxs]
    NB = sum(nblk) + 5
    perm = rng.permutation(NB).astype(np.int32)
    MB = max(nblk + [1]) + 1
    tables = np.full((S, MB), -1, dtype=np.int32)
    pos = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[pos:pos + n]
        pos += n
    if fp8:
        kc = torch.full((NB, Hkv, B, D), 0x7F, dtype=torch.uint8)            # E4M3 NaN code
        vc = kc.clone()
        codes = lambda shape: torch.from_numpy(rng.integers(0, 0x7E, size=shape, dtype=np.uint8) |
                                               (rng.integers(0, 2, size=shape, dtype=np.uint8) << 7))
    else:
        kc = I.nan_pool((NB, Hkv, B, D))
        vc = I.nan_pool((NB, Hkv, B, D))
        codes = lambda shape: I.bf16_normal(shape, int(rng.integers(1 << 30)))
    for s, c in enumerate(ctxs):
        for j in range(c - 1):                       # the cached positions; c - 1 is the new one
            blk, off = tables[s, j // B], j % B
            kc[blk, :, off] = codes((Hkv, D))
            vc[blk, :, off] = codes((Hkv, D))
    k_new = I.bf16_normal((S, Hkv, D), seed * 7 + 1)
    v_new = I.bf16_normal((S, Hkv, D), seed * 7 + 2)
    q = I.bf16_normal((S, Hq, D), seed * 7 + 3)
    slots = np.array([(tables[s, (c - 1) // B] * B + (c - 1) % B) if c > 0 else -1 for s, c in enumerate(ctxs)],
                     dtype=np.int64)
    return q, kc, vc, k_new, v_new, tables, np.array(ctxs, dtype=np.int32), slots


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else (t.view(torch.int32) if t.dtype == torch.float32
                                                                   else t)


def _both(q, kc, vc, k_new, v_new, tables, ctx, slots, B, Hq, Hkv, D, out_dtype, P=0, fp8=False, scales=(0.01, 0.02),
          max_ctx=None):
    dev = "cuda"
    q, k_new, v_new = q.to(dev), k_new.to(dev), v_new.to(dev)
    tab, ctx_d = torch.from_numpy(tables).to(dev), torch.from_numpy(ctx).to(dev)
    max_ctx = int(ctx.max()) if max_ctx is None else max_ctx
    ws = api.decode_workspace(q.shape[0], Hq, D, max_ctx, P)
    res = []
    for fused in (False, True):
        k_, v_ = kc.clone().to(dev), vc.clone().to(dev)
        out = torch.full(q.shape, float("nan"), dtype=out_dtype, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        if fused:
            api.pa_decode_append(out, q, k_, v_, k_new, v_new, tab, ctx_d, B, 1 / math.sqrt(D), Hq, Hkv, D, max_ctx,
                                 partition_size=P, workspace=ws, status=st,
                                 k_scale=scales[0] if fp8 else None, v_scale=scales[1] if fp8 else None)
        else:
            sl = torch.from_numpy(slots).to(dev)
            if fp8:
                api.pa_reshape_and_cache_fp8(k_, v_, k_new, v_new, sl, scales[0], scales[1], status=st)
                api.pa_decode_fp8(out, q, k_, v_, tab, ctx_d, B, 1 / math.sqrt(D), scales[0], scales[1], Hq, Hkv, D,
                                  max_ctx, partition_size=P, workspace=ws, status=st)
            else:
                api.pa_reshape_and_cache(k_, v_, k_new, v_new, sl, status=st)
                api.pa_decode(out, q, k_, v_, tab, ctx_d, B, 1 / math.sqrt(D), Hq, Hkv, D, max_ctx,
                              partition_size=P, workspace=ws, status=st)
        torch.cuda.synchronize()
        res.append((out, k_, v_, int(st.item())))
    return res


CASES = [
    # name, Hq, Hkv, D, B, ctxs, partition
    ("g4_d128_b16", 32, 8, 128, 16, [1, 17, 300, 1024, 2049], 0),
    ("g4_d128_b16_split", 32, 8, 128, 16, [1, 16, 700, 2049], 256),
    ("g2_d64_b8", 8, 4, 64, 8, [2, 9, 64, 513], 64),
    ("g1_d128_b32", 8, 8, 128, 32, [31, 32, 33, 1000], 0),
    ("g16_d128_b16_two_sub_blocks", 32, 2, 128, 16, [5, 400, 1500], 512),
    ("g8_d64_b16", 16, 2, 64, 16, [16, 161], 0),
]


@pytest.mark.parametrize("name,Hq,Hkv,D,B,ctxs,P", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_append_equals_cache_write_then_decode(name, Hq, Hkv, D, B, ctxs, P, out_dtype):
    q, kc, vc, k_new, v_new, tab, ctx, slots = _problem(1, Hq, Hkv, D, B, ctxs)
    (o1, k1, v1, s1), (o2, k2, v2, s2) = _both(q, kc, vc, k_new, v_new, tab, ctx, slots, B, Hq, Hkv, D, out_dtype, P)
    assert s1 == s2 == 0
    assert torch.equal(_bits(k1), _bits(k2)) and torch.equal(_bits(v1), _bits(v2)), "caches differ"
    assert torch.equal(_bits(o1), _bits(o2)), "outputs differ"
    if out_dtype == torch.float32 and name == "g4_d128_b16":     # and both match the oracle
        want = A.paged_decode(to_bits(q), to_bits(k2.cpu()), to_bits(v2.cpu()), tab, ctx, 1 / math.sqrt(D), B)
        assert_attention_close(out_to_f64(o2), want, True, "append vs oracle")


FP8_CASES = [
    # name, Hq, Hkv, D, B, ctxs, partition: G = 4 with an even KV head count takes two heads per block
    ("g4_two_heads_b16", 32, 8, 128, 16, [1, 17, 300, 2049], 0),
    ("g4_two_heads_b8_split", 16, 4, 128, 8, [2, 700, 1025], 256),
    ("g4_one_head_b32", 12, 3, 128, 32, [33, 500], 0),
    ("g2_b16", 8, 4, 128, 16, [16, 1000], 512),
]


@pytest.mark.parametrize("name,Hq,Hkv,D,B,ctxs,P", FP8_CASES, ids=[c[0] for c in FP8_CASES])
def test_append_fp8_equals_cache_write_then_decode(name, Hq, Hkv, D, B, ctxs, P):
    q, kc, vc, k_new, v_new, tab, ctx, slots = _problem(2, Hq, Hkv, D, B, ctxs, fp8=True)
    (o1, k1, v1, s1), (o2, k2, v2, s2) = _both(q, kc, vc, k_new, v_new, tab, ctx, slots, B, Hq, Hkv, D, torch.float32,
                                               P, fp8=True, scales=(4.0 / 448, 3.0 / 448))
    assert s1 == s2 == 0
    assert torch.equal(k1, k2) and torch.equal(v1, v2), "FP8 caches differ"
    assert torch.equal(_bits(o1), _bits(o2)), "outputs differ"


def test_append_skips_empty_and_clamped_contexts():
    """Context 0 appends nothing and gives zeros; a context above the stated
    maximum is clamped, flagged and appends nothing; the others append."""
    Hq, Hkv, D, B = 8, 2, 64, 16
    q, kc, vc, k_new, v_new, tab, ctx, slots = _problem(3, Hq, Hkv, D, B, [40, 1, 90])
    ctx = np.array([40, 0, 90], dtype=np.int32)
    dev = "cuda"
    k_, v_ = kc.clone().to(dev), vc.clone().to(dev)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    max_ctx = 64                                           # below the third context: clamped
    api.pa_decode_append(out, q.to(dev), k_, v_, k_new.to(dev), v_new.to(dev), torch.from_numpy(tab).to(dev),
                         torch.from_numpy(ctx).to(dev), B, 0.125, Hq, Hkv, D, max_ctx,
                         workspace=api.decode_workspace(3, Hq, D, max_ctx, 0), status=st)
    torch.cuda.synchronize()
    assert st.item() & api.PA_DEV_BAD_CONTEXT
    kb, kb0 = to_bits(k_.cpu()), to_bits(kc)
    changed = np.argwhere((kb != kb0).any(axis=(1, 3)))            # (block, slot) pairs written
    s0 = slots[0]
    assert changed.tolist() == [[s0 // B, s0 % B]], changed.tolist()
    np.testing.assert_array_equal(kb[s0 // B, :, s0 % B], to_bits(k_new[0]))
    assert (out[1] == 0).all()


def test_append_argument_errors():
    Hq, Hkv, D, B = 8, 2, 64, 16
    q, kc, vc, k_new, v_new, tab, ctx, slots = _problem(4, Hq, Hkv, D, B, [20])
    dev = "cuda"
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    with pytest.raises(ValueError):
        api.pa_decode_append(out, q.to(dev), kc.to(dev), vc.to(dev), k_new[:, :1].to(dev), v_new.to(dev),
                             torch.from_numpy(tab).to(dev), torch.from_numpy(ctx).to(dev), B, 0.125, Hq, Hkv, D, 20)
