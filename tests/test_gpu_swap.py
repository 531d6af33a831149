"""GPU parity of swapping ("PagedAttention: Virtual Memory for the KV Cache",
section 19, items 3 and 4): pa_swap_blocks moves blocks between device pools
and page-locked host pools bit for bit like the oracle's swap_blocks; a batch
swapped out, its device blocks reused by others, and swapped back in decodes
exactly as before; a request preempted by recomputation (freed, then
re-admitted through the prefix cache) decodes exactly as before."""
import math

import numpy as np
import pytest
import torch

from oracle import cache_ops as C
from _gpu_util import to_bits

pytestmark = pytest.mark.gpu

api = pytest.importorskip("paged_kv_cache_124_gb300.api")
from paged_kv_cache_124_gb300 import inputs as I  # noqa: E402

HQ, HKV, D, B = 32, 8, 128, 16


def _pools(n_layers, nb, device, pinned=False, seed=0):
    shape = (nb, HKV, B, D)
    out = []
    for l in range(n_layers):
        k = I.bf16_normal(shape, seed * 100 + 2 * l)
        v = I.bf16_normal(shape, seed * 100 + 2 * l + 1)
        if device == "cuda":
            k, v = k.cuda(), v.cuda()
        elif pinned:
            k, v = k.pin_memory(), v.pin_memory()
        out.append((k, v))
    return [p[0] for p in out], [p[1] for p in out]


@pytest.mark.parametrize("pairs_on_host", [False, True])
def test_swap_blocks_round_trip_bit_exact(pairs_on_host):
    L, NB, NH = 3, 40, 24
    dk, dv = _pools(L, NB, "cuda", seed=1)
    hk, hv = _pools(L, NH, "cpu", pinned=True, seed=2)
    rng = np.random.default_rng(0)
    out_pairs = np.stack([rng.permutation(NB)[:17], rng.permutation(NH)[:17]], 1).astype(np.int32)
    # oracle on host copies
    ref_hk = [to_bits(t).copy() for t in hk]
    ref_hv = [to_bits(t).copy() for t in hv]
    for l in range(L):
        C.swap_blocks(ref_hk[l], ref_hv[l], to_bits(dk[l]), to_bits(dv[l]), out_pairs.tolist())
    p = torch.from_numpy(out_pairs)
    p = p.pin_memory() if pairs_on_host else p.cuda()
    api.pa_swap_blocks(hk, hv, dk, dv, p)
    torch.cuda.synchronize()
    for l in range(L):
        assert np.array_equal(to_bits(hk[l]), ref_hk[l]) and np.array_equal(to_bits(hv[l]), ref_hv[l])
    # and back into other device blocks
    back = np.stack([out_pairs[:, 1], rng.permutation(NB)[:17]], 1).astype(np.int32)
    ref_dk = [to_bits(t).copy() for t in dk]
    ref_dv = [to_bits(t).copy() for t in dv]
    for l in range(L):
        C.swap_blocks(ref_dk[l], ref_dv[l], ref_hk[l], ref_hv[l], back.tolist())
    api.pa_swap_blocks(dk, dv, hk, hv, torch.from_numpy(back).cuda())
    torch.cuda.synchronize()
    for l in range(L):
        assert np.array_equal(to_bits(dk[l]), ref_dk[l]) and np.array_equal(to_bits(dv[l]), ref_dv[l])


def test_swap_blocks_flags_and_rejects():
    dk, dv = _pools(1, 8, "cuda")
    hk, hv = _pools(1, 4, "cpu", pinned=True)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_swap_blocks(hk, hv, dk, dv, torch.tensor([[0, 9], [1, 1]], dtype=torch.int32, device="cuda"), status=st)
    torch.cuda.synchronize()
    assert st.item() & api.PA_DEV_BAD_BLOCK_ID
    with pytest.raises(ValueError):                   # pageable host memory
        api.pa_swap_blocks([torch.zeros_like(hk[0], device="cpu")], [hv[0]], dk, dv,
                           torch.tensor([[0, 0]], dtype=torch.int32, device="cuda"))


def _decode(alloc, seqs, k, v, q, max_ctx):
    tables, ctx = alloc.build_tables(seqs, max(len(alloc.block_table(s)) for s in seqs))
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = api.decode_workspace(len(seqs), HQ, D, max_ctx)
    api.pa_decode(out, q, k, v, torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda(), B, 1 / math.sqrt(D),
                  HQ, HKV, D, max_ctx, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu()


def _write(alloc, seq, toks, start, k, v, seed):
    n = len(toks) - start
    slots = torch.from_numpy(alloc.slot_mapping(seq, start, n)).cuda()
    kk, vv = I.prefix_kv(seed, 0, toks, start, len(toks), HKV, D)
    api.pa_reshape_and_cache(k, v, kk.cuda(), vv.cuda(), slots)


def test_preemption_by_swapping_then_by_recompute():
    NB, NH, seed = 120, 80, 11
    alloc = api.BlockAllocator(NB, B)
    assert alloc.enable_prefix_caching(True) == 0 and alloc.enable_swap(NH) == 0
    k = I.nan_pool((NB, HKV, B, D)).cuda()
    v = I.nan_pool((NB, HKV, B, D)).cuda()
    hk = I.nan_pool((NH, HKV, B, D)).pin_memory()
    hv = I.nan_pool((NH, HKV, B, D)).pin_memory()
    docs = I.prompt_documents(seed, [400, 650])
    toks = {}
    for s in range(4):
        toks[s] = docs[s % 2] + [int(t) for t in np.random.default_rng(s).integers(0, 32000, size=20 + 7 * s)]
        st, hit = alloc.allocate_tokens(s, toks[s])
        assert st == 0
        _write(alloc, s, toks[s], hit, k, v, seed)
    q = I.decode_q(seed, 0, 4, HQ, D).cuda()
    max_ctx = 1024
    before = _decode(alloc, [0, 1, 2, 3], k, v, q, max_ctx)

    # swap out sequences 1 and 3 (they share document 1's blocks), let others take the freed blocks
    st, pairs = alloc.swap_out([1, 3])
    assert st == 0 and len(pairs) > 0
    api.pa_swap_blocks([hk], [hv], [k], [v], torch.from_numpy(pairs).cuda())
    # more than the free list holds, so some of the swapped sequences' cached blocks are evicted too
    n_fill = alloc.num_free() + min(20, alloc.num_cached())
    filler = [int(t) for t in np.random.default_rng(99).integers(0, 32000, size=n_fill * B)]
    assert alloc.allocate_tokens(10, filler)[0] == 0
    _write(alloc, 10, filler, 0, k, v, seed + 1)             # overwrites blocks the swapped sequences left
    assert alloc.free(10) == 0
    st, pairs = alloc.swap_in([1, 3])
    assert st == 0
    api.pa_swap_blocks([k], [v], [hk], [hv], torch.from_numpy(pairs).cuda())
    after_swap = _decode(alloc, [0, 1, 2, 3], k, v, q, max_ctx)
    assert torch.equal(after_swap, before)

    # preempt sequence 2 by recomputation: free it, re-admit the same tokens,
    # recompute only what the prefix cache no longer holds
    assert alloc.free(2) == 0
    st, hit = alloc.allocate_tokens(2, toks[2])
    assert st == 0 and hit >= len(docs[0]) // B * B
    _write(alloc, 2, toks[2], hit, k, v, seed)
    after_recompute = _decode(alloc, [0, 1, 2, 3], k, v, q, max_ctx)
    assert torch.equal(after_recompute, before)
