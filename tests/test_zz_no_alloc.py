"""pa_decode_static_scratch: the decode entry point for callers that cannot
give the library device memory (code running where cudaMalloc is not allowed
or not wanted, or a host framework that owns every device allocation).  It
must give bit-for-bit the results of pa_decode with a caller workspace and
the same partition size (both run the same kernels; only the scratch address
differs), on two calls in a row (the second call finds the first call's
leftovers in the shared static array), allocate no device memory while it
runs, and refuse problems larger than its fixed scratch.

Kept in a file that pytest collects last, so that a run stopping at the first
failure has already run every other test."""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

api = pytest.importorskip("paged_kv_cache_124_gb300.api")


def _problem(seed, lens, Hq=32, Hkv=8, D=128, B=16):
    rng = np.random.default_rng(seed)
    nblk = [-(-L // B) for L in lens]
    NB = sum(nblk) + 3
    perm = rng.permutation(NB)
    tables = np.full((len(lens), max(nblk)), -1, dtype=np.int32)
    pos = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[pos:pos + n]
        pos += n
    bits = lambda shape: torch.from_numpy(rng.standard_normal(size=shape).astype(np.float32)).to(torch.bfloat16)
    kc, vc = bits((NB, Hkv, B, D)).cuda(), bits((NB, Hkv, B, D)).cuda()
    q = bits((len(lens), Hq, D)).cuda()
    return q, kc, vc, torch.from_numpy(tables).cuda(), torch.tensor(lens, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_static_scratch_matches_workspace_decode_twice(out_dtype):
    Hq, Hkv, D, B, P = 32, 8, 128, 16, 256
    for call, (seed, lens) in enumerate([(1, [1000, 300, 2048, 17]), (2, [2048, 5, 999, 1500])]):
        q, kc, vc, tab, ctx = _problem(seed, lens, Hq, Hkv, D, B)
        max_ctx = 2048
        scale = 1.0 / math.sqrt(D)
        ref = torch.empty(q.shape, dtype=out_dtype, device="cuda")
        ws = api.decode_workspace(len(lens), Hq, D, max_ctx, P)
        assert ws is not None                                   # the split path is exercised
        api.pa_decode(ref, q, kc, vc, tab, ctx, B, scale, Hq, Hkv, D, max_ctx, partition_size=P, workspace=ws)
        got = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        allocs = torch.cuda.memory_stats()["allocation.all.allocated"]
        free_before = torch.cuda.mem_get_info()[0]
        api.pa_decode_static_scratch(got, q, kc, vc, tab, ctx, B, scale, Hq, Hkv, D, max_ctx, partition_size=P,
                                     status=st)
        torch.cuda.synchronize()
        # no device allocation, through PyTorch's allocator or around it
        assert torch.cuda.memory_stats()["allocation.all.allocated"] == allocs
        assert torch.cuda.mem_get_info()[0] == free_before
        assert st.item() == 0
        assert torch.equal(got, ref), "static scratch call %d differs from pa_decode" % call


def test_static_scratch_refuses_problems_larger_than_its_array():
    Hq, Hkv, D, B = 32, 8, 128, 16
    q, kc, vc, tab, ctx = _problem(3, [64], Hq, Hkv, D, B)
    max_ctx, P, S = 8192, 64, 1100    # 1100 x 32 heads x 128 partitions of statistics: far above the array
    need = api.pa_decode_workspace_size(S, Hq, D, max_ctx, P)
    assert need > api.PA_STATIC_SCRATCH_BYTES
    qS = q.expand(S, -1, -1).contiguous()
    out = torch.empty_like(qS)
    tabS = tab.expand(S, -1).contiguous()
    ctxS = ctx.expand(S).contiguous()
    with pytest.raises(api.PAError) as e:
        api.pa_decode_static_scratch(out, qS, kc, vc, tabS, ctxS, B, 0.1, Hq, Hkv, D, max_ctx, partition_size=P)
    assert e.value.status == api.PA_ERR_WORKSPACE
