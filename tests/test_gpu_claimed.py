"""GPU parity of the claimed decode schedule: a batch with many head groups
(at least two waves of resident blocks) and ragged lengths split into
partitions, where the resident blocks claim the (sequence, head group,
partition) items that exist instead of one block per possible partition.
Outputs match the oracle ("PagedAttention in vLLM: scattered memory, exact
attention", sections 10 and 11) within the decode tolerance, repeated calls
and CUDA-graph replays give the same bits (the claim counters are left at
zero), and the fused append gives the bits of the two separate calls."""
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

D, HQ, HKV, B = 128, 32, 8, 16
NAN16 = 0x7FC1


def _lens(S, seed):
    """Ragged contexts: lognormal around 200, clipped to [1, 2500], with a
    one-position context, a zero context and one of 2500 among them."""
    rng = np.random.default_rng(seed)
    lens = np.clip(np.round(200 * np.exp(rng.normal(size=S))), 1, 2500).astype(np.int32)
    lens[0], lens[1], lens[2] = 1, 0, 2500
    return lens


def _bf16_problem(lens, seed):
    rng = np.random.default_rng(seed)
    nblk = [max(1, -(-int(L) // B)) for L in lens]
    NB = sum(nblk) + 3
    perm = rng.permutation(NB)
    tables = np.full((len(lens), max(nblk)), -1, dtype=np.int32)
    pos = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[pos:pos + n]
        pos += n
    kc = to_bits(I.bf16_normal((NB, HKV, B, D), seed * 10 + 1))
    vc = to_bits(I.bf16_normal((NB, HKV, B, D), seed * 10 + 2))
    for s, L in enumerate(lens):                 # NaN in every slot past a context
        for i in range(int(L), nblk[s] * B):
            kc[tables[s, i // B], :, i % B] = NAN16
            vc[tables[s, i // B], :, i % B] = NAN16
    q = to_bits(I.bf16_normal((len(lens), HQ, D), seed * 10 + 3))
    return q, kc, vc, tables


def _units(fp8):
    return HKV // 2 if fp8 else HKV


def _claimed_regime(S, fp8):
    """The library claims work when the head groups fill two waves of resident blocks."""
    props = torch.cuda.get_device_properties(0)
    per_sm = 3
    return S * _units(fp8) >= 2 * per_sm * props.multi_processor_count


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_claimed_bf16_matches_oracle_and_repeats(out_dtype):
    S = 200
    assert _claimed_regime(S, False)
    lens = _lens(S, 1)
    q, kc, vc, tables = _bf16_problem(lens, 1)
    P, max_ctx = 512, int(lens.max())
    dev = lambda a: torch.from_numpy(a).cuda()
    out = torch.empty(S, HQ, D, dtype=out_dtype, device="cuda")
    ws = api.decode_workspace(S, HQ, D, max_ctx, P)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (from_bits(q), from_bits(kc), from_bits(vc), dev(tables), dev(lens), B, 1 / math.sqrt(D), HQ, HKV, D,
            max_ctx)
    api.pa_decode(out, *args, partition_size=P, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert not ws[:8].any().item()               # claim counters back at zero
    ref = A.paged_decode(q, kc, vc, tables, lens, 1 / math.sqrt(D), B)
    assert_attention_close(out_to_f64(out), ref, out_dtype == torch.float32, "claimed bf16 decode")
    first = out.clone()
    for _ in range(2):
        api.pa_decode(out, *args, partition_size=P, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert torch.equal(out, first)


def test_claimed_decode_in_a_cuda_graph():
    S = 200
    lens = _lens(S, 2)
    q, kc, vc, tables = _bf16_problem(lens, 2)
    P, max_ctx = 512, int(lens.max())
    dev = lambda a: torch.from_numpy(a).cuda()
    out = torch.empty(S, HQ, D, dtype=torch.bfloat16, device="cuda")
    ws = api.decode_workspace(S, HQ, D, max_ctx, P)
    args = (from_bits(q), from_bits(kc), from_bits(vc), dev(tables), dev(lens), B, 1 / math.sqrt(D), HQ, HKV, D,
            max_ctx)
    api.pa_decode(out, *args, partition_size=P, workspace=ws)
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            api.pa_decode(out, *args, partition_size=P, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)


def test_claimed_append_equals_the_two_calls():
    S = 200
    lens = _lens(S, 3)
    lens[1] = 5                                   # the fused append needs a position to append to
    q, kc, vc, tables = _bf16_problem(lens, 3)
    P, max_ctx = 512, int(lens.max())
    dev = lambda a: torch.from_numpy(a).cuda()
    k_new = I.bf16_normal((S, HKV, D), 31).cuda()
    v_new = I.bf16_normal((S, HKV, D), 32).cuda()
    slots = torch.tensor([int(tables[s, (L - 1) // B]) * B + (int(L) - 1) % B for s, L in enumerate(lens)],
                         dtype=torch.int64, device="cuda")
    common = (dev(tables), dev(lens), B, 1 / math.sqrt(D), HQ, HKV, D, max_ctx)
    qd = from_bits(q)
    kc1, vc1 = from_bits(kc), from_bits(vc)
    out1 = torch.empty(S, HQ, D, dtype=torch.bfloat16, device="cuda")
    ws = api.decode_workspace(S, HQ, D, max_ctx, P)
    api.pa_reshape_and_cache(kc1, vc1, k_new, v_new, slots)
    api.pa_decode(out1, qd, kc1, vc1, *common, partition_size=P, workspace=ws)
    kc2, vc2 = from_bits(kc), from_bits(vc)
    out2 = torch.empty_like(out1)
    api.pa_decode_append(out2, qd, kc2, vc2, k_new, v_new, *common, partition_size=P, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)
    bits = lambda t: t.view(torch.int16)             # the unused slots hold NaN patterns
    assert torch.equal(bits(kc1), bits(kc2)) and torch.equal(bits(vc1), bits(vc2))


def test_claimed_fp8_matches_oracle():
    """E4M3 codes drawn directly (no NaN code in a context; NaN codes past
    every context); 30 sequences compared with the oracle over the
    dequantised values of their blocks."""
    S = 240
    assert _claimed_regime(S, True)
    lens = _lens(S, 4)
    lens[1] = 7
    k_scale, v_scale = 0.01, 0.02
    rng = np.random.default_rng(4)
    nblk = [-(-int(c) // B) for c in lens]
    NB = sum(nblk) + 3
    perm = I.permutation(NB, 4)
    tables = np.full((S, max(nblk)), -1, dtype=np.int32)
    codes = lambda: (rng.integers(0, 0x60, size=(NB, HKV, B, D)) | (rng.integers(0, 2, size=(NB, HKV, B, D)) << 7))
    kc, vc = codes().astype(np.uint8), codes().astype(np.uint8)
    pos = 0
    for s, c in enumerate(lens):
        for lb in range(nblk[s]):
            tables[s, lb] = int(perm[pos])
            pos += 1
        for i in range(int(c), nblk[s] * B):     # NaN codes past the context
            kc[tables[s, i // B], :, i % B] = Q.NAN_CODE
            vc[tables[s, i // B], :, i % B] = Q.NAN_CODE
    q = to_bits(I.bf16_normal((S, HQ, D), 43))
    P, max_ctx = 512, int(lens.max())
    dev = lambda a: torch.from_numpy(a).cuda()
    out = torch.empty(S, HQ, D, dtype=torch.float32, device="cuda")
    ws = api.decode_workspace(S, HQ, D, max_ctx, P)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_decode_fp8(out, from_bits(q), dev(kc), dev(vc), dev(tables), dev(lens), B, 1 / math.sqrt(D), k_scale,
                      v_scale, HQ, HKV, D, max_ctx, partition_size=P, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert not ws[:8].any().item()
    got = out_to_f64(out)
    sample = [0, 1, 2] + sorted(rng.choice(np.arange(3, S), size=27, replace=False).tolist())
    for s in sample:
        blocks = tables[s, :max(1, nblk[s])]
        kd = Q.dequantize(kc[blocks], k_scale)
        vd = Q.dequantize(vc[blocks], v_scale)
        ref = A.paged_decode(q[s:s + 1], kd, vd, np.arange(len(blocks))[None, :], lens[s:s + 1],
                             1 / math.sqrt(D), B)
        assert_attention_close(got[s:s + 1], ref, True, "claimed fp8 decode, sequence %d" % s)
