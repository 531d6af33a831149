"""End-to-end parity on the five workloads: the same scenario is replayed by
the CUDA path (C++ block manager + kernels, through the C ABI) and by the
oracle (reference allocator + oracle cache ops); pools must agree bit for
bit, block tables exactly, and decode outputs within tolerance."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from _gpu_util import assert_attention_close, out_to_f64, to_bits
from _oracle_replay import OracleReplay

pytestmark = pytest.mark.gpu

api = pytest.importorskip("paged_kv_cache_124_gb300.api")
from paged_kv_cache_124_gb300 import inputs as I  # noqa: E402
from paged_kv_cache_124_gb300.runner import ScenarioRunner  # noqa: E402


def _decode(run, layer, out_dtype, partition=0):
    sc = run.sc
    tables, ctx, max_ctx = run.decode_metadata()
    q = I.decode_q(sc.seed, layer, len(sc.decode_seqs), sc.n_q_heads, sc.d_head).cuda()
    out = torch.empty(q.shape, dtype=out_dtype, device="cuda")
    ws = api.decode_workspace(q.shape[0], sc.n_q_heads, sc.d_head, max_ctx, partition)
    api.pa_decode(out, q, run.k_caches[layer], run.v_caches[layer], tables, ctx, sc.block_size, sc.scale,
                  sc.n_q_heads, sc.n_kv_heads, sc.d_head, max_ctx, partition_size=partition, workspace=ws,
                  status=run.status)
    torch.cuda.synchronize()
    return out


def _check_scenario(sc, layers_checked=None, data_device="cpu", partitions=(0,), decode_all_layers=False):
    run = ScenarioRunner(sc, data_device=data_device).replay()
    torch.cuda.synchronize()
    layers = list(range(sc.n_layers)) if layers_checked is None else layers_checked
    data_fn = None
    if data_device != "cpu":
        def data_fn(kind, layer, index, n):
            fn = I.prefill_kv if kind == "prefill" else I.append_kv
            k, v = fn(sc.seed, layer, index, n, sc.n_kv_heads, sc.d_head, data_device)
            return to_bits(k), to_bits(v)
    ref = OracleReplay(sc, layers, data_fn).replay()
    # block tables and lengths
    tab_ref, len_ref = ref.tables()
    tables, ctx, _ = run.decode_metadata()
    assert np.array_equal(tables.cpu().numpy()[:, :tab_ref.shape[1]], tab_ref)
    assert np.array_equal(ctx.cpu().numpy(), len_ref)
    assert run.cow_pairs_total == len(ref.cow_pairs)
    # pools, bit for bit
    for l in layers:
        assert np.array_equal(to_bits(run.k_caches[l]), ref.k[l]), "K pool layer %d" % l
        assert np.array_equal(to_bits(run.v_caches[l]), ref.v[l]), "V pool layer %d" % l
    # decode
    errs = []
    for l in layers:
        q_bits = to_bits(I.decode_q(sc.seed, l, len(sc.decode_seqs), sc.n_q_heads, sc.d_head))
        want = A.paged_decode(q_bits, ref.k[l], ref.v[l], tab_ref, len_ref, sc.scale, sc.block_size)
        for P in partitions:
            for dt in (torch.float32, torch.bfloat16):
                got = _decode(run, l, dt, P)
                errs.append(assert_attention_close(out_to_f64(got), want, dt == torch.float32,
                                                   "%s layer %d P=%d %s" % (sc.name, l, P, dt)))
    if decode_all_layers:
        for l in range(sc.n_layers):
            got = _decode(run, l, torch.bfloat16)
            assert torch.isfinite(got.float()).all()
    assert run.status.item() == 0
    return run, ref, errs


@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4])
def test_tiny_gqa(seed):
    sc = I.tiny_gqa(seed)
    run, ref, _ = _check_scenario(sc, partitions=(0, 64))
    assert run.alloc.build_tables(sc.decode_seqs, 3)[1].tolist() == [2, 16, 17, 38]


@pytest.mark.parametrize("seed", [0, 1])
def test_batch64_8b(seed):
    _check_scenario(I.batch64_8b(seed), partitions=(0, 256))


@pytest.mark.parametrize("B", [16, 32])
def test_long_context_split(B):
    _check_scenario(I.long_context(0, B), partitions=(0, 4096))


def test_cow_parallel_sampling():
    sc = I.cow_sampling(0)
    run, ref, _ = _check_scenario(sc)
    # reading of the trace: the first 7 writers of every 8-way shared tail copy it
    assert run.cow_pairs_total == 16 * 7
    # siblings share every full prompt block and differ from the tail on
    tab, _ = ref.tables()
    full = 2003 // 16
    for p in range(16):
        fam = tab[p * 8:(p + 1) * 8]
        assert (fam[:, :full] == fam[0, :full]).all()
        assert len(set(fam[:, full].tolist())) == 8


@pytest.mark.parametrize("B", [8, 16, 32])
def test_mixed_continuous_batching_32_layers(B):
    sc = I.mixed_batch(0, B)
    run, _, _ = _check_scenario(sc, layers_checked=[0, sc.n_layers - 1], data_device="cuda",
                                decode_all_layers=True)
    st = run.alloc.stats()
    assert st["num_used"] >= 0.85 * sc.num_blocks


def test_fork_siblings_decode_identically_on_shared_prefix():
    """Identical outputs across CoW forks: a parent and its forks decoded
    before they diverge see the same cache and give the same bits."""
    sc = dataclasses.replace(I.cow_sampling(3, n_prompts=2, prompt_len=301, n_samples=4, max_new=1),
                             decode_seqs=list(range(8)))
    sc.ops = [op for op in sc.ops if op[0] not in ("append",)]
    run = ScenarioRunner(sc).replay()
    tables, ctx, max_ctx = run.decode_metadata()
    q1 = I.decode_q(5, 0, 1, sc.n_q_heads, sc.d_head).cuda()
    q = q1.expand(8, -1, -1).contiguous()
    out = torch.empty_like(q, dtype=torch.float32)
    ws = api.decode_workspace(8, sc.n_q_heads, sc.d_head, max_ctx)
    api.pa_decode(out, q, run.k_caches[0], run.v_caches[0], tables, ctx, sc.block_size, sc.scale,
                  sc.n_q_heads, sc.n_kv_heads, sc.d_head, max_ctx, workspace=ws)
    torch.cuda.synchronize()
    o = out.cpu()
    for p in range(2):
        for j in range(1, 4):
            assert torch.equal(o[p * 4 + j], o[p * 4])
    assert not torch.equal(o[0], o[4])
