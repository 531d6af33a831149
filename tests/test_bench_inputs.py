"""Host-side inputs and work counts of the bench workloads.  The FLOP and
byte counts behind the roofline figures are recounted term by term from the
workloads' drawn sizes.  The
copy-on-write pairs of the CoW sampling config (16 prompts of 2,003 tokens,
8 samples each, one appended token per sample) that the cache-ops workload
copies come from the C++ block manager; the oracle allocator replaying the
same operations must plan the same pairs, and their number follows from the
pages' rule that each writer of a shared tail block copies it except the
last ("PagedAttention: Virtual Memory for the KV Cache", sections 15-16).
The continuous-batching workload's lengths follow its stated recipe."""
import math

import numpy as np
import pytest

api = pytest.importorskip("paged_kv_cache_124_gb300.api")

import bench  # noqa: E402
from oracle.allocator import RefAllocator  # noqa: E402
from paged_kv_cache_124_gb300 import inputs as I  # noqa: E402


def test_cow_pairs_match_the_oracle_allocator():
    sc, slots, pairs, nb = bench._cache_ops_inputs(0, 16, api)
    n_prompts, samples = len(sc.ctxs), 8
    ref = RefAllocator(nb, sc.block_size)
    assert ref.set_free_order(list(sc.free_order) + list(range(sc.num_blocks, nb))) == 0
    for s, c in enumerate(sc.ctxs):
        assert ref.allocate(s * samples, c) == 0
        for f in range(1, samples):
            assert ref.fork(s * samples, s * samples + f) == 0
    want = []
    for s in range(n_prompts * samples):
        st, _, src, dst = ref.append_slot(s)
        assert st == 0
        if src >= 0:
            want.append((src, dst))
    assert pairs.tolist() == [list(p) for p in want]
    # 2,003 = 125 * 16 + 3: the tail block is shared by 8 samples; the first 7
    # writers copy it, the 8th writes in place
    assert len(pairs) == n_prompts * (samples - 1) == 112
    srcs = pairs[:, 0].tolist()
    assert len(set(srcs)) == n_prompts and all(srcs.count(x) == samples - 1 for x in set(srcs))
    assert len(set(pairs[:, 1].tolist())) == len(pairs)             # fresh destinations
    assert not set(pairs[:, 1].tolist()) & set(srcs)


def test_prefill_slots_are_the_new_positions_of_each_prompt():
    sc, slots, _, _ = bench._cache_ops_inputs(0, 16, api)
    assert len(slots) == sum(sc.news) == 16 * 2003
    assert len(set(slots.tolist())) == len(slots)                   # one slot per position
    assert slots.min() >= 0 and slots.max() < sc.num_blocks * sc.block_size


def test_prefill_flops_closed_form_and_pair_count():
    """The prefill roofline's numerator: 4 d FLOPs per (query head, visible
    key) pair.  Whole prompts see p + 1 keys at position p, n (n + 1) / 2
    pairs per head; a chunk over a cached prefix is counted pair by pair."""
    assert bench.prefill_flops([2003] * 16, [2003] * 16, 32, 128) == 16 * (2003 * 2004 // 2) * 4 * 128 * 32
    ctxs, news = [10, 7, 1, 300], [4, 7, 1, 17]
    pairs = sum(1 for c, n in zip(ctxs, news) for p in range(c - n, c) for j in range(c) if j <= p)
    assert bench.prefill_flops(ctxs, news, 3, 64) == pairs * 4 * 64 * 3


def test_decode_algorithmic_bytes_of_the_headline_batch():
    """The decode roofline's numerator for the 64-sequence 8B-shaped batch,
    counted term by term from its drawn contexts: one K and one V row of
    d_head bf16 values per cached position and KV head, q read and the
    output written once, and the 4-byte table entries and context lengths in
    use; the cache write reads and writes each new token's K and V rows."""
    from paged_kv_cache_124_gb300 import inputs as I
    sc = I.batch64_8b(0)
    ctx = np.asarray(I.uniform_ints(64, 512, 4096, 1), dtype=np.int64)
    assert int(ctx.sum()) == 143905
    kv = sum(int(c) * sc.d_head * 2 * 2 for c in ctx for _ in range(sc.n_kv_heads))
    qo = 64 * sc.n_q_heads * sc.d_head * 2 * 2
    tab = sum((int(c) + sc.block_size - 1) // sc.block_size for c in ctx) * 4 + 64 * 4
    dec, write = bench.algorithmic_bytes(sc, ctx, 64)
    assert dec == kv + qo + tab == 590519796
    assert write == 64 * sc.n_kv_heads * 2 * sc.d_head * 2 * 2


def test_cpu_baseline_runs_the_oracle_on_every_core_and_on_one():
    """The all-core leg starts one worker process per host core on a
    compacted copy of the sample; both legs report positive rates and the
    all-core leg says how many cores it used."""
    from paged_kv_cache_124_gb300 import inputs as I
    sc = I.tiny_gqa(0)
    line = bench.cpu_baseline(sc, 0.2)
    assert line["kind"] == "oracle" and line["value"] > 0
    assert "all_cores_failed" not in line, line.get("all_cores_failed")
    if bench.host_threads() > 1:
        assert line["cores"] == bench.host_threads()
        assert line["single_thread"]["cores"] == 1 and line["single_thread"]["value"] > 0


def test_worker_pool_time_is_the_slowest_worker():
    from paged_kv_cache_124_gb300 import inputs as I
    sc = I.tiny_gqa(0)
    rep, tab, lens, q = bench._oracle_sample(sc, list(range(len(sc.decode_seqs))))
    t = bench._oracle_time_procs(sc, rep, tab, lens, q, 2, 3)
    assert 0 < t < 60


def _small_prefill():
    from types import SimpleNamespace
    return SimpleNamespace(name="small_prefill", ctxs=[300, 200], news=[300, 64], block_size=16, n_kv_heads=2,
                           n_q_heads=8, d_head=64, scale=0.125)


def test_prefill_worker_pool_time_is_the_slowest_worker():
    """Each worker takes a contiguous share of the sampled rows as one chunk
    at their positions (chunking leaves the oracle's output unchanged: pinned
    in the oracle's prefill tests)."""
    t = bench._prefill_oracle_time_procs(_small_prefill(), 40, 2, 2)
    assert 0 < t < 60


def test_prefill_cpu_baseline_reports_both_legs():
    line = bench.prefill_cpu_baseline(_small_prefill(), 0.2)
    assert line["kind"] == "oracle" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert "all_cores_failed" not in line, line.get("all_cores_failed")
    if bench.host_threads() > 1:
        assert line["cores"] == bench.host_threads()
        assert line["single_thread"]["cores"] == 1 and line["single_thread"]["value"] > 0


def test_quantiles():
    assert bench._quantiles([5.0, 1.0, 3.0, 2.0, 4.0]) == (3.0, 1.0, 5.0)
    assert bench._quantiles([2.0]) == (2.0, 2.0, 2.0)


def test_lognormal_lengths_have_the_requested_median_and_sigma():
    """The continuous-batching lengths: lognormal with median 700 and
    log-space sigma 1 (reading O11), rounded and clipped."""
    x = I.lognormal_ints(200000, 700, 1.0, 1, 10 ** 9, 5)
    assert abs(np.median(x) / 700 - 1) < 0.01
    assert abs(np.std(np.log(x)) - 1.0) < 0.01
    y = I.lognormal_ints(5000, 700, 1.0, 1, 16384, 6)
    assert y.min() >= 1 and y.max() <= 16384 and (y == 16384).any()


def test_mixed_batch_recipe():
    """256 sequences whose decode contexts are the lognormal draw (each a
    prompt of ctx - 1 tokens and one appended token), the 8B head shape, 32
    layers, and a pool sized for 90 % occupancy."""
    sc = I.mixed_batch(0, 16)
    ctx = I.lognormal_ints(256, 700, 1.0, 1, 16384, 1)
    toks = {}
    for op in sc.ops:
        if op[0] == "alloc" and op[1] < 256:
            toks[op[1]] = op[2]
        elif op[0] == "append":
            toks[op[1]] += 1
    assert [toks[i] for i in range(256)] == ctx.tolist()
    assert sc.decode_seqs == list(range(256))
    assert (sc.n_q_heads, sc.n_kv_heads, sc.d_head, sc.n_layers) == (32, 8, 128, 32)
    need = sum(-(-int(c) // 16) for c in ctx)
    assert sc.num_blocks == math.ceil(need / 0.9)


def test_profiled_traffic_needs_both_source_hashes():
    """A committed ncu traffic figure is reported only while both the kernel's
    source and the device helpers it includes hash as they did at capture;
    either one changed gives no traffic (null in the bench line)."""
    other = bench.PREFILL_SOURCE                                       # any file with another hash
    assert bench.profiled_traffic(bench.PROFILE_SUMMARY, other) is None
    assert bench.profiled_traffic(bench.PROFILE_SUMMARY, bench.KERNEL_SOURCE, other) is None
    text = open(bench.PROFILE_SUMMARY).read()
    assert "common_header_sha256_16:" in text and "kernel_source_sha256_16:" in text


def test_seeded_draws_are_reproducible_and_leave_the_global_generators_alone():
    """Both sides of every comparison draw their inputs from these generators,
    so a draw must depend on its seed only: the same seed gives the same bits
    whatever was drawn before, another seed other bits, and the global torch
    and NumPy generators are neither read nor advanced."""
    import torch
    torch.manual_seed(123)
    np.random.seed(123)
    want_torch = torch.rand(4)
    want_np = np.random.rand(4)
    torch.manual_seed(123)
    np.random.seed(123)
    a = I.bf16_bits(I.bf16_normal((3, 5, 7), 42))
    k1, v1 = I.prefill_kv(0, 1, 2, 9, 2, 8)
    p1 = I.permutation(50, 7)
    n1 = I.lognormal_ints(20, 700, 1.0, 1, 16384, 3)
    assert torch.equal(torch.rand(4), want_torch) and np.array_equal(np.random.rand(4), want_np)
    torch.rand(1000)                                  # the global state moves; the draws must not
    assert np.array_equal(I.bf16_bits(I.bf16_normal((3, 5, 7), 42)), a)
    k2, v2 = I.prefill_kv(0, 1, 2, 9, 2, 8)
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16)) and torch.equal(v1.view(torch.int16),
                                                                                  v2.view(torch.int16))
    assert np.array_equal(I.permutation(50, 7), p1) and np.array_equal(I.lognormal_ints(20, 700, 1.0, 1, 16384, 3), n1)
    assert not np.array_equal(I.bf16_bits(I.bf16_normal((3, 5, 7), 43)), a)
    assert not torch.equal(I.prefill_kv(0, 1, 3, 9, 2, 8)[0].view(torch.int16), k1.view(torch.int16))
    assert not torch.equal(k1.view(torch.int16), v1.view(torch.int16))   # keys and values are separate draws
