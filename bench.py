#!/usr/bin/env python3
"""Benchmark of the paged decode-attention path on one GB300 (or N replicas).

One step = one decode step of the 8B-shaped batch: pa_reshape_and_cache of
the step's new token for every sequence, then pa_decode (partition kernel +
log-sum-exp merge kernel) over the whole batch.  Inputs are resident in HBM;
the KV bytes a step reads (about 604 MB) exceed the 129 MB L2, so no flush
is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --workload prefill_prompts_8b|chunked_prefill_8b   (prefill path)

Prints one JSON line.  The value is decode KV GB/s: the algorithmic bytes of
a step (every cached K/V row read once, q, out, block tables, context
lengths, and the new rows read and written) divided by the step time.
--impl reference times the CPU oracle on a bounded sample of the same
workload instead.
"""
import os

# The oracle's NumPy work runs BLAS on one thread per process (the all-core
# CPU leg starts one worker process per core); fix BLAS threads before NumPy
# loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import dataclasses  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import re  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_124_gb300 import inputs as I  # noqa: E402

METRIC = "paged decode-attn KV GB/s (frac of HBM peak); seqs/s at 8B GQA shape"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_partition_kernel_batch64_8b.md")
PROFILE_SUMMARY_FP8 = os.path.join(ROOT, "profiles", "decode_partition_kernel_fp8_batch64_8b.md")
KERNEL_SOURCE = os.path.join(ROOT, "paged_kv_cache_124_gb300", "csrc", "pa_decode.cu")
COMMON_HEADER = os.path.join(ROOT, "paged_kv_cache_124_gb300", "csrc", "pa_common.cuh")
PREFILL_PROFILE = os.path.join(ROOT, "profiles", "prefill_kernel_prefill_prompts_8b.md")
CACHE_OPS_PROFILE = os.path.join(ROOT, "profiles", "copy_blocks_kernel_cache_ops_8b.md")
CACHE_OPS_SOURCE = os.path.join(ROOT, "paged_kv_cache_124_gb300", "csrc", "pa_cache_ops.cu")
PREFILL_SOURCE = os.path.join(ROOT, "paged_kv_cache_124_gb300", "csrc", "pa_prefill.cu")

# NVTX range around each arm's K timed steps (an ncu launch list can be
# limited to it with --nvtx --nvtx-include "timed_steps/")
TIMED_RANGE = "timed_steps"

PREFILL_METRIC = "paged prefill-attn TFLOP/s (causal, 8B GQA shape; frac of bf16 tensor peak)"
PREFILL_WORKLOADS = {
    "prefill_prompts_8b": lambda seed, B: I.prefill_prompts(seed, B),
    "chunked_prefill_8b": lambda seed, B: I.chunked_prefill(seed, B),
}

WORKLOADS = {
    "batch64_8b": lambda seed, B, L: I.batch64_8b(seed, B),
    "long_context": lambda seed, B, L: I.long_context(seed, B),
    "cow_sampling": lambda seed, B, L: I.cow_sampling(seed, block_size=B),
    "mixed_batch": lambda seed, B, L: I.mixed_batch(seed, B, n_layers=L),
    "tiny_gqa": lambda seed, B, L: I.tiny_gqa(seed),
}


def workload_scenario(args, seed):
    """The decode workload's scenario; the continuous-batching step runs
    every one of its 32 layers unless --layers says otherwise."""
    layers = args.layers or 32
    return WORKLOADS[args.workload](seed, args.block_size, layers)


# ----------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no collective on the data path)
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def reduce_timing(elapsed_s, units, world, device="cpu"):
    """Max of the elapsed times and sum of the units over all ranks: the
    whole job runs as long as its slowest replica."""
    if world == 1:
        return float(elapsed_s), float(units)
    t = torch.tensor([float(elapsed_s)], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def replica_seed(base_seed, rank):
    """Each replica decodes its own batch (weak scaling)."""
    return int(base_seed) + 1000 * int(rank)


# ----------------------------------------------------------------------------
# byte accounting
# ----------------------------------------------------------------------------

def algorithmic_bytes(sc, ctx, n_new_tokens, kv_bytes=2):
    """Bytes one step must move at minimum: decode reads each cached K and V
    row of each KV head once, q, the block-table entries in use and the
    context lengths, and writes out; reshape_and_cache reads and writes each
    new token's K and V rows.  kv_bytes: bytes per cached element (2 for
    bf16, 1 for FP8)."""
    ctx = np.asarray(ctx, dtype=np.int64)
    row = sc.d_head * 2
    kv = int(ctx.sum()) * sc.n_kv_heads * sc.d_head * kv_bytes * 2
    S = len(ctx)
    qo = 2 * S * sc.n_q_heads * row
    tables = int((-(-ctx // sc.block_size)).sum()) * 4 + S * 4
    decode = kv + qo + tables
    cache_write = 2 * n_new_tokens * sc.n_kv_heads * (row + sc.d_head * kv_bytes)
    return decode, cache_write


def measured_peak(key="hbm_gbs", fallback=FALLBACK_HBM_GBS):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)[key]), "measured"
    except Exception:
        return fallback, "fallback"


def prefill_flops(ctxs, news, n_q_heads, d_head):
    """Algorithmic FLOPs of causal prefill attention: new position p of a
    sequence scores p + 1 keys and sums p + 1 value rows, 2 * d_head FLOPs
    each, for every query head.  Masked work is not counted."""
    f = 0.0
    for c, n in zip(ctxs, news):
        p = np.arange(c - n, c, dtype=np.float64)
        f += float((p + 1).sum()) * 4 * d_head * n_q_heads
    return f


def _sha16(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def profiled_traffic(summary=PROFILE_SUMMARY, source=KERNEL_SOURCE, common=COMMON_HEADER):
    """DRAM bytes per launch of a kernel from its committed ncu summary, if
    the summary was taken on the current kernel source and the current
    device helpers it includes; else None."""
    try:
        text = open(summary).read()
        m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
        m_common = re.search(r"common_header_sha256_16:\s*([0-9a-f]+)", text)
        m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
        if (m_hash and m_common and m_tr and m_hash.group(1) == _sha16(source) and
                m_common.group(1) == _sha16(common)):
            return int(m_tr.group(1))
    except OSError:
        pass
    return None


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = []

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "100"] + self.sel, stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        text = open(self.path).read()
        os.unlink(self.path)
        return summarize_clocks(text)


def summarize_clocks(text):
    """Median SM clock, the highest maximum clock and the throttle reasons
    seen Active, from nvidia-smi rows of ClockSampler.FIELDS (csv, no header,
    no units); rows that do not parse are skipped.  None without a sample."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.strip().splitlines():
        r = [x.strip() for x in line.split(",")]
        if len(r) < 9:
            continue
        try:
            clk, clk_max = float(r[1]), float(r[2])
        except ValueError:
            continue
        sm.append(clk)
        mx.append(clk_max)
        for n, val in zip(names, r[5:9]):
            if val.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
            "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# our implementation
# ----------------------------------------------------------------------------

def _quantiles(xs):
    xs = sorted(xs)
    pick = lambda f: xs[min(len(xs) - 1, max(0, int(round(f * (len(xs) - 1)))))]
    return statistics.median(xs), pick(0.1), pick(0.9)


def run_ours(args, world, rank, local):
    from paged_kv_cache_124_gb300 import api
    from paged_kv_cache_124_gb300.runner import ScenarioRunner

    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    seed = replica_seed(args.seed, rank)
    sc = workload_scenario(args, seed)
    L = sc.n_layers
    # token data on the GPU generator for multi-layer workloads (tens of GB)
    run = ScenarioRunner(sc, device=dev, data_device="cpu" if L == 1 else dev).replay()
    tables, ctx, max_ctx = run.decode_metadata()
    S = len(sc.decode_seqs)
    ctx_h = ctx.cpu().numpy()
    # the step's new token per sequence is the last position of each context;
    # the slot the block manager planned for it is the one the fused call
    # derives from the block table (the same in every layer)
    slots_h = np.array([run.alloc.slot_mapping(s, run.alloc.seq_len(s) - 1, 1)[0] for s in sc.decode_seqs])
    tab_h = tables.cpu().numpy()
    B_ = sc.block_size
    assert slots_h.tolist() == [int(tab_h[i, (c - 1) // B_]) * B_ + (int(c) - 1) % B_ for i, c in enumerate(ctx_h)]
    kv_new = [I.append_kv(sc.seed, l, 10 ** 6, S, sc.n_kv_heads, sc.d_head) for l in range(L)]
    k_new = torch.stack([k for k, _ in kv_new]).to(dev)          # [L, S, Hkv, D]
    v_new = torch.stack([v for _, v in kv_new]).to(dev)
    q = torch.stack([I.decode_q(sc.seed, l, S, sc.n_q_heads, sc.d_head) for l in range(L)]).to(dev)
    out = torch.empty_like(q)
    P = args.partition
    ws = api.decode_workspace(S, sc.n_q_heads, sc.d_head, max_ctx, P, device=dev)
    kcs, vcs = run.k_caches, run.v_caches
    fp8 = args.kv_dtype == "fp8"
    scales = [(1.0, 1.0)] * L
    if fp8:
        # the same caches as E4M3 codes, scales from the data's range (setup, not timed)
        scales, k8, v8 = [], [], []
        for kc, vc in zip(kcs, vcs):
            ks = float(kc.float().nan_to_num(0.0).abs().amax()) / 448.0
            vs = float(vc.float().nan_to_num(0.0).abs().amax()) / 448.0
            scales.append((ks, vs))
            k8.append((kc.float() / ks).to(torch.float8_e4m3fn).view(torch.uint8))
            v8.append((vc.float() / vs).to(torch.float8_e4m3fn).view(torch.uint8))
        kcs, vcs = k8, v8
    stream = torch.cuda.current_stream(dev)
    dec_bytes, write_bytes = algorithmic_bytes(sc, ctx_h, S, 1 if fp8 else 2)     # per layer
    # our kernels per layer: the partition kernel (which also writes the new
    # token's K/V into the cache) and, when a sequence can span several
    # partitions, the merge kernel
    launches_per_layer = 1 + (1 if api.pa_decode_workspace_size(S, sc.n_q_heads, sc.d_head, max_ctx, P) else 0)

    def decode_call(l, q_, k_, v_, tables_, ctx_, st_):
        """One layer of the step: the new token's K/V appended at position
        ctx - 1 and decode attention over the cache (pa_decode_append)."""
        api.pa_decode_append(out[l], q_, kcs[l], vcs[l], k_, v_, tables_, ctx_, sc.block_size, sc.scale,
                             sc.n_q_heads, sc.n_kv_heads, sc.d_head, max_ctx, partition_size=P, workspace=ws,
                             stream=st_, k_scale=scales[l][0] if fp8 else None, v_scale=scales[l][1] if fp8 else None)

    def step():
        for l in range(L):
            decode_call(l, q[l], k_new[l], v_new[l], tables, ctx, stream)

    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    for _ in range(args.warmup):
        step()
    K = args.steps
    # Timed region: K whole steps (every layer's cache write and decode, one
    # fused call each) between two events.  The call of layer 0 of every
    # SAMPLE-th step is also bracketed by events: the isolated duration of one
    # call (an event between two kernels stops the second from overlapping the
    # first's drain, so only a sample of steps carries them).
    SAMPLE = 8
    ev_start, ev_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range((K + SAMPLE - 1) // SAMPLE)]
    barrier(world)
    torch.cuda.synchronize(dev)
    torch.cuda.nvtx.range_push(TIMED_RANGE)
    ev_start.record(stream)
    for i in range(K):
        for l in range(L):
            if l == 0 and i % SAMPLE == 0:
                a, b = ev_dec[i // SAMPLE]
                a.record(stream)
                decode_call(l, q[l], k_new[l], v_new[l], tables, ctx, stream)
                b.record(stream)
            else:
                decode_call(l, q[l], k_new[l], v_new[l], tables, ctx, stream)
    ev_end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    barrier(world)
    step_s = ev_start.elapsed_time(ev_end) / 1e3
    isolated_s = sum(a.elapsed_time(b) for a, b in ev_dec) / len(ev_dec) / 1e3
    total_s, total_bytes = reduce_timing(step_s, (dec_bytes + write_bytes) * L * K, world, dev)
    _, total_seqs = reduce_timing(step_s, S * K, world, dev)

    # ---- calls back to back: the kernels' average duration ------------------
    # Repetitions of CALLS pa_decode_append calls (layers in turn; each
    # rewrites the same rows) between two events, run for at least MIN_LOOP_S
    # in all, so that the clock sampler sees the load; median, p10 and p90 of
    # the per-call time over the repetitions.
    CALLS, MIN_REPS, MIN_LOOP_S = 200, 5, 1.2
    per_call = []
    t_loop = time.perf_counter()
    while len(per_call) < MIN_REPS or (time.perf_counter() - t_loop < MIN_LOOP_S and len(per_call) < 500):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for c in range(CALLS):
            decode_call(c % L, q[c % L], k_new[c % L], v_new[c % L], tables, ctx, stream)
        e1.record(stream)
        e1.synchronize()
        per_call.append(e0.elapsed_time(e1) / 1e3 / CALLS)
    loop_s = time.perf_counter() - t_loop
    clk = clocks.stop() if clocks else None
    dec_med, dec_p10, dec_p90 = _quantiles(per_call)
    step_per_layer_s = total_s / K / L
    if dec_med > step_per_layer_s * 1.02:
        raise RuntimeError("call (%.2f us back to back) longer than a whole step's layer (%.2f us): the "
                           "timing is inconsistent" % (dec_med * 1e6, step_per_layer_s * 1e6))

    # ---- end to end through the public API with host buffers ---------------
    # Every step copies its inputs from pinned host memory (q and the new K/V
    # rows of every layer, block tables, context lengths), runs every layer's
    # fused cache write and decode, copies the outputs back and waits for
    # them.  The step is issued once into a CUDA graph (the library's
    # calls are capturable) and replayed; the eager form is timed too.  The
    # inputs travel packed in one page-locked buffer (one copy per step; six
    # small copies each paid their own latency), and the calls read views of
    # its device twin.
    inputs = (q, k_new, v_new, tables, ctx)
    offs, total = [], 0
    for t in inputs:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    pack_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    pack_d = torch.empty(total, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(inputs, offs):
        nb = t.numel() * t.element_size()
        pack_h[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        views.append(pack_d[o:o + nb].view(t.dtype).view(t.shape))
    q_d, k_d, v_d, tables_d, ctx_d = views
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in inputs)
    d2h = out_h.numel() * out_h.element_size()

    def e2e_body(st):
        pack_d.copy_(pack_h, non_blocking=True)
        for l in range(L):
            decode_call(l, q_d[l], k_d[l], v_d[l], tables_d, ctx_d, st)
        out_h.copy_(out, non_blocking=True)

    def eager_step():
        e2e_body(stream)
        stream.synchronize()

    graph = torch.cuda.CUDAGraph()
    for _ in range(args.warmup):
        eager_step()
    with torch.cuda.graph(graph):
        e2e_body(torch.cuda.current_stream(dev))

    def graph_step():
        graph.replay()
        stream.synchronize()

    e2e_times = {}
    for name, fn in (("graph", graph_step), ("eager", eager_step)):
        for _ in range(args.warmup):
            fn()
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(K):
            fn()
        torch.cuda.synchronize(dev)
        e2e_times[name] = time.perf_counter() - t0
        barrier(world)
    e2e_total_s, e2e_bytes = reduce_timing(e2e_times["graph"], (dec_bytes + write_bytes) * L * K, world, dev)
    eager_total_s, _ = reduce_timing(e2e_times["eager"], 0, world, dev)

    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    achieved = (dec_bytes + write_bytes) / dec_med / 1e9
    value = total_bytes / total_s / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_s / K * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "kv_dtype": "fp8_e4m3" if fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": sc.name, "num_seqs": S, "n_layers": L,
                   "context_lens": {"batch64_8b": "uniform [512, 4096]", "long_context": "32,768 each",
                                    "mixed_batch": "lognormal (median 700, sigma 1) clipped to [1, 16384]"}.get(
                                        args.workload, "see workload"), "total_context": int(ctx_h.sum()),
                   "n_q_heads": sc.n_q_heads, "n_kv_heads": sc.n_kv_heads, "d_head": sc.d_head,
                   "block_size": sc.block_size, "num_blocks": sc.num_blocks, "placement": "seeded random",
                   "partition_size": P or "library default",
                   "l2": "inputs larger than L2 (%.0f MB KV read per layer vs 129 MB L2); no flush" %
                         (dec_bytes / 1e6),
                   "parallelism": "replicas (one batch per GPU)" if world > 1 else "single GPU"},
        "seqs_per_s": round(total_seqs / total_s, 1),
        "ms_per_layer": round(total_s / K / L * 1e3, 5),
        "roofline": {"bound": "hbm", "kernel": "pa_decode_append%s (decode_partition_kernel, which also "
                     "writes the new rows, + lse_merge_kernel)" % ("_fp8" if fp8 else ""),
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(PROFILE_SUMMARY_FP8 if fp8 else PROFILE_SUMMARY)
                     if args.workload == "batch64_8b" and sc.block_size == 16 and P == 0 else None,
                     "algorithmic_bytes_per_launch": int(dec_bytes + write_bytes),
                     "avg_launch_us": round(dec_med * 1e6, 2),
                     "launch_us_p10_p90": [round(dec_p10 * 1e6, 2), round(dec_p90 * 1e6, 2)],
                     "timing": "median over %d repetitions of %d pa_decode_append calls back to back between two events "
                               "(%.2f s of calls)" % (len(per_call), CALLS, loop_s),
                     "isolated_call_us": round(isolated_s * 1e6, 2),
                     "isolated_call_timing": "events around layer 0's call on every %d-th timed step (%d "
                                             "samples; the event pair keeps the call from overlapping the "
                                             "kernel before it)" % (SAMPLE, len(ev_dec)),
                     "step_frac": round(value / peak, 4)},
        "e2e": {"value": round(e2e_bytes / e2e_total_s / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_total_s / K * 1e3, 4), "issue": "CUDA graph of the step, replayed; inputs in one packed page-locked buffer, one copy in "
                "and one out per step, waited for",
                "eager_value": round(e2e_bytes / eager_total_s / 1e9, 2),
                "eager_ms_per_step": round(eager_total_s / K * 1e3, 4)},
        "gpu_launches": launches_per_layer * L * K,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sc, args.cpu_seconds)
    return line


# ----------------------------------------------------------------------------
# prefill (causal attention of many new positions per sequence)
# ----------------------------------------------------------------------------

def _prefill_metadata(sc, api):
    """Block tables and the new positions' slots from the C++ block manager
    (seeded free order), for every sequence's full context."""
    alloc = api.BlockAllocator(sc.num_blocks, sc.block_size)
    assert alloc.set_free_order(sc.free_order) == 0
    for s, c in enumerate(sc.ctxs):
        assert alloc.allocate(s, c) == 0
    seqs = list(range(len(sc.ctxs)))
    tables, ctx = alloc.build_tables(seqs, max(len(alloc.block_table(s)) for s in seqs))
    slots = np.concatenate([alloc.slot_mapping(s, c - n, n) for s, (c, n) in enumerate(zip(sc.ctxs, sc.news))])
    return tables, ctx, slots


def run_prefill_ours(args, world, rank, local):
    from paged_kv_cache_124_gb300 import api

    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    seed = replica_seed(args.seed, rank)
    sc = PREFILL_WORKLOADS[args.workload](seed, args.block_size)
    tables_h, ctx_h, slots_h = _prefill_metadata(sc, api)
    kc, vc = I.prefill_pool(sc, dev)
    q = I.prefill_q(sc, dev)
    k_new, v_new = I.prefill_new_kv(sc, dev)
    out = torch.empty_like(q)
    tables, ctx = torch.from_numpy(tables_h).to(dev), torch.from_numpy(ctx_h).to(dev)
    qs = torch.from_numpy(sc.query_start).to(dev)
    slots = torch.from_numpy(slots_h).to(dev)
    max_q = max(sc.news)
    stream = torch.cuda.current_stream(dev)
    flops = prefill_flops(sc.ctxs, sc.news, sc.n_q_heads, sc.d_head)
    T = int(sum(sc.news))

    fp8 = args.kv_dtype == "fp8"
    ks = vs = 1.0
    if fp8:
        # the same caches as E4M3 codes, scales from the data's range (setup, not timed); the step's new
        # rows are then quantised by pa_reshape_and_cache_fp8
        ks = float(kc.float().nan_to_num(0.0).abs().amax()) / 448.0
        vs = float(vc.float().nan_to_num(0.0).abs().amax()) / 448.0
        kc = (kc.float() / ks).to(torch.float8_e4m3fn).view(torch.uint8)
        vc = (vc.float() / vs).to(torch.float8_e4m3fn).view(torch.uint8)
    # the call's workspace (V, and for FP8 also K, staged) is
    # allocated once, outside the timed region
    if fp8:
        workspace = api.prefill_fp8_workspace(len(sc.news), tables_h.shape[1], sc.block_size, sc.n_kv_heads,
                                              sc.d_head, dev)
    else:
        workspace = api.prefill_workspace(len(sc.news), tables_h.shape[1], sc.block_size, sc.n_kv_heads, sc.d_head,
                                          dev)

    def cache_write(k_, v_, slots_, st):
        if fp8:
            api.pa_reshape_and_cache_fp8(kc, vc, k_, v_, slots_, ks, vs, stream=st)
        else:
            api.pa_reshape_and_cache(kc, vc, k_, v_, slots_, stream=st)

    def attention(q_, tables_, qs_, ctx_, st):
        if fp8:
            api.pa_prefill_fp8(out, q_, kc, vc, tables_, qs_, ctx_, max_q, sc.block_size, sc.scale, ks, vs,
                               sc.n_q_heads, sc.n_kv_heads, sc.d_head, stream=st, workspace=workspace)
        else:
            api.pa_prefill(out, q_, kc, vc, tables_, qs_, ctx_, max_q, sc.block_size, sc.scale, sc.n_q_heads,
                           sc.n_kv_heads, sc.d_head, stream=st, workspace=workspace)

    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    for _ in range(args.warmup):
        cache_write(k_new, v_new, slots, stream)
        attention(q, tables, qs, ctx, stream)
    K = args.steps
    SAMPLE = 4
    ev_start, ev_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_att = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range((K + SAMPLE - 1) // SAMPLE)]
    barrier(world)
    torch.cuda.synchronize(dev)
    torch.cuda.nvtx.range_push(TIMED_RANGE)
    ev_start.record(stream)
    for i in range(K):
        cache_write(k_new, v_new, slots, stream)
        if i % SAMPLE == 0:
            a, b = ev_att[i // SAMPLE]
            a.record(stream)
            attention(q, tables, qs, ctx, stream)
            b.record(stream)
        else:
            attention(q, tables, qs, ctx, stream)
    ev_end.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    barrier(world)
    step_s = ev_start.elapsed_time(ev_end) / 1e3
    isolated_s = sum(a.elapsed_time(b) for a, b in ev_att) / len(ev_att) / 1e3
    total_s, total_flops = reduce_timing(step_s, flops * K, world, dev)
    _, total_tokens = reduce_timing(step_s, T * K, world, dev)

    # pa_prefill calls back to back: repetitions of CALLS calls between two
    # events, run for at least MIN_LOOP_S in all; median, p10, p90 per call
    CALLS, MIN_REPS, MIN_LOOP_S = 20, 5, 1.2
    per_call = []
    t_loop = time.perf_counter()
    while len(per_call) < MIN_REPS or (time.perf_counter() - t_loop < MIN_LOOP_S and len(per_call) < 200):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(CALLS):
            attention(q, tables, qs, ctx, stream)
        e1.record(stream)
        e1.synchronize()
        per_call.append(e0.elapsed_time(e1) / 1e3 / CALLS)
    loop_s = time.perf_counter() - t_loop
    clk = clocks.stop() if clocks else None
    att_s, att_p10, att_p90 = _quantiles(per_call)
    if att_s > total_s / K * 1.02:
        raise RuntimeError("prefill call (%.1f us back to back) longer than a whole step (%.1f us): the timing is "
                           "inconsistent" % (att_s * 1e6, total_s / K * 1e6))

    # end to end with host buffers: q, the new K/V rows, slots, tables, query
    # starts and context lengths in; the attention output back
    q_h = q.cpu().pin_memory()
    k_h, v_h = k_new.cpu().pin_memory(), v_new.cpu().pin_memory()
    slots_hp, tables_hp = slots.cpu().pin_memory(), tables.cpu().pin_memory()
    qs_hp, ctx_hp = qs.cpu().pin_memory(), ctx.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    q_d, k_d, v_d = torch.empty_like(q), torch.empty_like(k_new), torch.empty_like(v_new)
    slots_d, tables_d, qs_d, ctx_d = (torch.empty_like(slots), torch.empty_like(tables), torch.empty_like(qs),
                                      torch.empty_like(ctx))
    pairs = ((q_d, q_h), (k_d, k_h), (v_d, v_h), (slots_d, slots_hp), (tables_d, tables_hp), (qs_d, qs_hp),
             (ctx_d, ctx_hp))
    h2d = sum(src.numel() * src.element_size() for _, src in pairs)
    d2h = out_h.numel() * out_h.element_size()

    def e2e_step():
        for dst, src in pairs:
            dst.copy_(src, non_blocking=True)
        cache_write(k_d, v_d, slots_d, stream)
        attention(q_d, tables_d, qs_d, ctx_d, stream)
        out_h.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(args.warmup):
        e2e_step()
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(K):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_s, e2e_flops = reduce_timing(time.perf_counter() - t0, flops * K, world, dev)
    barrier(world)

    if rank != 0:
        return None
    peak, peak_kind = measured_peak("bf16_tflops", 1900.0)
    peak_sus, _ = measured_peak("bf16_tflops_sustained", 1700.0)
    achieved = flops / att_s / 1e12
    kv_bytes = sum(sc.ctxs) * sc.n_kv_heads * sc.d_head * 2 * (1 if fp8 else 2)
    line = {
        "metric": PREFILL_METRIC, "value": round(total_flops / total_s / 1e12, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(total_s / K * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "kv_dtype": "fp8_e4m3" if fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": sc.name, "num_seqs": len(sc.ctxs), "new_tokens": T, "context_lens":
                   "all %d" % sc.ctxs[0] if len(set(sc.ctxs)) == 1 else "prefix U[2048, 8192] + 512",
                   "total_context": int(sum(sc.ctxs)), "n_q_heads": sc.n_q_heads, "n_kv_heads": sc.n_kv_heads,
                   "d_head": sc.d_head, "block_size": sc.block_size, "num_blocks": sc.num_blocks,
                   "placement": "seeded random (block manager free order)",
                   "l2": "inputs larger than L2 (%.0f MB K/V + %.0f MB q/out vs 129 MB L2); no flush" %
                         (kv_bytes / 1e6, 2 * q.numel() * 2 / 1e6),
                   "parallelism": "replicas (one batch per GPU)" if world > 1 else "single GPU"},
        "tokens_per_s": round(total_tokens / total_s, 1),
        "roofline": {"bound": "tensor", "kernel": "pa_prefill_fp8 (stage_kv_f8_kernel + prefill_kernel<128, fp8>)" if fp8
                     else "pa_prefill (stage_v_kernel<128> + prefill_kernel<128>)", "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind + " bf16 burst", "peak_sustained": peak_sus,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(PREFILL_PROFILE, PREFILL_SOURCE)
                     if sc.name == "prefill_prompts_8b" and not fp8 else None,
                     "algorithmic_flops_per_launch": flops, "avg_launch_us": round(att_s * 1e6, 2),
                     "launch_us_p10_p90": [round(att_p10 * 1e6, 2), round(att_p90 * 1e6, 2)],
                     "timing": "median over %d repetitions of %d pa_prefill calls back to back between two events "
                               "(%.2f s of calls)" % (len(per_call), CALLS, loop_s),
                     "isolated_call_us": round(isolated_s * 1e6, 2),
                     "isolated_call_timing": "events around pa_prefill on every %d-th timed step (%d samples)" %
                                             (SAMPLE, len(ev_att)),
                     "step_frac": round(total_flops / total_s / 1e12 / peak, 4)},
        "e2e": {"value": round(e2e_flops / e2e_s / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_s / K * 1e3, 4)},
        # reshape_and_cache, the staging (V; FP8: K and V), prefill_kernel
        "gpu_launches": 3 * K,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(sc, args.cpu_seconds)
    return line


def _prefill_oracle_sample(sc, seq, rows):
    """The oracle's inputs for the last `rows` new positions of one sequence
    (its whole context is gathered), drawn on the CPU."""
    c, n = sc.ctxs[seq], sc.news[seq]
    B = sc.block_size
    nb = -(-c // B)
    rng_k = I.bf16_bits(I.bf16_normal((nb, sc.n_kv_heads, B, sc.d_head), 11 + seq))
    rng_v = I.bf16_bits(I.bf16_normal((nb, sc.n_kv_heads, B, sc.d_head), 12 + seq))
    q = I.bf16_bits(I.bf16_normal((rows, sc.n_q_heads, sc.d_head), 13 + seq))
    tables = np.arange(nb, dtype=np.int32)[None, :]
    return q, rng_k, rng_v, tables, np.array([0, rows], dtype=np.int32), np.array([c - n + n], dtype=np.int32)


def _prefill_oracle_time(sc, seq, rows):
    from oracle import attention as A
    q, kc, vc, tables, qs, ctx = _prefill_oracle_sample(sc, seq, rows)
    t0 = time.perf_counter()
    A.paged_prefill(q, kc, vc, tables, qs, ctx, sc.scale, sc.block_size)
    t = time.perf_counter() - t0
    c = int(ctx[0])
    return t, prefill_flops([c], [rows], sc.n_q_heads, sc.d_head)


def prefill_cpu_baseline(sc, budget_s):
    """The oracle as it stands, on a bounded sample: the last query rows of
    the first sequence (all heads, over its whole context), as many as fit
    about budget_s, on one thread and (the reported value) on every host
    core at once, one worker process per core with a share of the rows."""
    rows = 1
    t, f = _prefill_oracle_time(sc, 0, rows)
    while t < budget_s / 2 and rows < sc.news[0]:
        rows = min(sc.news[0], max(rows + 1, int(rows * min(8.0, budget_s / max(t, 1e-3)))))
        t, f = _prefill_oracle_time(sc, 0, rows)
    desc = ("fp64 oracle prefill of the last %d of %d new positions of sequence 0 (context %d, all %d query heads) "
            "of %s" % (rows, sc.news[0], sc.ctxs[0], sc.n_q_heads, sc.name))
    one = {"value": round(f / t / 1e12, 8), "cores": 1, "sample": desc + ", %.1f s, 1 thread" % t}
    procs = host_threads()
    if procs <= 1:
        return dict(one, unit="TFLOP/s", kind="oracle")
    rows_all = min(sc.news[0], rows * procs)            # about as long per core as the one-thread leg
    try:
        t_all = _prefill_oracle_time_procs(sc, rows_all, procs, 1)
    except Exception as e:                             # the one-thread leg stands alone
        return dict(one, unit="TFLOP/s", kind="oracle", all_cores_failed=str(e)[:200])
    c = sc.ctxs[0]
    f_all = prefill_flops([c], [rows_all], sc.n_q_heads, sc.d_head)
    value = f_all / t_all / 1e12
    return {"value": round(value, 8), "unit": "TFLOP/s", "cores": procs, "kind": "oracle",
            "sample": "fp64 oracle prefill of the last %d of %d new positions of sequence 0 (context %d, all %d "
                      "query heads) of %s, %.1f s, %d worker processes at once, a share of the rows each" %
                      (rows_all, sc.news[0], c, sc.n_q_heads, sc.name, t_all, procs),
            "single_thread": one, "speedup_all_cores": round(value / max(one["value"], 1e-12), 1)}


def run_prefill_reference(args, world, rank):
    if rank != 0:
        return None
    sc = PREFILL_WORKLOADS[args.workload](args.seed, args.block_size)
    rows = max(1, args.ref_seqs_per_step)
    samples = []
    for i in range(args.warmup + args.steps):
        seq = i % len(sc.ctxs)
        t, f = _prefill_oracle_time(sc, seq, rows)
        if i >= args.warmup:
            samples.append((t, f))
    tot_t = sum(x[0] for x in samples)
    value = sum(x[1] for x in samples) / tot_t / 1e12
    desc = ("fp64 oracle prefill, the last %d new position(s) of one sequence of %s per step (rotating), all %d "
            "query heads" % (rows, sc.name, sc.n_q_heads))
    return {"impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 8), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_t / len(samples) * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": sc.name, "rows_per_step": rows},
            "cpu_baseline": {"value": round(value, 8), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 8), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------
# swapping (blocks of preempted sequences to page-locked host memory and back)
# ----------------------------------------------------------------------------

SWAP_METRIC = "paged KV swap GB/s (device<->host block moves, 8B GQA shape; frac of measured link copy)"
SWAP_LAYERS = 8
SWAP_SEQS = 16


def _link_copy_peak(dev, nbytes=1 << 30, reps=5):
    """Plain copy-engine bandwidth of this GPU's host link, per direction:
    cudaMemcpyAsync of one contiguous page-locked buffer (best of reps)."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = {}
    for name, dst, src in (("d2h", h, d), ("h2d", d, h)):
        t = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            dst.copy_(src, non_blocking=True)
            b.record()
            torch.cuda.synchronize(dev)
            t.append(a.elapsed_time(b) / 1e3)
        best[name] = nbytes / min(t) / 1e9
    del h, d
    return best


def run_swap_ours(args, world, rank, local):
    from paged_kv_cache_124_gb300 import api
    from paged_kv_cache_124_gb300.runner import ScenarioRunner

    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    seed = replica_seed(args.seed, rank)
    sc = I.batch64_8b(seed, args.block_size)
    run = ScenarioRunner(sc, device=dev, data_device="cpu").replay()
    alloc = run.alloc
    L = SWAP_LAYERS
    # every layer holds the same block placement; the payload of layer 0 is real, the others are copies of it
    kc = [run.k_caches[0]] + [run.k_caches[0].clone() for _ in range(L - 1)]
    vc = [run.v_caches[0]] + [run.v_caches[0].clone() for _ in range(L - 1)]
    victims = list(range(SWAP_SEQS))
    n_blocks = sum(len(alloc.block_table(s)) for s in victims)
    assert alloc.enable_swap(n_blocks) == 0
    shape = (n_blocks,) + tuple(kc[0].shape[1:])
    hk = [torch.empty(shape, dtype=torch.bfloat16).pin_memory() for _ in range(L)]
    hv = [torch.empty(shape, dtype=torch.bfloat16).pin_memory() for _ in range(L)]
    block_bytes = 2 * int(np.prod(shape[1:])) * 2 * L          # K and V, all layers
    stream = torch.cuda.current_stream(dev)
    before = [t.clone() for t in (kc[0], vc[0])]
    tab0 = alloc.build_tables(victims, max(len(alloc.block_table(s)) for s in victims))[0]

    # Page-locked pair lists, two per direction: a list is rewritten only once
    # the copy that read it has run (its event), so the host never waits on
    # the copy just issued.
    ring = {d: [torch.empty((n_blocks, 2), dtype=torch.int32).pin_memory() for _ in range(2)] for d in ("out", "in")}
    ring_ev = {d: [None, None] for d in ("out", "in")}
    counter = [0]

    def issue(direction, pairs, dst_k, dst_v, src_k, src_v):
        slot = counter[0] & 1
        if ring_ev[direction][slot] is not None:
            ring_ev[direction][slot].synchronize()
        buf = ring[direction][slot][:len(pairs)]
        buf.copy_(torch.from_numpy(pairs))
        api.pa_swap_blocks(dst_k, dst_v, src_k, src_v, buf, stream=stream)
        ev_ = torch.cuda.Event()
        ev_.record(stream)
        ring_ev[direction][slot] = ev_

    def step():
        st, out_pairs = alloc.swap_out(victims)
        assert st == 0
        issue("out", out_pairs, hk, hv, kc, vc)
        st, in_pairs = alloc.swap_in(victims)
        assert st == 0
        issue("in", in_pairs, kc, vc, hk, hv)
        counter[0] += 1
        return len(out_pairs) + len(in_pairs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    K = args.steps
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    moved = 0
    for _ in range(K):
        moved += step()
    torch.cuda.synchronize(dev)
    elapsed = time.perf_counter() - t0
    barrier(world)
    clk = clocks.stop() if clocks else None
    total_s, total_bytes = reduce_timing(elapsed, moved * block_bytes, world, dev)
    # one out-kernel and one in-kernel timed alone with events, for the roofline
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    st, out_pairs = alloc.swap_out(victims)
    pairs_h = torch.from_numpy(out_pairs).pin_memory()
    ev[0].record(stream)
    api.pa_swap_blocks(hk, hv, kc, vc, pairs_h, stream=stream)
    ev[1].record(stream)
    st, in_pairs = alloc.swap_in(victims)
    pairs_h2 = torch.from_numpy(in_pairs).pin_memory()
    ev[2].record(stream)
    api.pa_swap_blocks(kc, vc, hk, hv, pairs_h2, stream=stream)
    ev[3].record(stream)
    torch.cuda.synchronize(dev)
    out_s = ev[0].elapsed_time(ev[1]) / 1e3
    in_s = ev[2].elapsed_time(ev[3]) / 1e3
    out_gbs = len(out_pairs) * block_bytes / out_s / 1e9
    in_gbs = len(in_pairs) * block_bytes / in_s / 1e9
    # payload check: after all the round trips the victims' blocks hold what they held at the start
    tab_after, ctx_v = alloc.build_tables(victims, tab0.shape[1])
    for i in range(len(victims)):
        nb = -(-int(ctx_v[i]) // sc.block_size)
        for a, b in ((before[0], kc[0]), (before[1], vc[0])):
            # compare bit patterns: the blocks' unused tail slots hold NaN
            if not torch.equal(a[torch.from_numpy(tab0[i, :nb]).long().to(dev)].view(torch.int16),
                               b[torch.from_numpy(tab_after[i, :nb]).long().to(dev)].view(torch.int16)):
                raise RuntimeError("swap round trip changed the payload of sequence %d" % victims[i])
    if rank != 0:
        return None
    link = _link_copy_peak(dev)
    peak = min(link["d2h"], link["h2d"])
    line = {
        "metric": SWAP_METRIC, "value": round(total_bytes / total_s / 1e9, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(total_s / K * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bytes moved)", "data": "synthetic",
        "config": {"workload": "swap_8b", "sequences_swapped": SWAP_SEQS, "layers": L, "blocks_per_direction":
                   n_blocks, "block_bytes_all_layers_kv": block_bytes, "block_size": sc.block_size,
                   "n_kv_heads": sc.n_kv_heads, "d_head": sc.d_head,
                   "step": "swap_out plan + pa_swap_blocks to pinned host, swap_in plan + pa_swap_blocks back",
                   "l2": "each direction moves %.2f GB (> 129 MB L2); no flush" % (n_blocks * block_bytes / 1e9)},
        "roofline": {"bound": "host link", "kernel": "swap_blocks_kernel", "achieved": round(min(out_gbs, in_gbs), 1),
                     "out_gbs": round(out_gbs, 1), "in_gbs": round(in_gbs, 1), "peak": round(peak, 1),
                     "peak_kind": "measured in this run: cudaMemcpyAsync of 1 GiB page-locked (d2h %.1f, h2d %.1f GB/s)"
                                  % (link["d2h"], link["h2d"]),
                     "unit": "GB/s", "frac": round(min(out_gbs, in_gbs) / peak, 4), "traffic": None},
        "e2e": {"value": round(total_bytes / total_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(n_blocks * block_bytes), "d2h_bytes_per_step": int(n_blocks * block_bytes),
                "note": "swapping is host<->device by definition: value is already end to end (planning included)"},
        "gpu_launches": 2 * K,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = swap_cpu_baseline(sc, args.cpu_seconds)
    return line


def swap_cpu_baseline(sc, budget_s):
    """The oracle's swap_blocks (NumPy copies of whole blocks) on host pools of
    the same block shape, as many block moves as fit about budget_s."""
    from oracle import cache_ops as C
    shape = (sc.n_kv_heads, sc.block_size, sc.d_head)
    nb = 4096
    rng = np.random.default_rng(0)
    src_k = rng.integers(0, 65535, size=(nb,) + shape, dtype=np.uint16)
    src_v = src_k.copy()
    dst_k, dst_v = np.zeros_like(src_k), np.zeros_like(src_v)
    pairs = list(zip(rng.permutation(nb).tolist(), rng.permutation(nb).tolist()))
    moved, t = 0, 0.0
    t0 = time.perf_counter()
    while t < budget_s:
        C.swap_blocks(dst_k, dst_v, src_k, src_v, pairs)
        moved += len(pairs)
        t = time.perf_counter() - t0
    per_block = 2 * int(np.prod(shape)) * 2
    return {"value": round(moved * per_block / t / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "oracle swap_blocks between two host pools of %d blocks, %d block moves (K and V), %.1f s"
                      % (nb, moved, t)}


CACHE_OPS_METRIC = "paged KV cache write + CoW copy GB/s (HBM bytes read + written, frac of measured HBM)"
CACHE_OPS_LAYERS = 32          # copy_blocks copies a block in every layer of the 8B model


def _cache_ops_inputs(seed, block_size, api):
    """The 16 x 2,003-token prompts of the CoW sampling config: their new K/V
    rows and slots (block manager, seeded free order), and the copy-on-write
    pairs that forking each prompt into 8 samples and appending one token to
    every sample produces (the first 7 writers of each shared tail copy it)."""
    sc = I.prefill_prompts(seed, block_size)
    _, _, slots = _prefill_metadata(sc, api)
    n_prompts, samples = len(sc.ctxs), 8
    alloc = api.BlockAllocator(sc.num_blocks + n_prompts * samples, block_size)
    assert alloc.set_free_order(list(sc.free_order) + list(range(sc.num_blocks, sc.num_blocks + n_prompts * samples))) == 0
    pairs = []
    for s_, c in enumerate(sc.ctxs):
        assert alloc.allocate(s_ * samples, c) == 0
        for f in range(1, samples):
            assert alloc.fork(s_ * samples, s_ * samples + f) == 0
    for s_ in range(n_prompts * samples):
        st, _, src, dst = alloc.append_slot(s_)
        assert st == 0
        if src >= 0:
            pairs.append((src, dst))
    return sc, slots, np.asarray(pairs, dtype=np.int32), sc.num_blocks + n_prompts * samples


def run_cache_ops_ours(args, world, rank, local):
    from paged_kv_cache_124_gb300 import api

    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    seed = replica_seed(args.seed, rank)
    sc, slots_h, pairs_h, nb = _cache_ops_inputs(seed, args.block_size, api)
    L = CACHE_OPS_LAYERS
    shape = (nb, sc.n_kv_heads, sc.block_size, sc.d_head)
    g = torch.Generator(device=dev).manual_seed(seed)
    kc = [torch.randn(shape, generator=g, device=dev).bfloat16() for _ in range(L)]
    vc = [torch.randn(shape, generator=g, device=dev).bfloat16() for _ in range(L)]
    k_new, v_new = I.prefill_new_kv(sc, dev)
    slots = torch.from_numpy(slots_h).to(dev)
    pairs = torch.from_numpy(pairs_h).to(dev)
    T, P = int(slots_h.shape[0]), int(pairs_h.shape[0])
    row = sc.n_kv_heads * sc.d_head * 2
    write_bytes = 2 * T * row * 2 + T * 8                         # K and V rows read and written, slots read
    # K and V blocks: each distinct source read once (its copies to several
    # destinations reread it from L2), each destination written once
    blk_kv = 2 * sc.n_kv_heads * sc.block_size * sc.d_head * 2
    copy_bytes = (len(set(pairs_h[:, 0].tolist())) + P) * L * blk_kv
    stream = torch.cuda.current_stream(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(k_, v_, slots_, pairs_):
        api.pa_reshape_and_cache(kc[0], vc[0], k_, v_, slots_, status=status, stream=stream)
        api.pa_copy_blocks(kc, vc, pairs_, status=status, stream=stream)

    for _ in range(args.warmup):
        step(k_new, v_new, slots, pairs)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(K):
        a, b, c = ev[i]
        a.record(stream)
        api.pa_reshape_and_cache(kc[0], vc[0], k_new, v_new, slots, status=status, stream=stream)
        b.record(stream)
        api.pa_copy_blocks(kc, vc, pairs, status=status, stream=stream)
        c.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop() if clocks else None
    w_s = float(np.mean([a.elapsed_time(b) for a, b, _ in ev])) / 1e3
    c_s = float(np.mean([b.elapsed_time(c) for _, b, c in ev])) / 1e3
    total = ev[0][0].elapsed_time(ev[-1][2]) / 1e3
    total_s, total_bytes = reduce_timing(total, K * (write_bytes + copy_bytes), world, dev)
    if int(status.item()) != 0:
        raise RuntimeError("cache ops flagged status %d" % int(status.item()))
    # e2e through the same calls with host inputs: new K/V rows, slots and pairs copied in, the status word read back
    hk, hv = k_new.cpu().pin_memory(), v_new.cpu().pin_memory()
    hs, hp = torch.from_numpy(slots_h).pin_memory(), torch.from_numpy(pairs_h).pin_memory()
    hst = torch.zeros(1, dtype=torch.int32).pin_memory()
    dk, dv, ds, dp = torch.empty_like(k_new), torch.empty_like(v_new), torch.empty_like(slots), torch.empty_like(pairs)
    h2d = hk.numel() * 2 + hv.numel() * 2 + hs.numel() * 8 + hp.numel() * 4

    def e2e_step():
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        ds.copy_(hs, non_blocking=True)
        dp.copy_(hp, non_blocking=True)
        step(dk, dv, ds, dp)
        hst.copy_(status, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    KE = max(3, K // 4)
    e0.record(stream)
    for _ in range(KE):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s, _ = reduce_timing(e0.elapsed_time(e1) / 1e3, 0, world, dev)
    if rank != 0:
        return None
    peak, peak_kind = measured_peak("hbm_gbs", FALLBACK_HBM_GBS)
    copy_gbs, write_gbs = copy_bytes / c_s / 1e9, write_bytes / w_s / 1e9
    line = {
        "metric": CACHE_OPS_METRIC, "value": round(total_bytes / total_s / 1e9, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(total_s / K * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bit copies)", "data": "synthetic",
        "config": {"workload": "cache_ops_8b", "tokens_written": T, "cow_pairs": P,
                   "distinct_sources": len(set(pairs_h[:, 0].tolist())), "layers_copied": L,
                   "n_kv_heads": sc.n_kv_heads, "d_head": sc.d_head, "block_size": sc.block_size,
                   "pool_blocks_per_layer": nb,
                   "step": "pa_reshape_and_cache of the 16 x 2,003 prompt tokens (one layer) + pa_copy_blocks of the "
                           "copy-on-write pairs of forking each prompt into 8 samples (all %d layers)" % L,
                   "l2": "%.0f MB written and %.0f MB copied per step (> 129 MB L2); no flush"
                         % (write_bytes / 1e6, copy_bytes / 1e6)},
        "roofline": {"bound": "hbm", "kernel": "copy_blocks_kernel", "achieved": round(copy_gbs, 1), "peak": peak,
                     "peak_kind": peak_kind + " copy (read + write bytes)", "unit": "GB/s",
                     "frac": round(copy_gbs / peak, 4),
                     "traffic": profiled_traffic(CACHE_OPS_PROFILE, CACHE_OPS_SOURCE),
                     "algorithmic_bytes_per_launch": copy_bytes, "avg_launch_us": round(c_s * 1e6, 2)},
        "roofline_reshape_and_cache": {"bound": "hbm", "kernel": "reshape_and_cache_kernel",
                                       "achieved": round(write_gbs, 1), "peak": peak, "unit": "GB/s",
                                       "frac": round(write_gbs / peak, 4), "algorithmic_bytes_per_launch": write_bytes,
                                       "avg_launch_us": round(w_s * 1e6, 2)},
        "e2e": {"value": round((write_bytes + copy_bytes) / e2e_s * KE / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 4, "ms_per_step": round(e2e_s / KE * 1e3, 4)},
        "gpu_launches": 2 * K,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cache_ops_cpu_baseline(sc, slots_h, pairs_h, nb, args.cpu_seconds)
    return line


def cache_ops_cpu_baseline(sc, slots_h, pairs_h, nb, budget_s):
    """The oracle's reshape_and_cache and copy_blocks (plain loops over host
    pools of the same shape), as many tokens and pairs as fit about budget_s;
    bytes counted like the GPU's (read + written)."""
    from oracle import cache_ops as C
    rng = np.random.default_rng(0)
    shape = (nb, sc.n_kv_heads, sc.block_size, sc.d_head)
    kc = rng.integers(0, 65535, size=shape, dtype=np.uint16)
    vc = kc.copy()
    n_tok = 4096
    k = rng.integers(0, 65535, size=(n_tok, sc.n_kv_heads, sc.d_head), dtype=np.uint16)
    v = k.copy()
    row = sc.n_kv_heads * sc.d_head * 2
    blk = sc.n_kv_heads * sc.block_size * sc.d_head * 2
    moved, t = 0, 0.0
    t0 = time.perf_counter()
    while t < budget_s:
        C.reshape_and_cache(kc, vc, k, v, slots_h[:n_tok], sc.block_size)
        C.copy_blocks([kc], [vc], [tuple(p) for p in pairs_h.tolist()])
        moved += 2 * n_tok * row * 2 + 2 * len(pairs_h) * blk * 2
        t = time.perf_counter() - t0
    return {"value": round(moved / t / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "oracle reshape_and_cache of %d tokens + copy_blocks of %d pairs (one layer) per round, "
                      "host pools of %d blocks, %.1f s" % (n_tok, len(pairs_h), nb, t)}


# ----------------------------------------------------------------------------
# CPU oracle (the cpu_baseline leg and --impl reference)
# ----------------------------------------------------------------------------

def _oracle_sample(sc, seqs):
    """Oracle replay of the workload's layer 0 with only `seqs` materialised
    (every layer does the same work)."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from _oracle_replay import OracleReplay
    sub = dataclasses.replace(sc, decode_seqs=list(seqs))
    rep = OracleReplay(sub, layers=[0]).replay()
    tab, lens = rep.tables()
    q = I.bf16_bits(I.decode_q(sc.seed, 0, len(sc.decode_seqs), sc.n_q_heads, sc.d_head))[list(seqs)]
    return rep, tab, lens, q


def _oracle_time(sc, rep, tab, lens, q):
    from oracle import attention as A
    t0 = time.perf_counter()
    A.paged_decode(q, rep.k[0], rep.v[0], tab, lens, sc.scale, sc.block_size)
    return time.perf_counter() - t0


def _oracle_time_procs(sc, rep, tab, lens, q, procs, reps):
    """Seconds the oracle takes to decode the sample `reps` times on `procs`
    host cores at once: the sample (its blocks compacted into a small pool)
    goes to a temporary directory, and one worker process per core
    (tests/_oracle_pool.py, started fresh, not forked from this process)
    decodes its share of the sequences (longest first, each to the least
    loaded worker).  All start together; the slowest worker's time counts."""
    import shutil
    B = sc.block_size
    nblk = [-(-int(c) // B) for c in lens]
    used = sorted(set(int(b) for i, n in enumerate(nblk) for b in tab[i, :n]))
    remap = {b: i for i, b in enumerate(used)}
    ctab = np.full(tab.shape, -1, dtype=np.int64)
    for i, n in enumerate(nblk):
        ctab[i, :n] = [remap[int(b)] for b in tab[i, :n]]
    load = [0] * procs
    assign = [[] for _ in range(procs)]
    for i in sorted(range(len(lens)), key=lambda i: -int(lens[i])):
        w = load.index(min(load))
        assign[w].append(i)
        load[w] += int(lens[i])
    d = tempfile.mkdtemp(prefix="oracle_pool_")
    try:
        np.save(os.path.join(d, "k.npy"), rep.k[0][used])
        np.save(os.path.join(d, "v.npy"), rep.v[0][used])
        np.save(os.path.join(d, "tab.npy"), ctab)
        np.save(os.path.join(d, "lens.npy"), np.asarray(lens, dtype=np.int64))
        np.save(os.path.join(d, "q.npy"), np.asarray(q))
        with open(os.path.join(d, "meta.json"), "w") as f:
            json.dump({"assign": assign, "block_size": B, "scale": sc.scale, "reps": reps}, f)
        return _pool_elapsed(d, procs)
    finally:
        shutil.rmtree(d, ignore_errors=True)


def _pool_elapsed(d, procs):
    """Start one oracle worker per core on the sample in directory d
    (tests/_oracle_pool.py), release them together once all are ready, and
    return the slowest one's seconds."""
    worker = os.path.join(ROOT, "tests", "_oracle_pool.py")
    ps = [subprocess.Popen([sys.executable, worker, d, str(w)], stdin=subprocess.PIPE, stdout=subprocess.PIPE,
                           text=True) for w in range(procs)]
    try:
        for p_ in ps:
            if p_.stdout.readline().strip() != "ready":
                raise RuntimeError("oracle worker failed to start")
        for p_ in ps:
            p_.stdin.write("go\n")
            p_.stdin.flush()
        elapsed = [json.loads(p_.stdout.readline())["elapsed"] for p_ in ps]
    finally:
        for p_ in ps:
            if p_.poll() is None:
                p_.wait(timeout=600)
    return max(elapsed)


def _prefill_oracle_time_procs(sc, rows, procs, reps):
    """Seconds the oracle takes to compute the last `rows` new positions of
    sequence 0 `reps` times on `procs` host cores at once: each worker
    process takes a contiguous share of the rows (as one chunk at their
    positions) over the sequence's whole context."""
    import shutil
    q, kc, vc, tables, _, ctx = _prefill_oracle_sample(sc, 0, rows)
    first_pos = int(ctx[0]) - rows                    # position of sampled row 0
    # shares of equal work: row r attends to first_pos + r + 1 keys
    work = np.cumsum(np.arange(first_pos + 1, first_pos + rows + 1, dtype=np.float64))
    cuts = [0] + [int(np.searchsorted(work, work[-1] * w / procs)) for w in range(1, procs)] + [rows]
    d = tempfile.mkdtemp(prefix="oracle_pool_")
    try:
        np.save(os.path.join(d, "k.npy"), kc)
        np.save(os.path.join(d, "v.npy"), vc)
        np.save(os.path.join(d, "tab.npy"), tables)
        np.save(os.path.join(d, "q.npy"), q)
        with open(os.path.join(d, "meta.json"), "w") as f:
            json.dump({"mode": "prefill", "assign": [[cuts[w], cuts[w + 1]] for w in range(procs)],
                       "block_size": sc.block_size, "scale": sc.scale, "reps": reps, "first_pos": first_pos}, f)
        return _pool_elapsed(d, procs)
    finally:
        shutil.rmtree(d, ignore_errors=True)


def host_threads():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _cpu_leg(sc, budget_s, procs):
    """The oracle as it stands on a bounded sample: the first sequences of
    the workload, as many as fit about budget_s on `procs` cores, repeated
    while a pass takes under half of it."""
    def timed(rep, tab, lens, q, reps):
        if procs <= 1:
            return sum(_oracle_time(sc, rep, tab, lens, q) for _ in range(reps))
        return _oracle_time_procs(sc, rep, tab, lens, q, procs, reps)

    n = min(len(sc.decode_seqs), max(1, procs))
    rep, tab, lens, q = _oracle_sample(sc, list(range(n)))
    t = timed(rep, tab, lens, q, 1)
    while t < budget_s / 2 and n < len(sc.decode_seqs):
        n = min(len(sc.decode_seqs), max(n + 1, int(n * min(8.0, budget_s / max(t, 1e-3)))))
        rep, tab, lens, q = _oracle_sample(sc, list(range(n)))
        t = timed(rep, tab, lens, q, 1)
    reps = 1
    if t < budget_s / 2:
        reps = max(1, int(budget_s / 2 / max(t, 1e-3)))
        t = timed(rep, tab, lens, q, reps)
    dec_bytes, _ = algorithmic_bytes(sc, lens, 0)
    value = reps * dec_bytes / t / 1e9
    sample = ("fp64 oracle decode of the first %d of %d sequences (%d positions, all %d query heads) of %s, "
              "layer 0, %d time(s), %.1f s, %s" % (n, len(sc.decode_seqs), int(np.sum(lens)), sc.n_q_heads,
                                                   sc.name, reps, t, "1 thread" if procs <= 1 else
                                                   "%d worker processes at once, whole sequences each" % procs))
    return value, sample, t


def cpu_baseline(sc, budget_s):
    """The oracle as it stands, on every host core at once (one worker
    process per core) and on one core; each leg gets about half the
    budget."""
    procs = host_threads()
    v1, s1, _ = _cpu_leg(sc, budget_s / 2, 1)
    line = {"value": round(v1, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": s1}
    if procs > 1:
        try:
            vn, sn, _ = _cpu_leg(sc, budget_s / 2, procs)
        except Exception as e:                 # the worker pool is a baseline, not the measurement
            line["all_cores_failed"] = "%s: %s" % (type(e).__name__, e)
            return line
        line = {"value": round(vn, 4), "unit": UNIT, "cores": procs, "kind": "oracle", "sample": sn,
                "single_thread": {"value": round(v1, 4), "cores": 1, "sample": s1},
                "speedup_all_cores": round(vn / v1, 2)}
    return line


def run_reference(args, world, rank):
    if rank != 0:
        return None
    sc = workload_scenario(args, args.seed)
    threads = host_threads()
    per_step = max(1, args.ref_seqs_per_step or threads)
    samples = []
    S = len(sc.decode_seqs)
    for i in range(args.warmup + args.steps):
        seqs = [(i * per_step + j) % S for j in range(per_step)]
        rep, tab, lens, q = _oracle_sample(sc, seqs)
        t = (_oracle_time_procs(sc, rep, tab, lens, q, threads, 1) if threads > 1 else
             _oracle_time(sc, rep, tab, lens, q))
        if i >= args.warmup:
            samples.append((t, algorithmic_bytes(sc, lens, 0)[0], len(seqs)))
    tot_t = sum(s[0] for s in samples)
    tot_b = sum(s[1] for s in samples)
    value = tot_b / tot_t / 1e9
    desc = ("fp64 oracle decode, %d sequence(s) of %s per step (rotating), layer 0, all %d query heads, "
            "%d worker process(es) at once, whole sequences each" % (per_step, sc.name, sc.n_q_heads, threads))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / len(samples) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": sc.name, "num_seqs_per_step": per_step},
            "seqs_per_s": round(sum(s[2] for s in samples) / tot_t, 3),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(PREFILL_WORKLOADS) + ["swap_8b", "cache_ops_8b"],
                   default="batch64_8b")
    p.add_argument("--block-size", type=int, default=16)
    p.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                   help="cache element type of the decode workloads (fp8: E4M3 with per-cache scales)")
    p.add_argument("--partition", type=int, default=0, help="positions per partition (0 = library default)")
    p.add_argument("--layers", type=int, default=0,
                   help="layers of the mixed_batch step (0 = all 32: 32 x (reshape_and_cache + pa_decode))")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--ref-seqs-per-step", type=int, default=0,
                   help="sequences the reference arm decodes per step (0 = one per host core)")
    args = p.parse_args(argv)
    world, rank, local = dist_env()
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    prefill = args.workload in PREFILL_WORKLOADS
    if args.workload == "cache_ops_8b":
        if args.impl == "reference":
            line = None
            if rank == 0:
                from paged_kv_cache_124_gb300 import api
                sc, slots_h, pairs_h, nb = _cache_ops_inputs(args.seed, args.block_size, api)
                cb = cache_ops_cpu_baseline(sc, slots_h, pairs_h, nb, args.cpu_seconds)
                line = {"impl": "reference", "metric": CACHE_OPS_METRIC, "value": cb["value"], "unit": "GB/s",
                        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bit copies)", "data": "synthetic",
                        "config": {"workload": "cache_ops_8b"}, "cpu_baseline": cb,
                        "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        else:
            line = run_cache_ops_ours(args, world, rank, local)
    elif args.workload == "swap_8b":
        if args.impl == "reference":
            line = None
            if rank == 0:
                cb = swap_cpu_baseline(I.batch64_8b(args.seed, args.block_size), args.cpu_seconds)
                line = {"impl": "reference", "metric": SWAP_METRIC, "value": cb["value"], "unit": "GB/s",
                        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bytes moved)", "data": "synthetic",
                        "config": {"workload": "swap_8b"}, "cpu_baseline": cb,
                        "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        else:
            line = run_swap_ours(args, world, rank, local)
    elif args.impl == "reference":
        line = (run_prefill_reference if prefill else run_reference)(args, world, rank)
    else:
        line = (run_prefill_ours if prefill else run_ours)(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
