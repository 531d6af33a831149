"""Seeded synthetic inputs for the paged decode workloads.

This module only draws random numbers and writes down workload scenarios:
tensor values, context lengths, physical-placement permutations and the
sequence of block-manager operations (allocate / fork / append / free) that a
scenario performs.  It holds none of the attention, address-translation,
scatter or copy arithmetic; both the CUDA path and the CPU oracle replay the
same scenario with their own code.  The only arithmetic here is pool sizing
(how many blocks a pool has), which is part of a scenario's definition.

Every draw comes from an explicitly seeded generator that it owns (never the
global one), so every side that draws on the CPU sees the same bits.  Large
multi-layer workloads may draw their keys and values on the device with a
seeded device generator instead; a side that compares against those copies
the drawn tensors back rather than drawing them again.  Tensor values are
N(0, 1) rounded to bf16.
"""

import dataclasses
import math
from typing import List, Tuple

import numpy as np
import torch

NAN_BF16_BITS = 0x7FC1      # quiet-NaN bf16 pattern used to pre-fill pools


def bf16_normal(shape, seed):
    """N(0, 1) samples rounded to bf16 (round-to-nearest-even), CPU tensor."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def bf16_bits(t):
    """uint16 NumPy view of a CPU bf16 tensor's bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def nan_pool(shape, device="cpu"):
    """A bf16 tensor whose every element is the NaN sentinel pattern."""
    return torch.full(shape, NAN_BF16_BITS, dtype=torch.int16, device=device).view(torch.bfloat16)


def permutation(n, seed):
    return np.random.default_rng(int(seed)).permutation(int(n)).astype(np.int32)


def uniform_ints(n, lo, hi, seed):
    """n integers uniform on [lo, hi] inclusive."""
    return np.random.default_rng(int(seed)).integers(lo, hi + 1, size=n).astype(np.int64)


def lognormal_ints(n, median, sigma, lo, hi, seed):
    """n integers from a lognormal with the given median and log-space sigma,
    rounded to nearest and clipped to [lo, hi]."""
    x = np.random.default_rng(int(seed)).lognormal(mean=math.log(median), sigma=sigma, size=n)
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


# ----------------------------------------------------------------------------
# Scenarios
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Scenario:
    """One workload: shapes plus the block-manager operations that build its
    caches.  ops is a list of tuples:
        ("free_order", int32 array)   blocks leave the free list from its end
        ("alloc", seq, n_tokens)      prefill of n_tokens (written afterwards)
        ("fork", parent, child)
        ("append", seq)               one decode token for seq
        ("step",)                     end of one engine step (flush writes)
        ("free", seq)
    decode_seqs lists the sequences decoded at the end, in batch order."""
    name: str
    n_q_heads: int
    n_kv_heads: int
    d_head: int
    block_size: int
    num_blocks: int
    n_layers: int
    ops: List[Tuple]
    decode_seqs: List[int]
    seed: int

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d_head)


def _blocks(n_tokens, block_size):
    return -(-int(n_tokens) // block_size)


def tiny_gqa(seed=0):
    """4 sequences with prompts {1, 15, 16, 37}, 4 query / 2 KV heads, d=64,
    B=16, a 32-block pool handed out in a seeded random order; one decode
    token per sequence (contexts {2, 16, 17, 38} at decode)."""
    lens = [1, 15, 16, 37]
    ops = [("free_order", permutation(32, seed))]
    ops += [("alloc", i, n) for i, n in enumerate(lens)]
    ops += [("append", i) for i in range(4)] + [("step",)]
    return Scenario("tiny_gqa_s4_h4x2_d64_b16", 4, 2, 64, 16, 32, 1, ops, list(range(4)), seed)


def decode_batch(num_seqs, lo, hi, block_size=16, seed=0, n_q_heads=32, n_kv_heads=8,
                 d_head=128, n_layers=1, pool_margin=0.10, name=None):
    """num_seqs sequences whose decode context is uniform on [lo, hi]: prefill
    context-1 tokens, then one decode token each.  The pool has the blocks the
    batch needs plus pool_margin, handed out in a seeded random order."""
    ctx = uniform_ints(num_seqs, lo, hi, seed + 1)
    need = sum(_blocks(c, block_size) for c in ctx)
    nb = int(math.ceil(need * (1.0 + pool_margin)))
    ops = [("free_order", permutation(nb, seed + 2))]
    ops += [("alloc", i, int(c) - 1) for i, c in enumerate(ctx) if c > 1]
    ops += [("alloc", i, 1) for i, c in enumerate(ctx) if c <= 1]
    ops += [("append", i) for i, c in enumerate(ctx) if c > 1] + [("step",)]
    return Scenario(name or f"decode_s{num_seqs}_ctx{lo}-{hi}_b{block_size}", n_q_heads, n_kv_heads,
                    d_head, block_size, nb, n_layers, ops, list(range(num_seqs)), seed)


def batch64_8b(seed=0, block_size=16):
    """8B-shaped decode batch: 64 sequences, contexts uniform on [512, 4096],
    32 query / 8 KV heads, d=128, pool = needed blocks + 10%, random placement."""
    return decode_batch(64, 512, 4096, block_size, seed, name=f"batch64_8b_ctx512-4096_b{block_size}")


def long_context(seed=0, block_size=16, num_seqs=8, context=32768):
    """Long-context split path: num_seqs sequences of `context` tokens."""
    return decode_batch(num_seqs, context, context, block_size, seed,
                        name=f"long_s{num_seqs}_ctx{context}_b{block_size}")


def cow_sampling(seed=0, n_prompts=16, prompt_len=2003, n_samples=8, max_new=64, block_size=16):
    """Parallel sampling: n_prompts prompts of prompt_len tokens, each forked
    into n_samples sequences (the prompt's own sequence plus n_samples-1
    forks) sharing the prompt's blocks; every sample then appends U{1..max_new}
    tokens, one per engine step.  Sequence ids: prompt p, sample j ->
    p * n_samples + j (j = 0 is the original)."""
    new = uniform_ints(n_prompts * n_samples, 1, max_new, seed + 1)
    shared_full = prompt_len // block_size          # prompt blocks never copied
    need = n_prompts * _blocks(prompt_len, block_size) + \
        sum(_blocks(prompt_len + int(n), block_size) - shared_full for n in new)
    nb = int(math.ceil(need * 1.10))
    ops = [("free_order", permutation(nb, seed + 2))]
    for p in range(n_prompts):
        ops.append(("alloc", p * n_samples, prompt_len))
    ops.append(("step",))
    for p in range(n_prompts):
        for j in range(1, n_samples):
            ops.append(("fork", p * n_samples, p * n_samples + j))
    for step in range(max_new):
        any_append = False
        for sid in range(n_prompts * n_samples):
            if new[sid] > step:
                ops.append(("append", sid))
                any_append = True
        if any_append:
            ops.append(("step",))
    return Scenario(f"cow_p{n_prompts}x{n_samples}_len{prompt_len}_b{block_size}", 32, 8, 128,
                    block_size, nb, 1, ops, list(range(n_prompts * n_samples)), seed)


def mixed_batch(seed=0, block_size=16, num_seqs=256, n_layers=32, median=700, sigma=1.0,
                lo=1, hi=16384, occupancy=0.90):
    """Continuous-batching decode step: num_seqs sequences with lognormal
    context lengths (median, sigma, clipped to [lo, hi]), n_layers layers, a
    pool sized so the batch fills `occupancy` of it after a seeded churn of
    filler sequences (allocated and released around the real ones) has
    scattered the free list."""
    rng = np.random.default_rng(seed + 3)
    ctx = lognormal_ints(num_seqs, median, sigma, lo, hi, seed + 1)
    need = sum(_blocks(c, block_size) for c in ctx)
    nb = int(math.ceil(need / occupancy))
    ops = [("free_order", permutation(nb, seed + 2))]
    free = nb
    fillers = {}
    next_filler = 10 ** 6
    # fillers take about half of the pool first
    while free > nb // 2:
        n = int(rng.integers(1, 64 * block_size))
        b = _blocks(n, block_size)
        if b > free - nb // 2:
            break
        ops.append(("alloc", next_filler, n))
        fillers[next_filler] = b
        free -= b
        next_filler += 1
    for i, c in enumerate(ctx):
        c = int(c)
        prompt = max(c - 1, 1)
        b_need = _blocks(c, block_size)
        while free < b_need + 1 and fillers:
            victim = list(fillers)[int(rng.integers(len(fillers)))]
            ops.append(("free", victim))
            free += fillers.pop(victim)
        ops.append(("alloc", i, prompt))
        free -= _blocks(prompt, block_size)
        if rng.random() < 0.5 and fillers:
            victim = list(fillers)[int(rng.integers(len(fillers)))]
            ops.append(("free", victim))
            free += fillers.pop(victim)
    for victim in list(fillers):
        ops.append(("free", victim))
    ops.append(("step",))
    ops += [("append", i) for i, c in enumerate(ctx) if c > 1] + [("step",)]
    return Scenario(f"mixed_s{num_seqs}_lognorm{median}_L{n_layers}_b{block_size}", 32, 8, 128,
                    block_size, nb, n_layers, ops, list(range(num_seqs)), seed)


# ----------------------------------------------------------------------------
# Token data: a deterministic function of (seed, kind, layer, index), so that
# each side can draw exactly the tensors it needs.
# ----------------------------------------------------------------------------

def _mix(seed, kind, a, b):
    return (int(seed) * 1000003 + kind * 7919 + int(a) * 104729 + int(b) * 15485863) % (1 << 62)


def _normal(shape, seed, device):
    if str(device) == "cpu":
        return bf16_normal(shape, seed)
    g = torch.Generator(device=device).manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)


def prefill_kv(seed, layer, seq, n_tokens, n_kv_heads, d_head, device="cpu"):
    """Keys and values [n_tokens, n_kv_heads, d_head] of a sequence's prompt
    in one layer."""
    k = _normal((n_tokens, n_kv_heads, d_head), _mix(seed, 1, layer, seq), device)
    v = _normal((n_tokens, n_kv_heads, d_head), _mix(seed, 2, layer, seq), device)
    return k, v


def append_kv(seed, layer, step, n_tokens, n_kv_heads, d_head, device="cpu"):
    """Keys and values of the n_tokens positions appended in engine step
    `step` (one per appending sequence, in operation order)."""
    k = _normal((n_tokens, n_kv_heads, d_head), _mix(seed, 3, layer, step), device)
    v = _normal((n_tokens, n_kv_heads, d_head), _mix(seed, 4, layer, step), device)
    return k, v


def decode_q(seed, layer, num_seqs, n_q_heads, d_head, device="cpu"):
    """Queries [num_seqs, n_q_heads, d_head] of one decode step in one layer."""
    return _normal((num_seqs, n_q_heads, d_head), _mix(seed, 5, layer, 0), device)


# ----------------------------------------------------------------------------
# Prefix-cache workloads: prompts built from shared documents, and KV that is
# a deterministic function of the whole prefix up to each position, so that a
# reused block is right only if it holds exactly its own prefix's KV.
# ----------------------------------------------------------------------------

_M64 = (1 << 64) - 1


def _splitmix(x):
    x = (x + 0x9E3779B97F4A7C15) & _M64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & _M64
    return x ^ (x >> 31)


def prompt_documents(seed, lengths, vocab=32000):
    """Shared documents (system prompts, retrieved passages): token id lists
    of the given lengths."""
    rng = np.random.default_rng(int(seed))
    return [[int(t) for t in rng.integers(0, vocab, size=int(n))] for n in lengths]


def prefix_digests(tokens):
    """One 64-bit digest per position, each covering every token up to and
    including that position."""
    out, h = [], 0x243F6A8885A308D3
    for t in tokens:
        h = _splitmix(h ^ (int(t) & 0xFFFFFFFF))
        out.append(h)
    return out


def prefix_kv(seed, layer, tokens, start, end, n_kv_heads, d_head):
    """Keys and values [end - start, n_kv_heads, d_head] (CPU bf16) for
    positions start .. end-1 of a token sequence: each position's rows are
    uniform on [-2, 2), drawn from a counter generator keyed by the digest of
    its whole prefix, the layer and the seed."""
    dig = np.array(prefix_digests(tokens[:end])[start:], dtype=np.uint64)
    n = n_kv_heads * d_head
    ctr = np.arange(2 * n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        x = dig[:, None] ^ np.uint64((int(seed) * 0x632BE59BD9B4E019 + int(layer) * 0x8CB92BA72F3D8DD7) & _M64)
        x = x + ctr[None, :] * np.uint64(0x9E3779B97F4A7C15)
        x = (x ^ (x >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        x = (x ^ (x >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        x = x ^ (x >> np.uint64(31))
    u = (x >> np.uint64(40)).astype(np.float64) / float(1 << 24) * 4.0 - 2.0
    t = torch.from_numpy(u.astype(np.float32)).to(torch.bfloat16)
    t = t.view(len(dig), 2, n_kv_heads, d_head)
    return t[:, 0].contiguous(), t[:, 1].contiguous()


# ----------------------------------------------------------------------------
# Prefill workloads: each sequence has ctx positions, the last n of them new
# (a whole prompt when n = ctx, a chunk over a cached prefix otherwise).
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class PrefillScenario:
    name: str
    n_q_heads: int
    n_kv_heads: int
    d_head: int
    block_size: int
    ctxs: List[int]
    news: List[int]
    num_blocks: int
    free_order: np.ndarray        # block manager free list (seeded random placement)
    seed: int

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d_head)

    @property
    def query_start(self):
        return np.concatenate([[0], np.cumsum(self.news)]).astype(np.int32)


def _prefill_scenario(name, seed, block_size, ctxs, news, n_q_heads=32, n_kv_heads=8, d_head=128):
    nblk = [_blocks(c, block_size) for c in ctxs]
    num_blocks = int(math.ceil(sum(nblk) * 1.1)) + 1
    return PrefillScenario(name, n_q_heads, n_kv_heads, d_head, block_size, [int(c) for c in ctxs],
                           [int(n) for n in news], num_blocks, permutation(num_blocks, seed + 17), seed)


def prefill_prompts(seed=0, block_size=16, num_seqs=16, prompt_len=2003):
    """Whole-prompt prefill: the 16 prompts of 2,003 tokens of the parallel
    sampling workload, before they are forked."""
    return _prefill_scenario("prefill_prompts_8b", seed, block_size, [prompt_len] * num_seqs, [prompt_len] * num_seqs)


def chunked_prefill(seed=0, block_size=16, num_seqs=8, chunk=512, lo=2048, hi=8192):
    """Chunked prefill: a 512-token chunk per sequence on top of a cached
    prefix of U[2048, 8192] positions."""
    prefix = uniform_ints(num_seqs, lo, hi, seed + 5)
    return _prefill_scenario("chunked_prefill_8b", seed, block_size, [int(p) + chunk for p in prefix],
                             [chunk] * num_seqs)


def prefill_pool(sc, device):
    """K and V pools [num_blocks, Hkv, B, D] bf16 with N(0,1) values in every
    slot (the cached prefix, and placeholders where the new positions will be
    written); drawn on `device`."""
    shape = (sc.num_blocks, sc.n_kv_heads, sc.block_size, sc.d_head)
    k = _normal(shape, _mix(sc.seed, 6, 0, 0), device)
    v = _normal(shape, _mix(sc.seed, 7, 0, 0), device)
    return k, v


def prefill_q(sc, device):
    """Queries [sum(news), Hq, D] of the new positions."""
    return _normal((int(sum(sc.news)), sc.n_q_heads, sc.d_head), _mix(sc.seed, 8, 0, 0), device)


def prefill_new_kv(sc, device):
    """Keys and values [sum(news), Hkv, D] of the new positions (written into
    the pool by reshape_and_cache before the attention)."""
    T = int(sum(sc.news))
    k = _normal((T, sc.n_kv_heads, sc.d_head), _mix(sc.seed, 9, 0, 0), device)
    v = _normal((T, sc.n_kv_heads, sc.d_head), _mix(sc.seed, 10, 0, 0), device)
    return k, v
