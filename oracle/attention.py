"""Paged attention (single-query decode and causal prefill), restated from
its definition.

Oracle; test infrastructure only.  Everything here is float64 NumPy with
plain loops over sequences, heads and blocks, so that a reader can check it
against the pages line by line.

Definition ([P1] section 1; [P2] section 10): for one query row q and the S
cached key/value rows of its sequence,

    s = scale * q K^T,      a = softmax(s),      o = a V.

The softmax subtracts the score maximum before exponentiating; the common
factor exp(-m) cancels, so the result is unchanged ([P2] section 11, first
paragraph).  With scale = 1/sqrt(d_head) this is the attention formula of
[P1] section 1.

Paging ([P1] section 7; [P2] section 5): position i of a sequence lives in
physical block block_table[i // B] at offset i % B.  Reading the cache means
looping over the sequence's blocks b = 0 .. ceil(S/B) - 1 and, in the last
one, reading only the positions below S ([P1] section 13, items 2 and 4).

Grouped-query attention ([P1] section 1; [P2] section 7): n_q_heads query
heads share n_kv_heads KV heads.  The pages do not fix which query head reads
which KV head; this oracle takes contiguous groups, query head g reading KV
head g // (n_q_heads / n_kv_heads).

A context length of 0 yields an all-zero output row (the pages forbid empty
prompts, so this is a defensive convention of the interface).
"""

import numpy as np


def bf16_to_f64(bits):
    """Decode bf16 bit patterns (uint16) to float64 exactly.

    A bf16 value is the upper 16 bits of an IEEE-754 binary32 value, so the
    pattern shifted left by 16 and read as binary32 is the value itself."""
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):     # NaN payloads stay NaN
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def translate(i, block_size, block_table_row):
    """Address translation of one token position ([P1] section 7):
    logical block floor(i / B), offset i % B, physical id from the table."""
    logical_block = i // block_size
    offset = i % block_size
    return int(block_table_row[logical_block]), offset


def gather_kv(k_cache, v_cache, block_table_row, context_len, block_size):
    """Gather one sequence's keys and values into contiguous arrays.

    k_cache, v_cache: [num_blocks, n_kv_heads, block_size, d_head], float64,
    or uint16 bf16 bit patterns (decoded exactly as they are gathered).
    Returns K, V of shape [n_kv_heads, context_len, d_head] in logical token
    order: the contiguous layout of [P1] section 12 for one sequence.

    Loops over the sequence's blocks b = 0 .. ceil(S/B) - 1; the last block
    contributes only its valid positions ([P1] section 13, items 2 and 4;
    [P1] section 20, the valid length of the final block)."""
    n_kv_heads, d_head = k_cache.shape[1], k_cache.shape[3]
    to_f64 = bf16_to_f64 if k_cache.dtype == np.uint16 else (lambda x: x)
    K = np.empty((n_kv_heads, context_len, d_head), dtype=np.float64)
    V = np.empty((n_kv_heads, context_len, d_head), dtype=np.float64)
    n_blocks = -(-context_len // block_size)
    for b in range(n_blocks):
        phys, _ = translate(b * block_size, block_size, block_table_row)
        valid = min(block_size, context_len - b * block_size)
        K[:, b * block_size: b * block_size + valid, :] = to_f64(k_cache[phys, :, :valid, :])
        V[:, b * block_size: b * block_size + valid, :] = to_f64(v_cache[phys, :, :valid, :])
    return K, V


def softmax_attention(q, K, V, scale):
    """Textbook attention of one query row over contiguous K [S, d], V [S, d]:
    scores, max-subtracted softmax, weighted sum of value rows."""
    s = scale * (K @ q)
    m = s.max()
    e = np.exp(s - m)
    a = e / e.sum()
    return a @ V


def kv_head_of(q_head, n_q_heads, n_kv_heads):
    """KV head read by a query head: contiguous groups of G = Hq / Hkv."""
    return q_head // (n_q_heads // n_kv_heads)


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale, block_size):
    """Decode attention for a batch, through the block tables.

    q:            [S, n_q_heads, d_head] float64 (or uint16 bf16 bits)
    k/v_cache:    [num_blocks, n_kv_heads, block_size, d_head] float64
                  (or uint16 bf16 bits)
    block_tables: [S, max_blocks_per_seq] integer
    context_lens: [S] integer
    returns       [S, n_q_heads, d_head] float64
    """
    if q.dtype == np.uint16:
        q = bf16_to_f64(q)
    S, n_q_heads, d_head = q.shape
    n_kv_heads = k_cache.shape[1]
    assert n_q_heads % n_kv_heads == 0
    out = np.zeros((S, n_q_heads, d_head), dtype=np.float64)
    for s in range(S):
        ctx = int(context_lens[s])
        if ctx <= 0:
            continue
        K, V = gather_kv(k_cache, v_cache, block_tables[s], ctx, block_size)
        for g in range(n_q_heads):
            h = kv_head_of(g, n_q_heads, n_kv_heads)
            out[s, g] = softmax_attention(q[s, g], K[h], V[h], scale)
    return out


def dense_decode(q, K_dense, V_dense, context_lens, scale):
    """The same attention over a contiguous cache [S, n_kv_heads, max_len, d]
    ([P1] section 12, contiguous layout).  Paged and dense results must agree
    ([P1] section 20, paged-versus-dense check; [P2] section 10)."""
    S, n_q_heads, d_head = q.shape
    n_kv_heads = K_dense.shape[1]
    out = np.zeros((S, n_q_heads, d_head), dtype=np.float64)
    for s in range(S):
        ctx = int(context_lens[s])
        if ctx <= 0:
            continue
        for g in range(n_q_heads):
            h = kv_head_of(g, n_q_heads, n_kv_heads)
            out[s, g] = softmax_attention(q[s, g], K_dense[s, h, :ctx], V_dense[s, h, :ctx], scale)
    return out


# ----------------------------------------------------------------------------
# Prefill: many query positions per sequence, causal ([P2] sections 4 and 8)
# ----------------------------------------------------------------------------

def paged_prefill(q, k_cache, v_cache, block_tables, query_start, context_lens, scale, block_size):
    """Causal attention of the new positions of each sequence.

    Sequence s has context length C = context_lens[s]; its last
    n = query_start[s+1] - query_start[s] positions are new.  New position
    p = C - n + i is query row query_start[s] + i and attends to positions
    0 .. p of its sequence only: during prefill a token cannot depend on the
    tokens after it ([P2] section 4, causal attention; [P2] section 8, n
    queries against up to n keys).  Keys and values are read through the
    block table exactly as for decode.

    q: [T, n_q_heads, d_head] float64 or uint16 bf16 bits; returns
    [T, n_q_heads, d_head] float64 (rows not covered by any sequence are 0).
    """
    if q.dtype == np.uint16:
        q = bf16_to_f64(q)
    T, n_q_heads, d_head = q.shape
    n_kv_heads = k_cache.shape[1]
    out = np.zeros((T, n_q_heads, d_head), dtype=np.float64)
    for s in range(len(context_lens)):
        C = int(context_lens[s])
        row0, n = int(query_start[s]), int(query_start[s + 1]) - int(query_start[s])
        if n <= 0:
            continue
        K, V = gather_kv(k_cache, v_cache, block_tables[s], C, block_size)
        for i in range(n):
            p = C - n + i
            for g in range(n_q_heads):
                h = kv_head_of(g, n_q_heads, n_kv_heads)
                out[row0 + i, g] = softmax_attention(q[row0 + i, g], K[h, :p + 1], V[h, :p + 1], scale)
    return out


# ----------------------------------------------------------------------------
# Split computation and exact merge ([P2] sections 10 and 11)
# ----------------------------------------------------------------------------

def page_sums(scores, V):
    """Unnormalised per-page sums of [P2] section 10: Z = sum_i exp(s_i),
    N = sum_i exp(s_i) v_i.  The output is (sum of N) / (sum of Z)."""
    e = np.exp(np.asarray(scores, dtype=np.float64))
    return e @ np.asarray(V, dtype=np.float64), e.sum()


def block_summary(scores, V):
    """Stable per-block summary of [P2] section 11: m_b = max of the block's
    scores, z_b = sum exp(s_i - m_b), u_b = sum exp(s_i - m_b) v_i."""
    s = np.asarray(scores, dtype=np.float64)
    m = s.max()
    e = np.exp(s - m)
    return m, e.sum(), e @ np.asarray(V, dtype=np.float64)


def merge_summaries(summaries):
    """Exact merge of block summaries ([P2] section 11): m = max_b m_b,
    z = sum_b exp(m_b - m) z_b, u = sum_b exp(m_b - m) u_b.  Returns (m, z, u);
    the attention output is u / z."""
    m = max(sb[0] for sb in summaries)
    z = 0.0
    u = 0.0
    for m_b, z_b, u_b in summaries:
        w = np.exp(m_b - m)
        z = z + w * z_b
        u = u + w * np.asarray(u_b, dtype=np.float64)
    return m, z, u


def partition_summaries(q_row, K, V, scale, partition_size):
    """Split one (sequence, query head) problem into consecutive partitions
    of partition_size positions and summarise each ([P1] section 13: split
    implementations hand each segment of the sequence's blocks to a different
    worker and keep partial sums plus reduction statistics; [P2] section 11
    gives the statistics).  Returns a list of (m_b, z_b, u_b)."""
    s = scale * (K @ q_row)
    out = []
    for start in range(0, len(s), partition_size):
        stop = min(start + partition_size, len(s))
        out.append(block_summary(s[start:stop], V[start:stop]))
    return out
