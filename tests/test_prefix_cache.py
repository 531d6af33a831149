"""Automatic prefix caching in the block manager.

The oracle restatement is pinned by the pages' traces (tests/golden/
p2_prefix_cache.json) and by a content invariant that does not depend on how
the cache is indexed: if every position's KV is a function of its whole
prefix ("PagedAttention in vLLM: scattered memory, exact attention",
section 6), then after any sequence of admissions, appends, copy-on-write
copies, forks and releases, every live sequence must find in its block
table exactly the KV of its own prefix.  The C++ manager is then checked
against the oracle operation by operation, and against the same traces
and invariant, through the C ABI."""
import numpy as np
import pytest

from oracle import allocator as AL
from _golden import load

api = pytest.importorskip("paged_kv_cache_124_gb300.api")

STATUS_MAP = {AL.OK: api.PA_OK, AL.FAIL_NO_BLOCKS: api.PA_FAIL_NO_BLOCKS, AL.ERR_INVALID_ARG: api.PA_ERR_INVALID_ARG,
              AL.ERR_UNKNOWN_SEQ: api.PA_ERR_UNKNOWN_SEQ, AL.ERR_DUPLICATE_SEQ: api.PA_ERR_DUPLICATE_SEQ,
              AL.ERR_SWAPPED: api.PA_ERR_SWAPPED}
TRACES = {k: v for k, v in load("p2_prefix_cache.json").items() if not k.startswith("_")}


class _OracleView:
    """Uniform interface over the oracle, with the C ABI's status codes."""

    def __init__(self, nb, bs):
        self.m = AL.RefAllocator(nb, bs)

    def enable(self, on):
        return STATUS_MAP[self.m.enable_prefix_caching(on)]

    def tokens(self, s, ids):
        st, hit = self.m.allocate_tokens(s, ids)
        return STATUS_MAP[st], hit

    def alloc(self, s, n):
        return STATUS_MAP[self.m.allocate(s, n)]

    def append_token(self, s, t):
        r = self.m.append_token(s, t)
        return (STATUS_MAP[r[0]],) + tuple(r[1:])

    def append_slot(self, s):
        r = self.m.append_slot(s)
        return (STATUS_MAP[r[0]],) + tuple(r[1:])

    def fork(self, p, c):
        return STATUS_MAP[self.m.fork(p, c)]

    def free(self, s):
        return STATUS_MAP[self.m.free(s)]

    def table(self, s):
        return list(self.m.block_tables[s])

    def ref(self, b):
        return self.m.ref_counts[b]

    def num_free(self):
        return self.m.num_free()

    def num_cached(self):
        return self.m.num_cached()

    def cached_list(self):
        return self.m.cached_list()

    def enable_swap(self, n):
        return STATUS_MAP[self.m.enable_swap(n)]

    def swap_out(self, seqs):
        st, pairs = self.m.swap_out(seqs)
        return STATUS_MAP[st], [tuple(p) for p in pairs]

    def swap_in(self, seqs):
        st, pairs = self.m.swap_in(seqs)
        return STATUS_MAP[st], [tuple(p) for p in pairs]

    def num_free_host(self):
        return len(self.m.host_free)

    def is_swapped(self, s):
        return -1 if s not in self.m.block_tables else int(s in self.m.swapped)


class _AbiView:
    def __init__(self, nb, bs):
        self.m = api.BlockAllocator(nb, bs)

    def enable(self, on):
        return self.m.enable_prefix_caching(on)

    def tokens(self, s, ids):
        return self.m.allocate_tokens(s, ids)

    def alloc(self, s, n):
        return self.m.allocate(s, n)

    def append_token(self, s, t):
        return self.m.append_token(s, t)

    def append_slot(self, s):
        return self.m.append_slot(s)

    def fork(self, p, c):
        return self.m.fork(p, c)

    def free(self, s):
        return self.m.free(s)

    def table(self, s):
        return self.m.block_table(s)

    def ref(self, b):
        return self.m.ref_count(b)

    def num_free(self):
        return self.m.num_free()

    def num_cached(self):
        return self.m.num_cached()

    def cached_list(self):
        return self.m.cached_list()

    def enable_swap(self, n):
        return self.m.enable_swap(n)

    def swap_out(self, seqs):
        st, pairs = self.m.swap_out(seqs)
        return st, [tuple(int(v) for v in p) for p in pairs]

    def swap_in(self, seqs):
        st, pairs = self.m.swap_in(seqs)
        return st, [tuple(int(v) for v in p) for p in pairs]

    def num_free_host(self):
        return self.m.num_free_host()

    def is_swapped(self, s):
        return self.m.is_swapped(s)


VIEWS = {"oracle": _OracleView, "abi": _AbiView}


def _run_trace(view_cls, tr):
    m = view_cls(tr["num_blocks"], tr["block_size"])
    assert m.enable(tr["caching"]) == 0
    for op in tr["ops"]:
        kind = op[0]
        if kind == "tokens":
            assert m.tokens(op[1], op[2]) == (op[3], op[4]), op
        elif kind == "alloc":
            assert m.alloc(op[1], op[2]) == op[3], op
        elif kind == "append_token":
            assert m.append_token(op[1], op[2])[0] == 0, op
        elif kind == "free":
            assert m.free(op[1]) == 0
        elif kind == "check":
            c = op[1]
            for s, t in c.get("table", {}).items():
                assert m.table(int(s)) == t, (s, op)
            for b, r in c.get("refs", {}).items():
                assert m.ref(int(b)) == r, (b, op)
            if "num_cached" in c:
                assert m.num_cached() == c["num_cached"], op
            if "cached_list" in c:
                assert m.cached_list() == c["cached_list"], op
            if "num_free" in c:
                assert m.num_free() == c["num_free"], op
        else:
            raise AssertionError(kind)


@pytest.mark.parametrize("view", sorted(VIEWS))
@pytest.mark.parametrize("name", sorted(TRACES))
def test_golden_prefix_traces(view, name):
    _run_trace(VIEWS[view], TRACES[name])


class _ContentModel:
    """Shadow pool: slot -> the prefix (tuple of token ids) whose KV it holds.
    Written only where the caller would write KV: the positions past the
    cached ones at admission, each appended position, and copy-on-write
    copies of whole blocks."""

    def __init__(self, nb, bs):
        self.B = bs
        self.pool = [None] * (nb * bs)
        self.ids = {}          # seq -> its token ids (anonymous ids for unknown tokens)

    def admit(self, m, s, ids, cached):
        tab = m.table(s)
        self.ids[s] = list(ids)
        for i in range(cached, len(ids)):
            self.pool[tab[i // self.B] * self.B + i % self.B] = tuple(ids[:i + 1])

    def append(self, s, tok, slot, src, dst):
        if src >= 0:
            B = self.B
            self.pool[dst * B:(dst + 1) * B] = self.pool[src * B:(src + 1) * B]
        self.ids[s].append(tok)
        self.pool[slot] = tuple(self.ids[s])

    def check(self, m, live):
        for s in live:
            tab = m.table(s)
            for i in range(len(self.ids[s])):
                got = self.pool[tab[i // self.B] * self.B + i % self.B]
                assert got == tuple(self.ids[s][:i + 1]), (s, i)


def _churn(view_cls, seed, nb, bs, steps=1500, check_every=50):
    """Random admissions from a few shared documents, appends (with and
    without known token ids), forks and releases; checks the content
    invariant and block conservation as it goes.  Returns the manager."""
    rng = np.random.default_rng(seed)
    m = view_cls(nb, bs)
    assert m.enable(True) == 0
    docs = [list(rng.integers(0, 6, size=int(rng.integers(bs, 6 * bs)))) for _ in range(4)]
    cm = _ContentModel(nb, bs)
    live, nxt, anon = set(), 0, -1
    for step in range(steps):
        op = int(rng.integers(0, 10))
        if op <= 2:                                     # admit: document prefix + own suffix
            d = docs[int(rng.integers(0, len(docs)))]
            cut = int(rng.integers(0, len(d) + 1))
            ids = [int(x) for x in d[:cut]] + [int(x) for x in rng.integers(0, 6, size=int(rng.integers(0, 2 * bs)))]
            if not ids:
                ids = [1]
            st, hit = m.tokens(nxt, ids)
            if st == 0:
                assert hit % bs == 0 and hit <= len(ids)
                cm.admit(m, nxt, ids, hit)
                live.add(nxt)
            else:
                assert st == api.PA_FAIL_NO_BLOCKS and hit == 0
            nxt += 1
        elif op == 3 and live:                          # admit with unknown tokens
            n = int(rng.integers(1, 3 * bs))
            if m.alloc(nxt, n) == 0:
                ids = list(range(anon, anon - n, -1))
                anon -= n
                cm.admit(m, nxt, ids, 0)
                live.add(nxt)
            nxt += 1
        elif op in (4, 5, 6) and live:                  # append a known token
            s = int(rng.choice(sorted(live)))
            tok = int(rng.integers(0, 6))
            st, slot, src, dst = m.append_token(s, tok)
            if st == 0:
                cm.append(s, tok, slot, src, dst)
        elif op == 7 and live:                          # append an unknown token
            s = int(rng.choice(sorted(live)))
            st, slot, src, dst = m.append_slot(s)
            if st == 0:
                cm.append(s, anon, slot, src, dst)
                anon -= 1
        elif op == 8 and live:                          # fork
            s = int(rng.choice(sorted(live)))
            if m.fork(s, nxt) == 0:
                cm.ids[nxt] = list(cm.ids[s])
                live.add(nxt)
            nxt += 1
        elif live:                                      # release
            s = int(rng.choice(sorted(live)))
            assert m.free(s) == 0
            live.discard(s)
        if step % check_every == 0 or step == steps - 1:
            cm.check(m, live)
            in_use = set(b for s in live for b in m.table(s))
            assert all(m.ref(b) == 0 for b in m.cached_list())
            assert len(in_use) + m.num_free() + m.num_cached() == nb
    return m, live


@pytest.mark.parametrize("view", sorted(VIEWS))
@pytest.mark.parametrize("seed,nb,bs", [(0, 12, 4), (1, 40, 2), (2, 24, 8), (3, 30, 1)])
def test_content_invariant_under_churn(view, seed, nb, bs):
    m, _ = _churn(VIEWS[view], seed, nb, bs)
    assert m.num_cached() >= 0


@pytest.mark.parametrize("mask", [0xFFFFFFFFFFFFFFFF, 0x3, 0], ids=["hash", "4_buckets", "all_collide"])
@pytest.mark.parametrize("seed,nb,bs", [(5, 16, 4), (6, 48, 8), (7, 20, 2)])
def test_abi_matches_oracle_operation_by_operation(seed, nb, bs, mask):
    """The C++ manager against the oracle's exact (whole token prefix) keys,
    op by op; with the hash that buckets its prefixes cut to 2 bits or to
    none, every lookup meets colliding candidates, and the results must not
    change."""
    rng = np.random.default_rng(seed)
    ref, dut = _OracleView(nb, bs), _AbiView(nb, bs)
    assert dut.m.set_key_mask(mask) == 0
    assert ref.enable(True) == dut.enable(True) == 0
    docs = [[int(x) for x in rng.integers(0, 4, size=5 * bs)] for _ in range(3)]
    seqs = list(range(10))
    for _ in range(3000):
        op = int(rng.integers(0, 8))
        s = int(rng.choice(seqs))
        if op <= 1:
            d = docs[int(rng.integers(0, 3))]
            ids = d[:int(rng.integers(0, len(d)))] + [int(x) for x in rng.integers(0, 4, size=int(rng.integers(0, bs + 2)))]
            if not ids and rng.random() < 0.5:
                ids = [0]
            assert ref.tokens(s, ids) == dut.tokens(s, ids)
        elif op == 2:
            n = int(rng.integers(-1, 3 * bs))
            assert ref.alloc(s, n) == dut.alloc(s, n)
        elif op in (3, 4):
            t = int(rng.integers(0, 4))
            assert ref.append_token(s, t) == dut.append_token(s, t)
        elif op == 5:
            assert ref.append_slot(s) == dut.append_slot(s)
        elif op == 6:
            c = int(rng.choice(seqs))
            assert ref.fork(s, c) == dut.fork(s, c)
        else:
            assert ref.free(s) == dut.free(s)
    assert ref.cached_list() == dut.cached_list()
    assert ref.m.free_blocks == dut.m.free_list()
    assert [ref.ref(b) for b in range(nb)] == [dut.ref(b) for b in range(nb)]
    for s in seqs:
        if s in ref.m.block_tables:
            assert dut.table(s) == ref.table(s)
    st = dut.m.stats()
    assert st["num_cached"] == ref.num_cached()
    assert st["num_prompt_tokens"] == ref.m.num_prompt_tokens
    assert st["num_cached_tokens"] == ref.m.num_cached_tokens
    assert st["num_used"] + st["num_free"] + st["num_cached"] == nb
    # every interned prefix is let go once nothing holds it
    for s_ in seqs:
        assert dut.free(s_) == 0
    assert dut.m.num_prefix_nodes() >= dut.num_cached()
    assert dut.enable(False) == 0
    assert dut.m.num_prefix_nodes() == 0


def test_colliding_keys_never_match_another_prefix():
    """Two prefixes that end in the same block of tokens after different
    first blocks: with every hash colliding (mask 0), the second block of one
    must not be taken for the other's, however their parents' hashes
    compare.  The oracle's keys are whole token prefixes."""
    B = 4
    A_, B_, X, Y = [1, 1, 1, 1], [2, 2, 2, 2], [7, 7, 7, 7], [8, 8, 8, 8]
    for mask in (0xFFFFFFFFFFFFFFFF, 0):
        m = api.BlockAllocator(16, B)
        assert m.set_key_mask(mask) == 0
        assert m.enable_prefix_caching(True) == 0
        assert m.allocate_tokens(1, A_ + X) == (0, 0)
        assert m.allocate_tokens(2, B_ + Y) == (0, 0)
        assert m.allocate_tokens(3, B_ + X + [5]) == (0, B)          # B_ hits, then B_ + X is new
        assert m.block_table(3)[0] == m.block_table(2)[0]
        assert m.block_table(3)[1] not in (m.block_table(1)[1], m.block_table(2)[1])
        assert m.allocate_tokens(4, A_ + X + [6]) == (0, 2 * B)      # the real match is still found
        assert m.block_table(4)[:2] == m.block_table(1)
        assert m.allocate_tokens(5, B_ + X) == (0, 2 * B)            # and the one registered by sequence 3
        assert m.block_table(5) == m.block_table(3)[:2]
        ref = _OracleView(16, B)
        assert ref.enable(True) == 0
        for s_, ids in ((1, A_ + X), (2, B_ + Y), (3, B_ + X + [5]), (4, A_ + X + [6]), (5, B_ + X)):
            ref.tokens(s_, ids)
            assert ref.table(s_) == m.block_table(s_)


def test_key_mask_only_before_use():
    m = api.BlockAllocator(8, 4)
    assert m.enable_prefix_caching(True) == 0
    assert m.allocate_tokens(1, list(range(8))) == (0, 0)
    assert m.set_key_mask(0) == api.PA_ERR_INVALID_ARG          # a sequence exists
    assert m.free(1) == 0
    assert m.set_key_mask(0) == api.PA_ERR_INVALID_ARG          # its prefixes are still cached
    assert m.enable_prefix_caching(False) == 0 and m.num_prefix_nodes() == 0
    assert m.set_key_mask(0) == 0


def test_switching_off_releases_the_cache():
    for view in VIEWS.values():
        m = view(6, 4)
        assert m.enable(True) == 0
        assert m.tokens(1, list(range(12))) == (0, 0)
        assert m.enable(False) == api.PA_ERR_INVALID_ARG       # a sequence exists
        assert m.free(1) == 0 and m.cached_list() == [2, 1, 0]
        assert m.enable(False) == 0
        assert m.num_cached() == 0 and m.num_free() == 6
        assert m.tokens(2, list(range(12))) == (0, 0)           # nothing is remembered
        assert m.table(2) == [0, 1, 2]                           # the newest queued block leaves first


def test_hit_rate_statistic():
    a = api.BlockAllocator(16, 4)
    assert a.enable_prefix_caching(True) == 0
    doc = list(range(100, 116))
    assert a.allocate_tokens(1, doc + [1, 2]) == (0, 0)
    assert a.allocate_tokens(2, doc + [3]) == (0, 16)
    st = a.stats()
    assert st["num_prompt_tokens"] == 35 and st["num_cached_tokens"] == 16
    assert st["prefix_cache_hit_rate"] == pytest.approx(16 / 35)


def test_prefix_argument_errors():
    a = api.BlockAllocator(4, 4)
    assert a.allocate_tokens(1, []) == (api.PA_ERR_INVALID_ARG, 0)
    assert a.allocate_tokens(1, [1, 2]) == (0, 0)
    assert a.allocate_tokens(1, [1, 2]) == (api.PA_ERR_DUPLICATE_SEQ, 0)
    assert a.append_token(9, 1)[0] == api.PA_ERR_UNKNOWN_SEQ
    assert a.enable_prefix_caching(True) == api.PA_ERR_INVALID_ARG
