"""Swap-out/in in the block manager ("PagedAttention: Virtual Memory for the
KV Cache", section 19, item 4).  The oracle is pinned by hand-checked traces
(tests/golden/p1_swap_traces.json) and by a content invariant: with a
shadow payload for device and host blocks, moved exactly along the pairs
the manager returns, every running sequence reads its own prefix's KV on
the device and every swapped one on the host, after any mix of admissions,
appends, forks, releases and swaps.  The C++ manager matches the oracle
operation by operation and satisfies the same traces and invariant."""
import numpy as np
import pytest

from _golden import load
from test_prefix_cache import VIEWS, _AbiView, _OracleView

api = pytest.importorskip("paged_kv_cache_124_gb300.api")
TRACES = {k: v for k, v in load("p1_swap_traces.json").items() if not k.startswith("_")}


def _host_refs(m, b):
    return m.m.host_refs[b] if isinstance(m, _OracleView) else None


def _run(view_cls, tr):
    m = view_cls(tr["num_blocks"], tr["block_size"])
    assert m.enable_swap(tr["num_host_blocks"]) == 0
    for op in tr["ops"]:
        k = op[0]
        if k == "alloc":
            assert m.alloc(op[1], op[2]) == op[3], op
        elif k == "fork":
            assert m.fork(op[1], op[2]) == op[3], op
        elif k == "append":
            assert m.append_slot(op[1])[0] == op[2], op
        elif k in ("out", "in"):
            st, pairs = (m.swap_out if k == "out" else m.swap_in)(op[1])
            assert (st, [list(p) for p in pairs]) == (op[2], op[3]), op
        elif k == "free":
            assert m.free(op[1]) == 0
        elif k == "check":
            c = op[1]
            for q, t in c.get("table", {}).items():
                assert m.table(int(q)) == t, (q, op)
            for b, r in c.get("refs", {}).items():
                assert m.ref(int(b)) == r, (b, op)
            for q, v in c.get("swapped", {}).items():
                assert m.is_swapped(int(q)) == v, (q, op)
            if "host_free" in c:
                hf = m.m.host_free if isinstance(m, _OracleView) else None
                if hf is not None:
                    assert hf == c["host_free"], op
                else:
                    assert m.num_free_host() == len(c["host_free"]), op
            if "free" in c:
                fl = m.m.free_blocks if isinstance(m, _OracleView) else m.m.free_list()
                assert fl == c["free"], op
            for b, r in c.get("host_refs", {}).items():
                if isinstance(m, _OracleView):
                    assert m.m.host_refs[int(b)] == r, (b, op)
        else:
            raise AssertionError(k)


@pytest.mark.parametrize("view", sorted(VIEWS))
@pytest.mark.parametrize("name", sorted(TRACES))
def test_golden_swap_traces(view, name):
    _run(VIEWS[view], TRACES[name])


class _Payload:
    """Shadow KV: device slot -> prefix, host slot -> prefix, moved along the
    manager's pairs as pa_reshape_and_cache, pa_copy_blocks and
    pa_swap_blocks would."""

    def __init__(self, nb, nh, bs):
        self.B = bs
        self.dev = [None] * (nb * bs)
        self.host = [None] * (nh * bs)
        self.ids = {}

    def admit(self, m, s, ids):
        self.ids[s] = list(ids)
        tab = m.table(s)
        for i in range(len(ids)):
            self.dev[tab[i // self.B] * self.B + i % self.B] = tuple(ids[:i + 1])

    def append(self, s, tok, slot, src, dst):
        B = self.B
        if src >= 0:
            self.dev[dst * B:(dst + 1) * B] = self.dev[src * B:(src + 1) * B]
        self.ids[s].append(tok)
        self.dev[slot] = tuple(self.ids[s])

    def move(self, pairs, out):
        B = self.B
        src, dst = (self.dev, self.host) if out else (self.host, self.dev)
        for a, b in pairs:
            dst[b * B:(b + 1) * B] = src[a * B:(a + 1) * B]

    def check(self, m, live):
        for s in live:
            pool = self.host if m.is_swapped(s) == 1 else self.dev
            tab = m.table(s)
            for i in range(len(self.ids[s])):
                assert pool[tab[i // self.B] * self.B + i % self.B] == tuple(self.ids[s][:i + 1]), (s, i)


@pytest.mark.parametrize("view", sorted(VIEWS))
@pytest.mark.parametrize("seed,nb,nh,bs", [(0, 16, 12, 4), (1, 40, 20, 2), (2, 24, 30, 8)])
def test_payload_invariant_with_swaps(view, seed, nb, nh, bs):
    rng = np.random.default_rng(seed)
    m = VIEWS[view](nb, bs)
    assert m.enable_swap(nh) == 0
    pay = _Payload(nb, nh, bs)
    live, nxt = set(), 0
    for step in range(1500):
        op = int(rng.integers(0, 9))
        running = sorted(q for q in live if m.is_swapped(q) == 0)
        swapped = sorted(q for q in live if m.is_swapped(q) == 1)
        if op <= 1:
            n = int(rng.integers(1, 3 * bs))
            if m.alloc(nxt, n) == 0:
                pay.admit(m, nxt, list(range(nxt * 1000, nxt * 1000 + n)))
                live.add(nxt)
            nxt += 1
        elif op <= 3 and running:
            q = int(rng.choice(running))
            st, slot, src, dst = m.append_slot(q)
            if st == 0:
                pay.append(q, int(rng.integers(0, 10 ** 6)), slot, src, dst)
        elif op == 4 and running:
            q = int(rng.choice(running))
            if m.fork(q, nxt) == 0:
                pay.ids[nxt] = list(pay.ids[q])
                live.add(nxt)
            nxt += 1
        elif op == 5 and running:
            batch = [int(x) for x in rng.choice(running, size=min(len(running), int(rng.integers(1, 4))), replace=False)]
            st, pairs = m.swap_out(batch)
            if st == 0:
                pay.move(pairs, True)
            else:
                assert st == api.PA_FAIL_NO_BLOCKS and pairs == []
        elif op == 6 and swapped:
            batch = [int(x) for x in rng.choice(swapped, size=min(len(swapped), int(rng.integers(1, 4))), replace=False)]
            st, pairs = m.swap_in(batch)
            if st == 0:
                pay.move(pairs, False)
            else:
                assert st == api.PA_FAIL_NO_BLOCKS and pairs == []
        elif live:
            q = int(rng.choice(sorted(live)))
            assert m.free(q) == 0
            live.discard(q)
        if step % 25 == 0:
            pay.check(m, live)
            on_dev = {b for q in live if m.is_swapped(q) == 0 for b in m.table(q)}
            on_host = {h for q in live if m.is_swapped(q) == 1 for h in m.table(q)}
            assert len(on_dev) + m.num_free() + m.num_cached() == nb
            assert len(on_host) + m.num_free_host() == nh
    pay.check(m, live)


@pytest.mark.parametrize("seed,nb,nh,bs", [(3, 20, 10, 4), (4, 48, 32, 8)])
def test_abi_matches_oracle_with_swaps(seed, nb, nh, bs):
    rng = np.random.default_rng(seed)
    ref, dut = _OracleView(nb, bs), _AbiView(nb, bs)
    assert ref.enable_swap(nh) == dut.enable_swap(nh) == 0
    seqs = list(range(10))
    for _ in range(3000):
        op = int(rng.integers(0, 8))
        q = int(rng.choice(seqs))
        if op <= 1:
            n = int(rng.integers(-1, 3 * bs))
            assert ref.alloc(q, n) == dut.alloc(q, n)
        elif op == 2:
            assert ref.append_slot(q) == dut.append_slot(q)
        elif op == 3:
            c = int(rng.choice(seqs))
            assert ref.fork(q, c) == dut.fork(q, c)
        elif op in (4, 5):
            batch = [int(x) for x in rng.choice(seqs, size=int(rng.integers(1, 4)), replace=True)]
            fn = "swap_out" if op == 4 else "swap_in"
            assert getattr(ref, fn)(batch) == getattr(dut, fn)(batch), (fn, batch)
        else:
            assert ref.free(q) == dut.free(q)
    assert ref.m.free_blocks == dut.m.free_list()
    assert ref.num_free_host() == dut.num_free_host()
    for q in seqs:
        assert ref.is_swapped(q) == dut.is_swapped(q)
        if q in ref.m.block_tables:
            assert ref.table(q) == dut.table(q)
    assert [ref.ref(b) for b in range(nb)] == [dut.ref(b) for b in range(nb)]


def test_swap_argument_errors():
    a = api.BlockAllocator(8, 4)
    assert a.enable_swap(-1) == api.PA_ERR_INVALID_ARG
    assert a.enable_swap(4) == 0
    assert a.allocate(1, 5) == 0
    assert a.swap_out([9])[0] == api.PA_ERR_UNKNOWN_SEQ
    assert a.swap_out([1, 1])[0] == api.PA_ERR_INVALID_ARG
    assert a.swap_in([1])[0] == api.PA_ERR_INVALID_ARG          # not swapped out
    assert a.swap_out([1])[0] == 0
    assert a.swap_out([1])[0] == api.PA_ERR_SWAPPED
    assert a.enable_swap(8) == api.PA_ERR_INVALID_ARG           # something is out
    assert a.fork(1, 2) == api.PA_ERR_SWAPPED
    with pytest.raises(api.PAError):
        a.build_tables([1], 4)
    assert a.seq_len(1) == 5 and a.is_swapped(1) == 1


def test_operational_metrics_follow_the_operations():
    """The pool's operational metrics ("PagedAttention and KV Memory",
    Operational metrics: block-pool usage, preemptions by swapping, prefix
    cache hit rate, mean sequence length), counted by hand along a short
    history of admissions, a fork, swaps, appends and releases."""
    a = api.BlockAllocator(64, 16)
    assert a.enable_swap(32) == 0
    assert a.allocate(1, 40) == 0 and a.allocate(2, 16) == 0            # 3 + 1 blocks
    assert a.fork(1, 3) == 0                                            # shares seq 1's 3 blocks
    m = a.metrics()
    assert m == {"gpu_cache_usage_perc": 100.0 * 4 / 64, "num_preemption": 0, "prefix_cache_hit_rate": 0.0,
                 "avg_sequence_length": (40 + 16 + 40) / 3}
    st, pairs = a.swap_out([1, 3])                                      # one preemption per sequence
    assert st == 0 and len(pairs) == 3
    s = a.stats()
    assert s["num_swapped"] == 2 and s["num_swap_outs"] == 2 and s["num_used"] == 1
    assert a.metrics()["gpu_cache_usage_perc"] == 100.0 / 64
    st, pairs = a.swap_in([1])                                          # seq 3 stays on the host
    assert st == 0 and len(pairs) == 3
    s = a.stats()
    assert s["num_swapped"] == 1 and s["num_swap_outs"] == 2 and s["num_used"] == 4
    assert a.free(3) == 0                                               # releases its host blocks
    assert a.stats()["num_swapped"] == 0
    assert a.append_slot(2)[0] == 0                                     # 17 positions: a second block
    assert a.swap_out([2])[0] == 0
    m = a.metrics()
    assert m["num_preemption"] == 3 and m["avg_sequence_length"] == (40 + 17) / 2
    assert m["gpu_cache_usage_perc"] == 100.0 * 3 / 64
    assert a.stats()["num_context_tokens"] == 57


def test_metrics_of_an_empty_pool_and_prefix_hits():
    a = api.BlockAllocator(8, 4)
    assert a.metrics() == {"gpu_cache_usage_perc": 0.0, "num_preemption": 0, "prefix_cache_hit_rate": 0.0,
                           "avg_sequence_length": 0.0}
    assert a.enable_prefix_caching(True) == 0
    assert a.allocate_tokens(1, [5, 6, 7, 8, 9]) == (0, 0)
    assert a.allocate_tokens(2, [5, 6, 7, 8, 1, 2]) == (0, 4)           # the first full block is found
    assert a.metrics()["prefix_cache_hit_rate"] == 4 / 11
