"""Automatic prefix caching end to end on the GPU: requests built from shared
documents are admitted through the C++ block manager with prefix caching on,
only their uncached positions are written (reshape_and_cache), decode steps
append generated tokens (with copy-on-write for forked requests), requests
finish and new ones revive or evict idle cached blocks.  Every position's KV
is a function of its whole prefix, so the check is independent of the block
manager: each live request's pool rows must equal the KV of its own token
sequence bit for bit, and the paged decode must match the oracle's dense
attention over that KV ("PagedAttention: Virtual Memory for the KV Cache",
section 18; "PagedAttention in vLLM: scattered memory, exact attention",
section 6: prefix caching reuses work without changing results)."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from _gpu_util import assert_attention_close, out_to_f64, to_bits

pytestmark = pytest.mark.gpu

api = pytest.importorskip("paged_kv_cache_124_gb300.api")
from paged_kv_cache_124_gb300 import inputs as I  # noqa: E402

HQ, HKV, D, LAYERS = 32, 8, 128, 2
SCALE = 1.0 / math.sqrt(D)


class _Engine:
    def __init__(self, seed, block_size, num_blocks):
        self.seed, self.B, self.NB = seed, block_size, num_blocks
        self.alloc = api.BlockAllocator(num_blocks, block_size)
        assert self.alloc.enable_prefix_caching(True) == 0
        shape = (num_blocks, HKV, block_size, D)
        self.k = [I.nan_pool(shape).cuda() for _ in range(LAYERS)]
        self.v = [I.nan_pool(shape).cuda() for _ in range(LAYERS)]
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.live = {}
        self.next_id = 0
        self.revived = self.shared_live = self.evicting_admissions = 0

    def _write(self, seq, toks, start, end):
        if end <= start:
            return
        slots = torch.from_numpy(self.alloc.slot_mapping(seq, start, end - start)).cuda()
        for l in range(LAYERS):
            k, v = I.prefix_kv(self.seed, l, toks, start, end, HKV, D)
            api.pa_reshape_and_cache(self.k[l], self.v[l], k.cuda(), v.cuda(), slots, status=self.status)

    def admit(self, toks):
        queued = set(self.alloc.cached_list())
        in_use = {b for s in self.live for b in self.alloc.block_table(s)}
        free_before = self.alloc.num_free()
        seq = self.next_id
        self.next_id += 1
        st, hit = self.alloc.allocate_tokens(seq, toks)
        if st == api.PA_FAIL_NO_BLOCKS:
            return None
        assert st == 0
        tab = self.alloc.block_table(seq)
        hits = tab[:hit // self.B]
        self.revived += sum(b in queued for b in hits)
        self.shared_live += sum(b in in_use for b in hits)
        if len(tab) - len(hits) > free_before:
            self.evicting_admissions += 1
        self._write(seq, toks, hit, len(toks))
        self.live[seq] = list(toks)
        return hit

    def fork(self, seq):
        child = self.next_id
        self.next_id += 1
        assert self.alloc.fork(seq, child) == 0
        self.live[child] = list(self.live[seq])
        return child

    def decode_step(self, rng):
        seqs = sorted(self.live)
        slots, pairs, rows_k, rows_v = [], [], [[] for _ in range(LAYERS)], [[] for _ in range(LAYERS)]
        for s in seqs:
            tok = int(rng.integers(0, 32000))
            st, slot, src, dst = self.alloc.append_token(s, tok)
            if st != 0:
                continue
            if src >= 0:
                pairs.append((src, dst))
            toks = self.live[s] + [tok]
            self.live[s] = toks
            slots.append(slot)
            for l in range(LAYERS):
                k, v = I.prefix_kv(self.seed, l, toks, len(toks) - 1, len(toks), HKV, D)
                rows_k[l].append(k)
                rows_v[l].append(v)
        if pairs:
            api.pa_copy_blocks(self.k, self.v, torch.tensor(pairs, dtype=torch.int32, device="cuda"),
                               status=self.status)
        if slots:
            sm = torch.tensor(slots, dtype=torch.int64, device="cuda")
            for l in range(LAYERS):
                api.pa_reshape_and_cache(self.k[l], self.v[l], torch.cat(rows_k[l]).cuda(),
                                         torch.cat(rows_v[l]).cuda(), sm, status=self.status)

    def finish(self, seq):
        assert self.alloc.free(seq) == 0
        del self.live[seq]

    def check(self, qseed):
        seqs = sorted(self.live)
        maxb = max(len(self.alloc.block_table(s)) for s in seqs)
        tables, ctx = self.alloc.build_tables(seqs, maxb)
        max_ctx = int(ctx.max())
        t_dev, c_dev = torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda()
        for l in range(LAYERS):
            kb, vb = to_bits(self.k[l]), to_bits(self.v[l])
            Kd = np.zeros((len(seqs), HKV, max_ctx, D))
            Vd = np.zeros((len(seqs), HKV, max_ctx, D))
            for i, s in enumerate(seqs):
                toks = self.live[s]
                k, v = I.prefix_kv(self.seed, l, toks, 0, len(toks), HKV, D)
                pos = np.arange(len(toks))
                blk = tables[i, pos // self.B]
                got_k = kb[blk, :, pos % self.B]           # [L, Hkv, D]
                got_v = vb[blk, :, pos % self.B]
                assert np.array_equal(got_k, to_bits(k)), "K rows of request %d layer %d" % (s, l)
                assert np.array_equal(got_v, to_bits(v)), "V rows of request %d layer %d" % (s, l)
                Kd[i, :, :len(toks)] = A.bf16_to_f64(to_bits(k)).transpose(1, 0, 2)
                Vd[i, :, :len(toks)] = A.bf16_to_f64(to_bits(v)).transpose(1, 0, 2)
            q = I.decode_q(qseed, l, len(seqs), HQ, D)
            want = A.dense_decode(A.bf16_to_f64(to_bits(q)), Kd, Vd, ctx, SCALE)
            out = torch.empty((len(seqs), HQ, D), dtype=torch.float32, device="cuda")
            ws = api.decode_workspace(len(seqs), HQ, D, max_ctx)
            api.pa_decode(out, q.cuda(), self.k[l], self.v[l], t_dev, c_dev, self.B, SCALE, HQ, HKV, D, max_ctx,
                          workspace=ws, status=self.status)
            torch.cuda.synchronize()
            assert_attention_close(out_to_f64(out), want, True, "prefix-cache decode layer %d" % l)
        assert self.status.item() == 0


@pytest.mark.parametrize("block_size,num_blocks", [(16, 96), (32, 48), (8, 200)])
def test_prefix_cache_reuse_revive_evict(block_size, num_blocks):
    seed = 7
    rng = np.random.default_rng(seed)
    docs = I.prompt_documents(seed, [300, 517, 1024])
    eng = _Engine(seed, block_size, num_blocks)
    hits_total = 0
    for wave in range(5):
        for _ in range(6):
            d = docs[int(rng.integers(0, len(docs)))]
            cut = len(d) if rng.random() < 0.6 else int(rng.integers(1, len(d)))
            toks = d[:cut] + [int(t) for t in rng.integers(0, 32000, size=int(rng.integers(1, 40)))]
            hit = eng.admit(toks)
            hits_total += hit or 0
        if eng.live and wave % 2 == 1:
            eng.fork(sorted(eng.live)[0])
        for _ in range(3):
            eng.decode_step(rng)
        if eng.live:
            eng.check(qseed=seed * 100 + wave)
        for s in sorted(eng.live):
            if rng.random() < 0.6:
                eng.finish(s)
    st = eng.alloc.stats()
    assert hits_total > 0 and st["num_cached_tokens"] == hits_total
    assert eng.revived > 0 and eng.shared_live > 0 and eng.evicting_admissions > 0
    assert st["num_used"] + st["num_free"] + st["num_cached"] == num_blocks
