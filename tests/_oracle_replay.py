"""Oracle-side replay of a scenario: the reference allocator plans every
operation and the oracle cache ops move the payload in host pools of bf16
bit patterns (uint16).  Shares no code with the CUDA path; the token data
comes from the same seeded generators."""
import numpy as np

from oracle import allocator as AL
from oracle import cache_ops as C
from paged_kv_cache_124_gb300 import inputs as I


class OracleReplay:
    def __init__(self, sc, layers=None, data_fn=None):
        """layers: which layers to materialise (default all).  data_fn(kind,
        layer, index, n) may supply (k, v) uint16 arrays instead of drawing
        them on the CPU (kind 'prefill' with index = seq, or 'append' with
        index = step)."""
        self.sc = sc
        self.layers = list(range(sc.n_layers)) if layers is None else list(layers)
        self.alloc = AL.RefAllocator(sc.num_blocks, sc.block_size)
        shape = (sc.num_blocks, sc.n_kv_heads, sc.block_size, sc.d_head)
        self.k = {l: np.full(shape, I.NAN_BF16_BITS, dtype=np.uint16) for l in self.layers}
        self.v = {l: np.full(shape, I.NAN_BF16_BITS, dtype=np.uint16) for l in self.layers}
        self.decoded = set(sc.decode_seqs)
        self.data_fn = data_fn
        self.cow_pairs = []

    def _data(self, kind, layer, index, n):
        if self.data_fn is not None:
            return self.data_fn(kind, layer, index, n)
        sc = self.sc
        if kind == "prefill":
            k, v = I.prefill_kv(sc.seed, layer, index, n, sc.n_kv_heads, sc.d_head)
        else:
            k, v = I.append_kv(sc.seed, layer, index, n, sc.n_kv_heads, sc.d_head)
        return I.bf16_bits(k), I.bf16_bits(v)

    def replay(self):
        sc = self.sc
        B = sc.block_size
        pending = []
        step = 0
        for op in sc.ops:
            kind = op[0]
            if kind == "free_order":
                assert self.alloc.set_free_order(op[1]) == AL.OK
            elif kind == "alloc":
                _, seq, n = op
                assert self.alloc.allocate(seq, n) == AL.OK
                if seq in self.decoded:
                    slots = [self.alloc.slot_of(seq, i) for i in range(n)]
                    for l in self.layers:
                        k, v = self._data("prefill", l, seq, n)
                        C.reshape_and_cache(self.k[l], self.v[l], k, v, slots, B)
            elif kind == "fork":
                assert self.alloc.fork(op[1], op[2]) == AL.OK
            elif kind == "append":
                pending.append(op[1])
            elif kind == "step":
                if pending:
                    slots, pairs = [], []
                    for seq in pending:
                        st, slot, src, dst = self.alloc.append_slot(seq)
                        assert st == AL.OK
                        slots.append(slot)
                        if src >= 0:
                            pairs.append((src, dst))
                    self.cow_pairs += pairs
                    if pairs:
                        C.copy_blocks([self.k[l] for l in self.layers], [self.v[l] for l in self.layers], pairs)
                    for l in self.layers:
                        k, v = self._data("append", l, step, len(pending))
                        C.reshape_and_cache(self.k[l], self.v[l], k, v, slots, B)
                    step += 1
                pending = []
            elif kind == "free":
                assert self.alloc.free(op[1]) == AL.OK
        return self

    def tables(self):
        seqs = self.sc.decode_seqs
        lens = [self.alloc.seq_lengths[s] for s in seqs]
        mb = max(-(-L // self.sc.block_size) for L in lens)
        tab = np.full((len(seqs), mb), -1, dtype=np.int64)
        for i, s in enumerate(seqs):
            t = self.alloc.block_tables[s]
            tab[i, :len(t)] = t
        return tab, np.array(lens, dtype=np.int64)
