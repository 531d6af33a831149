"""Host orchestration of the paged KV path for one scenario.

Replays a scenario's block-manager operations through the C++ block manager
(api.BlockAllocator) and moves the payload with the library's kernels:

  alloc  -> pa_alloc_sequence, then pa_reshape_and_cache of the prompt's
            keys/values at the slots pa_alloc_slot_mapping gives;
  fork   -> pa_alloc_fork;
  append -> queued until the end of the step;
  step   -> pa_alloc_append_slots for the queued sequences, pa_copy_blocks
            for the copy-on-write pairs it returns (all layers), then
            pa_reshape_and_cache of the new positions (copies first, then
            writes: the order of the 35-token fork trace);
  free   -> pa_alloc_free.

Prompts of sequences that are not decoded (filler sequences that only shape
the free list) are allocated but not written.
"""

import numpy as np
import torch

from . import api
from . import inputs as I


class ScenarioRunner:
    def __init__(self, sc, device="cuda", data_device="cpu", n_layers=None):
        self.sc = sc
        self.device = torch.device(device)
        self.data_device = data_device
        self.n_layers = sc.n_layers if n_layers is None else n_layers
        self.alloc = api.BlockAllocator(sc.num_blocks, sc.block_size)
        shape = (sc.num_blocks, sc.n_kv_heads, sc.block_size, sc.d_head)
        self.k_caches = [I.nan_pool(shape, self.device) for _ in range(self.n_layers)]
        self.v_caches = [I.nan_pool(shape, self.device) for _ in range(self.n_layers)]
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.decoded = set(sc.decode_seqs)
        self.cow_pairs_total = 0

    def _write(self, layer, k, v, slots):
        slots_d = torch.from_numpy(np.ascontiguousarray(slots, dtype=np.int64)).to(self.device)
        api.pa_reshape_and_cache(self.k_caches[layer], self.v_caches[layer], k.to(self.device),
                                 v.to(self.device), slots_d, status=self.status)

    def replay(self):
        sc = self.sc
        pending = []
        step = 0
        for op in sc.ops:
            kind = op[0]
            if kind == "free_order":
                assert self.alloc.set_free_order(op[1]) == api.PA_OK
            elif kind == "alloc":
                _, seq, n = op
                assert self.alloc.allocate(seq, n) == api.PA_OK, op
                if seq in self.decoded:
                    slots = self.alloc.slot_mapping(seq, 0, n)
                    for layer in range(self.n_layers):
                        k, v = I.prefill_kv(sc.seed, layer, seq, n, sc.n_kv_heads, sc.d_head, self.data_device)
                        self._write(layer, k, v, slots)
            elif kind == "fork":
                assert self.alloc.fork(op[1], op[2]) == api.PA_OK, op
            elif kind == "append":
                pending.append(op[1])
            elif kind == "step":
                if pending:
                    st, slots, pairs, done = self.alloc.append_slots(pending)
                    assert st == api.PA_OK and done == len(pending), (st, done)
                    if len(pairs):
                        self.cow_pairs_total += len(pairs)
                        pd = torch.from_numpy(pairs).to(self.device)
                        api.pa_copy_blocks(self.k_caches, self.v_caches, pd, status=self.status)
                    for layer in range(self.n_layers):
                        k, v = I.append_kv(sc.seed, layer, step, len(pending), sc.n_kv_heads, sc.d_head,
                                           self.data_device)
                        self._write(layer, k, v, slots)
                    step += 1
                pending = []
            elif kind == "free":
                assert self.alloc.free(op[1]) == api.PA_OK
            else:
                raise ValueError(op)
        return self

    def decode_metadata(self):
        """Device block tables [S, max_blocks] int32, context lengths [S]
        int32, and the host max context length, for the decoded sequences."""
        lens = [self.alloc.seq_len(s) for s in self.sc.decode_seqs]
        max_ctx = max(lens)
        max_blocks = -(-max_ctx // self.sc.block_size)
        tables, ctx = self.alloc.build_tables(self.sc.decode_seqs, max_blocks)
        return (torch.from_numpy(tables).to(self.device), torch.from_numpy(ctx).to(self.device), max_ctx)
