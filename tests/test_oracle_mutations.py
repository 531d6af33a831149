"""Planted mistakes in the oracle are caught by its pins.  CPU only.

Each case copies one oracle module's source, makes one plausible mistake in
it (a dropped term or factor, a wrong sign, index or bound, swapped
operands, a changed constant of the number format, a changed list order),
loads the copy as a module of its own and runs the pin tests of that module
against the copy (page-printed worked examples and traces, closed forms,
format definitions, brute force, invariants): at least one of them must
fail.  The oracle's files are not changed; a mistake that no pin catches
makes its case fail here."""
import inspect
import os
import types

import numpy as np
import pytest

import oracle
import test_oracle_attention as TA
import test_oracle_host as TH
import test_oracle_prefill as TP
import test_oracle_quant as TQ
import test_prefix_cache as TPC
import test_swap as TS

ORACLE_DIR = os.path.dirname(os.path.abspath(oracle.__file__))

# The test modules that pin each oracle module, and the name they import it as.
PINS = {
    "attention": [(TA, "A"), (TP, "A"), (TH, "A")],
    "quant": [(TQ, "Q")],
    "cache_ops": [(TH, "C")],
    "sizing": [(TH, "Z")],
    "allocator": [(TH, "AL"), (TPC, "AL")],
}
# Tests that compare the oracle with the library's own block manager are not
# pins (they would catch a planted mistake by disagreeing with product code);
# tests run on both views run on the oracle's only.  test_swap reaches the
# oracle through test_prefix_cache's view.
NOT_PINS = ("abi_matches_oracle", "colliding_keys", "key_mask", "hit_rate", "prefix_argument_errors",
            "swap_argument_errors")
EXTRA_PIN_MODULES = {"allocator": [TS]}

# (module, original text, planted mistake, what the mistake is)
MUTANTS = [
    # attention: the definition, the paging, the grouping, the causal mask, the merge
    ("attention", "s = scale * (K @ q)\n", "s = K @ q\n", "score scale dropped"),
    ("attention", "a = e / e.sum()", "a = e / e.max()", "softmax normalised by its largest term"),
    ("attention", "    m = s.max()\n    e = np.exp(s - m)\n    a = e / e.sum()",
     "    m = s.min()\n    e = np.exp(s - m)\n    a = e / e.sum()", "minimum subtracted instead of maximum"),
    ("attention", "return a @ V", "return a @ V[::-1]", "value rows in reverse order"),
    ("attention", "logical_block = i // block_size", "logical_block = i % block_size",
     "logical block from the offset"),
    ("attention", "phys, _ = translate(b * block_size, block_size, block_table_row)",
     "phys, _ = translate(b, block_size, block_table_row)", "block index passed as a position"),
    ("attention", "valid = min(block_size, context_len - b * block_size)",
     "valid = min(block_size, context_len - b * block_size - 1)", "last position of each block dropped"),
    ("attention", "return q_head // (n_q_heads // n_kv_heads)", "return q_head % n_kv_heads",
     "interleaved instead of contiguous query-head groups"),
    ("attention", "K[h, :p + 1], V[h, :p + 1]", "K[h, :p + 2], V[h, :p + 2]",
     "causal mask lets a row see the next position"),
    ("attention", "K[h, :p + 1], V[h, :p + 1]", "K[h, :p], V[h, :p]", "causal mask hides the row's own position"),
    ("attention", "            p = C - n + i\n", "            p = i\n", "new positions counted from 0, not after the prefix"),
    ("attention", "w = np.exp(m_b - m)", "w = np.exp(m - m_b)", "merge weight with the wrong sign"),
    ("attention", "return m, e.sum(), e @ np.asarray(V, dtype=np.float64)",
     "return m, e.sum(), np.exp(s) @ np.asarray(V, dtype=np.float64)", "block value sum not shifted by its maximum"),
    ("attention", "return e @ np.asarray(V, dtype=np.float64), e.sum()",
     "return e @ np.asarray(V, dtype=np.float64), e.max()", "page normaliser is the largest term"),
    ("attention", "<< np.uint32(16)", "<< np.uint32(15)", "bf16 pattern shifted one bit short"),
    ("attention", "stop = min(start + partition_size, len(s))", "stop = min(start + partition_size - 1, len(s))",
     "each partition drops its last position"),
    ("attention", "V[:, b * block_size: b * block_size + valid, :] = to_f64(v_cache[phys, :, :valid, :])",
     "V[:, b * block_size: b * block_size + valid, :] = to_f64(k_cache[phys, :, :valid, :])", "values gathered from the key pool"),
    ("attention", "K_dense[s, h, :ctx], V_dense[s, h, :ctx]", "K_dense[s, h, :ctx], V_dense[s, h, 1:ctx + 1]",
     "dense reference reads values one position late"),
    # quant: the E4M3 format definition and the rounding rule
    ("quant", "(1.0 + m / 8.0) * 2.0 ** (e - 7)", "(1.0 + m / 8.0) * 2.0 ** (e - 8)", "exponent bias 8"),
    ("quant", "m * 2.0 ** -9", "m * 2.0 ** -10", "subnormal step 2^-10"),
    ("quant", "(1.0 + m / 8.0)", "(1.0 + m / 16.0)", "four fraction bits"),
    ("quant", "code = np.where(nan, NAN_CODE, code)", "code = np.where(nan | (np.abs(x) > 448.0), NAN_CODE, code)",
     "overflow gives NaN instead of saturating"),
    ("quant", "pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (code_hi % 2 == 0) & (code_lo % 2 != 0))",
     "pick_hi = d_hi <= d_lo", "ties rounded up instead of to the even code"),
    ("quant", "mag = np.where((e == 15) & (m == 7), np.nan, mag)", "mag = mag", "no NaN code"),
    ("quant", "sign = np.signbit(x).astype(np.int64) << 7", "sign = np.signbit(x).astype(np.int64) << 6",
     "sign bit in the wrong place"),
    ("quant", "np.asarray(x, dtype=np.float32) / np.float32(scale)", "np.asarray(x, dtype=np.float64) / float(scale)",
     "division in float64 instead of float32"),
    ("quant", "return e4m3_to_f64(codes) * float(np.float32(scale))", "return e4m3_to_f64(codes) / float(np.float32(scale))",
     "dequantisation divides by the scale"),
    # cache_ops: slot arithmetic and copy direction
    ("cache_ops", "block, offset = divmod(int(slot), block_size)", "offset, block = divmod(int(slot), block_size)",
     "block and offset swapped"),
    ("cache_ops", "if slot < 0:\n            continue", "if slot < -1:\n            continue",
     "slot -1 written instead of skipped"),
    ("cache_ops", "k_out[layer][dst] = k_out[layer][src]", "k_out[layer][src] = k_out[layer][dst]",
     "copy direction swapped for K"),
    ("cache_ops", "v_out[layer][dst] = v_out[layer][src]", "pass", "V not copied"),
    ("cache_ops", "        dst_k[dst] = src_k[src]\n", "        dst_k[src] = src_k[dst]\n", "swap copies K in the wrong direction"),
    # sizing: the closed forms
    ("sizing", "return 2 * n_layers * n_kv_heads * d_head * elem_bytes",
     "return n_layers * n_kv_heads * d_head * elem_bytes", "K only, V forgotten"),
    ("sizing", "return -(-n_tokens // block_size)", "return n_tokens // block_size", "floor instead of ceiling"),
    ("sizing", "return blocks_needed(n_tokens, block_size) * entry_bytes",
     "return blocks_needed(n_tokens, block_size) * 8", "8-byte table entries"),
    # allocator: free-list order, reference counts, copy on write
    ("allocator", "self.free_blocks = list(reversed(range(num_blocks)))", "self.free_blocks = list(range(num_blocks))",
     "free list not reversed"),
    ("allocator", "b = self.free_blocks.pop()", "b = self.free_blocks.pop(0)", "free list taken from the front"),
    ("allocator", "if self.ref_counts[tail] > 1:", "if self.ref_counts[tail] > 2:", "copy only when three share"),
    ("allocator", "                self.ref_counts[tail] -= 1\n", "", "shared tail keeps the writer's reference"),
    ("allocator", "for b in self.block_tables[parent]:\n            self.ref_counts[b] += 1",
     "for b in self.block_tables[parent]:\n            pass", "fork does not count the child's references"),
    ("allocator", "for b in self.block_tables[seq]:\n            self.ref_counts[b] -= 1",
     "for b in reversed(self.block_tables[seq]):\n            self.ref_counts[b] -= 1", "blocks released in reverse order"),
    ("allocator", "needed = -(-num_tokens // self.block_size)", "needed = num_tokens // self.block_size + 1",
     "one block too many for exact multiples"),
    ("allocator", "slot = tail * B + offset", "slot = tail * B + offset - 1", "append slot one before the tail position"),
    # allocator: prefix caching ([P1] sections 18-19, [P2] section 6) and swap planning ([P1] section 19)
    ("allocator", "keys = [tuple(tokens[:(i + 1) * B]) for i in range(full)]",
     "keys = [tuple(tokens[i * B:(i + 1) * B]) for i in range(full)]", "a block's key is its own tokens, not its prefix"),
    ("allocator", "b, _ = self.evict_queue.popitem(last=False)", "b, _ = self.evict_queue.popitem(last=True)",
     "the newest idle cached block evicted first"),
    ("allocator", "            self.evict_queue.pop(b, None)\n            self.ref_counts[b] += 1",
     "            self.ref_counts[b] += 1", "a revived block stays in the eviction queue"),
    ("allocator", "if self.caching and offset == B - 1:", "if self.caching and offset == B - 2:",
     "a generated block registered one position early"),
    ("allocator", "self.host_refs[h] = counts[b]", "self.host_refs[h] = 1", "host block of a shared block counted once"),
    ("allocator", "self.ref_counts[b] = counts[h]", "self.ref_counts[b] = 1", "swapped-in shared block counted once"),
    ("allocator", "if b not in counts:\n                    counts[b] = 0\n                    blocks.append(b)\n                counts[b] += 1",
     "counts[b] = counts.get(b, 0) + 1\n                blocks.append(b)", "a shared block swapped once per sharer"),
    # sizing: the tail waste and the capacity decision
    ("sizing", "return blocks_needed(n_tokens, block_size) * block_size - n_tokens", "return n_tokens % block_size",
     "tail waste as S mod B"),
    ("sizing", '"fits": slots <= pool_slots,', '"fits": slots < pool_slots,', "a batch that exactly fills the pool rejected"),
    ("sizing", '"deficit_slots": max(0, slots - pool_slots),', '"deficit_slots": max(0, pool_slots - slots),',
     "deficit with the wrong sign"),
    ("sizing", '"waste_frac": waste / slots if slots else 0.0,', '"waste_frac": waste / sum(lengths) if slots else 0.0,',
     "waste fraction of the tokens, not the slots"),
    # attention: translation offsets, the merge weights, partition scores, row and table indexing
    ("attention", "    offset = i % block_size\n", "    offset = i // block_size\n", "offset from the logical block"),
    ("attention", "m = max(sb[0] for sb in summaries)", "m = min(sb[0] for sb in summaries)",
     "merge takes the smallest block maximum"),
    ("attention", "z = z + w * z_b", "z = z + z_b", "block normalisers merged unweighted"),
    ("attention", "u = u + w * np.asarray(u_b, dtype=np.float64)", "u = u + np.asarray(u_b, dtype=np.float64)",
     "block value sums merged unweighted"),
    ("attention", "    s = scale * (K @ q_row)\n", "    s = K @ q_row\n", "partition scores unscaled"),
    ("attention", "out[row0 + i, g] = softmax_attention(q[row0 + i, g]", "out[row0 + i, g] = softmax_attention(q[i, g]",
     "prefill query rows not offset by the sequence's start"),
    ("attention", "K, V = gather_kv(k_cache, v_cache, block_tables[s], ctx, block_size)",
     "K, V = gather_kv(k_cache, v_cache, block_tables[0], ctx, block_size)", "every sequence read through the first table"),
    ("attention", "            out[s, g] = softmax_attention(q[s, g], K[h], V[h], scale)",
     "            out[s, g] = softmax_attention(q[s, g], K[0], V[0], scale)", "decode reads KV head 0 for every query head"),
    # quant: the sign of zero and NaN, subnormal codes
    ("quant", "sign = np.signbit(x).astype(np.int64) << 7", "sign = (x < 0).astype(np.int64) << 7",
     "negative zero and signed NaN lose their sign"),
    ("quant", "mag = np.where(e == 0, m * 2.0 ** -9,", "mag = np.where((e == 0) & (m == 0), m * 2.0 ** -9,",
     "subnormal codes read as normals"),
    # cache_ops: which rows land in the value pool
    ("cache_ops", "v_out[block, :, offset, :] = v[t]", "v_out[block, :, offset, :] = k[t]", "values written from the key rows"),
    ("cache_ops", "dst_v[dst] = src_v[src]", "dst_v[dst] = src_k[src]", "swap moves keys into the value pool"),
    # allocator: key registration, the eviction queue's order and accounting, host blocks, slot queries
    ("allocator", "        if key in self.cache_index:\n            return\n", "",
     "a later block with a known key replaces the first in the index"),
    ("allocator", "for b in reversed(idle_cached):\n            self.evict_queue[b] = None\n        del self.block_tables[seq]",
     "for b in idle_cached:\n            self.evict_queue[b] = None\n        del self.block_tables[seq]",
     "the shallowest idle block queued first"),
    ("allocator", "if self.caching and i < full:", "if self.caching and i < full - 1:", "the last full prompt block not registered"),
    ("allocator", "from_queue = sum(1 for b in hits if b in self.evict_queue)", "from_queue = 0",
     "hits taken out of the queue still counted as available"),
    ("allocator", "if self.free_blocks:\n            b = self.free_blocks.pop()",
     "if not self.evict_queue:\n            b = self.free_blocks.pop()", "cached blocks evicted while free blocks remain"),
    ("allocator", "return self.block_tables[seq][i // B] * B + i % B", "return self.block_tables[seq][i // B] * B + i // B",
     "slot offset from the logical block"),
    ("allocator", "self.host_free = list(reversed(range(num_host_blocks)))", "self.host_free = list(range(num_host_blocks))",
     "host blocks handed out from the top"),
    ("allocator", "            self.block_tables[q] = [to_dev[h] for h in self.block_tables[q]]",
     "            self.block_tables[q] = [to_dev[h] for h in reversed(self.block_tables[q])]",
     "swapped-in table in reverse order"),
]


def _mutant(module, old, new):
    with open(os.path.join(ORACLE_DIR, module + ".py")) as f:
        src = f.read()
    assert src.count(old) == 1, "the mistake's site must occur exactly once in oracle/%s.py" % module
    mod = types.ModuleType("oracle_mutant_" + module)
    mod.__package__ = "oracle"
    exec(compile(src.replace(old, new), "<oracle/%s.py with a planted mistake>" % module, "exec"), mod.__dict__)
    return mod


def _worked():
    """The worked-example fixture of the attention pins."""
    g = TA.load("p2_worked_attention.json")
    return {"g": g, "q": np.array(TA.ev_all(g["q"])), "K": np.array(TA.ev_all(g["K"])),
            "V": np.array(TA.ev_all(g["V"])), "scale": TA.ev(g["scale"])}


def _calls(fn):
    """The keyword-argument sets pytest would call a pin test with."""
    names, sets = [], [()]
    for mark in getattr(fn, "pytestmark", []):
        if mark.name != "parametrize":
            continue
        argnames = mark.args[0]
        argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
        values = [v if len(argnames) > 1 else (v,) for v in mark.args[1]]
        names += argnames
        sets = [s + tuple(v) for s in sets for v in values]
    params = inspect.signature(fn).parameters
    for s in sets:
        kw = dict(zip(names, s))
        if kw.get("view", "oracle") != "oracle":
            continue
        if "worked" in params:
            kw["worked"] = _worked()
        yield kw


def _pin_tests(module):
    mods = [tm for tm, _ in PINS[module]] + EXTRA_PIN_MODULES.get(module, [])
    for tm in mods:
        for name, fn in inspect.getmembers(tm, inspect.isfunction):
            if name.startswith("test_") and fn.__module__ == tm.__name__ and not any(x in name for x in NOT_PINS):
                yield tm.__name__ + "." + name, fn


def _first_failing_pin(module):
    for name, fn in _pin_tests(module):
        for kw in _calls(fn):
            try:
                with np.errstate(all="ignore"):
                    fn(**kw)
            except Exception:          # a failed assertion, or the mistake breaking the call
                return name
    return None


def test_pins_pass_on_the_oracle_itself():
    for module in PINS:
        assert _first_failing_pin(module) is None


@pytest.mark.parametrize("module,old,new,what", MUTANTS, ids=["%s: %s" % (m[0], m[3]) for m in MUTANTS])
def test_planted_mistake_is_caught(module, old, new, what, monkeypatch):
    mutant = _mutant(module, old, new)
    for tm, alias in PINS[module]:
        monkeypatch.setattr(tm, alias, mutant)
    assert _first_failing_pin(module) is not None, "no pin catches: " + what
