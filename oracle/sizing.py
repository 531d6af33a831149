"""KV-cache sizing arithmetic (oracle; test infrastructure only).

[P1] section 1 "The memory bottleneck in key-value serving": one key and one
value vector per cached position, per layer and per KV head, each d_head
elements wide.  [P2] section 4 states the same estimate with T tokens.
[P1] section 8 "Fragmentation boundaries under paging": a sequence of S
tokens holds ceil(S / B) blocks and wastes ceil(S / B) * B - S slots.
[P1] section 8 "Block table metadata footprint": one int32 per block.
"""


def kv_bytes_per_token(n_layers, n_kv_heads, d_head, elem_bytes):
    """Bytes one cached token position occupies over all layers: keys and
    values (factor 2) for every layer and KV head ([P1] section 1)."""
    return 2 * n_layers * n_kv_heads * d_head * elem_bytes


def kv_bytes(n_layers, n_tokens, n_kv_heads, d_head, elem_bytes):
    """Total KV bytes for n_tokens cached positions ([P2] section 4)."""
    return n_tokens * kv_bytes_per_token(n_layers, n_kv_heads, d_head, elem_bytes)


def blocks_needed(n_tokens, block_size):
    """Physical blocks a sequence of n_tokens occupies: ceil(S / B)
    ([P1] section 8, item 3)."""
    return -(-n_tokens // block_size)


def tail_waste_slots(n_tokens, block_size):
    """Unused slots in a sequence's last block: ceil(S / B) * B - S
    ([P1] section 8, item 3)."""
    return blocks_needed(n_tokens, block_size) * block_size - n_tokens


def block_table_bytes(n_tokens, block_size, entry_bytes=4):
    """Bytes of one sequence's block table, one int32 per block
    ([P1] section 8, "Block table metadata footprint")."""
    return blocks_needed(n_tokens, block_size) * entry_bytes


def capacity_plan(lengths, block_size, pool_slots):
    """Blocks, slots and tail waste of a batch, and whether it fits a pool
    of pool_slots token slots ([P1] section 10 worked capacity decision)."""
    blocks = [blocks_needed(s, block_size) for s in lengths]
    slots = sum(blocks) * block_size
    waste = sum(tail_waste_slots(s, block_size) for s in lengths)
    return {
        "blocks": sum(blocks),
        "slots": slots,
        "waste": waste,
        "waste_frac": waste / slots if slots else 0.0,
        "fits": slots <= pool_slots,
        "deficit_slots": max(0, slots - pool_slots),
    }
