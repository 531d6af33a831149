"""Cache-feeding operations on a host copy of the block pool (oracle).

Test infrastructure only.  Pools are NumPy arrays of any dtype (the tests
use uint16 bf16 bit patterns, so every comparison with the device is
bit-exact) laid out [num_blocks, n_kv_heads, block_size, d_head].

reshape_and_cache: each new token's key and value rows go to the slot the
block manager chose for it.  [P1] section 20 writes position i of a sequence
to storage[block][offset]; a slot number names that place in the pool as
physical_block * B + offset, the frame-times-size-plus-offset form of
[P2] section 2.  A negative slot means "no write" (interface convention for
padding tokens).

copy_blocks: the copy-on-write clone of a shared tail block into a freshly
allocated block ([P1] sections 15 and 16).  The whole block is copied, for
every KV head, in keys and in values, in every layer.
"""

import numpy as np


def reshape_and_cache(k_cache, v_cache, k, v, slot_mapping, block_size):
    """Write token t's rows k[t], v[t] ([n_kv_heads, d_head] each) at
    slot_mapping[t], in place; returns the two pools."""
    k_out, v_out = k_cache, v_cache
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        block, offset = divmod(int(slot), block_size)
        k_out[block, :, offset, :] = k[t]
        v_out[block, :, offset, :] = v[t]
    return k_out, v_out


def copy_blocks(k_caches, v_caches, pairs):
    """Overwrite block dst by block src in every layer's pools, for each
    (src, dst) pair in order, in place; returns the two lists of pools."""
    k_out, v_out = k_caches, v_caches
    for layer in range(len(k_out)):
        for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
            k_out[layer][dst] = k_out[layer][src]
            v_out[layer][dst] = v_out[layer][src]
    return k_out, v_out


def swap_blocks(dst_k, dst_v, src_k, src_v, pairs):
    """Move whole blocks between two pools of the same block shape (the
    payload side of swapping, [P1] section 19, item 4): for each (src, dst)
    pair, block src of the source pools is copied onto block dst of the
    destination pools, K and V.  In place on the destination."""
    for src, dst in pairs:
        dst_k[dst] = src_k[src]
        dst_v[dst] = src_v[src]
