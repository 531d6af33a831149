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
    """Return copies of the pools with token t's rows k[t], v[t]
    ([n_kv_heads, d_head] each) written at slot_mapping[t]."""
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        block, offset = divmod(int(slot), block_size)
        k_out[block, :, offset, :] = k[t]
        v_out[block, :, offset, :] = v[t]
    return k_out, v_out


def copy_blocks(k_caches, v_caches, pairs):
    """Return copies of every layer's pools with block dst overwritten by
    block src for each (src, dst) pair, applied in order."""
    k_out = [np.array(k, copy=True) for k in k_caches]
    v_out = [np.array(v, copy=True) for v in v_caches]
    for layer in range(len(k_out)):
        for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
            k_out[layer][dst] = k_out[layer][src]
            v_out[layer][dst] = v_out[layer][src]
    return k_out, v_out
