"""Reference block manager (oracle; test infrastructure only).

Restates the block-manager semantics of [P1] sections 14 to 17 and of its
section 20 teaching model, with one change of shape: appending a token here
only *plans* the step.  It returns the slot the new token's key and value go
to and, when the tail block was shared, the (src, dst) pair that the GPU must
copy first.  Moving the payload is left to reshape_and_cache and copy_blocks
(see cache_ops), so no payload lives in the manager.

Semantics restated:
  * The free list starts as the block ids in descending order and blocks are
    taken from its end, so a fresh manager hands out 0, 1, 2, ...; released
    blocks go back on the end ([P1] section 20).
  * Allocating a prompt of n > 0 tokens takes ceil(n / B) blocks with
    reference count 1.  If too few blocks are free, nothing changes and the
    call reports exhaustion ([P1] section 20; section 19 on exhaustion).
  * Fork copies the parent's block table and adds one reference to every
    block in it ([P1] section 16, step 2).
  * Append at position L = current length, offset L % B ([P1] sections 15, 16):
      - offset != 0 and tail shared (ref > 1): take a new block, count the
        copy (tail -> new), drop one reference of the tail, retarget the last
        table entry, write at offset in the new block;
      - offset != 0 and tail private: write in place;
      - offset == 0: take a new block and write at offset 0.
    On exhaustion nothing changes ([P1] section 20, test 4).
  * Release drops one reference per table entry, in table order, and puts a
    block back on the free list when its count reaches 0 ([P1] section 17).
    Releasing an unknown sequence does nothing.
"""

OK = 0
FAIL_NO_BLOCKS = 1
ERR_INVALID_ARG = -1
ERR_UNKNOWN_SEQ = -6
ERR_DUPLICATE_SEQ = -7


class RefAllocator:
    def __init__(self, num_blocks, block_size):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("pool size and block size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free_blocks = list(reversed(range(num_blocks)))
        self.ref_counts = [0] * num_blocks
        self.block_tables = {}
        self.seq_lengths = {}
        self.num_cow_copies = 0

    # -- set-up -------------------------------------------------------------
    def set_free_order(self, order):
        """Replace the free list by `order` (blocks are taken from its end),
        as [P1] section 20, test 3 does to force a non-identity placement.
        Allowed only while no block is in use."""
        order = [int(b) for b in order]
        if self.block_tables or sorted(order) != list(range(self.num_blocks)):
            return ERR_INVALID_ARG
        self.free_blocks = order
        return OK

    # -- sequence operations ------------------------------------------------
    def allocate(self, seq, num_tokens):
        if seq in self.block_tables:
            return ERR_DUPLICATE_SEQ
        if num_tokens <= 0:
            return ERR_INVALID_ARG
        needed = -(-num_tokens // self.block_size)
        if len(self.free_blocks) < needed:
            return FAIL_NO_BLOCKS
        table = []
        for _ in range(needed):
            b = self.free_blocks.pop()
            self.ref_counts[b] = 1
            table.append(b)
        self.block_tables[seq] = table
        self.seq_lengths[seq] = num_tokens
        return OK

    def fork(self, parent, child):
        if parent not in self.block_tables:
            return ERR_UNKNOWN_SEQ
        if child in self.block_tables:
            return ERR_DUPLICATE_SEQ
        for b in self.block_tables[parent]:
            self.ref_counts[b] += 1
        self.block_tables[child] = list(self.block_tables[parent])
        self.seq_lengths[child] = self.seq_lengths[parent]
        return OK

    def append_slot(self, seq):
        """Plan one appended position.  Returns (status, slot, cow_src, cow_dst);
        slot is -1 and cow_src/cow_dst are -1 when there is nothing to do."""
        if seq not in self.block_tables:
            return ERR_UNKNOWN_SEQ, -1, -1, -1
        B = self.block_size
        length = self.seq_lengths[seq]
        table = self.block_tables[seq]
        offset = length % B
        cow_src = cow_dst = -1
        if offset != 0:
            tail = table[-1]
            if self.ref_counts[tail] > 1:
                if not self.free_blocks:
                    return FAIL_NO_BLOCKS, -1, -1, -1
                new = self.free_blocks.pop()
                self.ref_counts[new] = 1
                self.ref_counts[tail] -= 1
                table[-1] = new
                cow_src, cow_dst = tail, new
                self.num_cow_copies += 1
                slot = new * B + offset
            else:
                slot = tail * B + offset
        else:
            if not self.free_blocks:
                return FAIL_NO_BLOCKS, -1, -1, -1
            new = self.free_blocks.pop()
            self.ref_counts[new] = 1
            table.append(new)
            slot = new * B
        self.seq_lengths[seq] = length + 1
        return OK, slot, cow_src, cow_dst

    def free(self, seq):
        if seq not in self.block_tables:
            return OK
        for b in self.block_tables[seq]:
            self.ref_counts[b] -= 1
            if self.ref_counts[b] == 0:
                self.free_blocks.append(b)
        del self.block_tables[seq]
        del self.seq_lengths[seq]
        return OK

    # -- queries --------------------------------------------------------------
    def slot_of(self, seq, i):
        """Pool slot of position i of a sequence ([P1] section 7)."""
        B = self.block_size
        return self.block_tables[seq][i // B] * B + i % B

    def num_free(self):
        return len(self.free_blocks)
