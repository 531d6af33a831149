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

Automatic prefix caching ([P1] section 18; [P2] section 6; [P3] "Prefix
caching"), off until enable_prefix_caching(True):
  * Only full blocks whose token ids are known are cached.  A block's key is
    the exact tuple of every token id from position 0 to the block's end, so
    two blocks match only when the whole prefix up to them is identical
    ([P2] section 6: equal text after a different prefix does not match).
  * A new prompt with known token ids looks its full blocks up from the
    first one and stops at the first miss; every hit is shared (count + 1),
    and a hit with count 0 leaves the eviction queue and goes back to 1
    ([P1] section 18).  The hits' positions need no prefill.  The remaining
    blocks are taken fresh and the full ones are registered under their
    keys at once, unless another block already holds that key.
  * A registered block whose count reaches 0 is queued for eviction rather
    than freed; within one release the deepest block is queued first.
  * A fresh block comes from the free list while it has any, else from the
    front (oldest) of the eviction queue, which forgets its key ([P1]
    section 19, item 2; [P2] section 6, the LRU-style free queue).
  * Appending a position with a known token id that fills the block
    registers it; appending without a token id forgets the sequence's
    tokens, so none of its later blocks is registered.
  * Running short is checked against the free list plus the queue (less the
    hits taken out of the queue); on failure nothing changes.

Swapping ([P1] section 19, item 4: move a preempted request's blocks to host
memory and back), enabled with a host pool of its own (a stack handing out
host blocks 0, 1, 2, ...):
  * swap_out(seqs) takes the distinct device blocks of the batch's tables in
    first-appearance order and gives each one host block whose count is the
    number of batch sequences using it; then each sequence, in batch order,
    releases its device table as free() would; its table now names host
    blocks.  Too few host blocks: nothing changes.
  * swap_in(seqs) is the mirror image: distinct host blocks in
    first-appearance order each get a fresh device block (free list, then the
    eviction queue) with the batch count; each sequence drops one reference
    per host block, and host blocks at 0 go back on the host stack.  Too few
    device blocks: nothing changes.
  * A swapped-out sequence accepts only free (which releases its host
    blocks); appends, forks and table reads report it as swapped.
"""
from collections import OrderedDict

OK = 0
FAIL_NO_BLOCKS = 1
ERR_INVALID_ARG = -1
ERR_UNKNOWN_SEQ = -6
ERR_DUPLICATE_SEQ = -7
ERR_SWAPPED = -8


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
        # prefix cache
        self.caching = False
        self.cache_index = {}          # prefix key -> block
        self.block_key = {}            # block -> prefix key (registered blocks)
        self.evict_queue = OrderedDict()   # zero-count registered blocks, oldest first
        self.seq_tokens = {}           # seq -> list of token ids, or None when unknown
        self.num_prompt_tokens = 0
        self.num_cached_tokens = 0
        # swap space
        self.host_free = []
        self.host_refs = []
        self.swapped = set()

    # -- prefix-cache helpers ----------------------------------------------
    def _available(self):
        return len(self.free_blocks) + len(self.evict_queue)

    def _take(self):
        """A fresh block with count 1: free list first, else evict the oldest
        zero-count cached block and forget its key."""
        if self.free_blocks:
            b = self.free_blocks.pop()
        else:
            b, _ = self.evict_queue.popitem(last=False)
            del self.cache_index[self.block_key.pop(b)]
        self.ref_counts[b] = 1
        return b

    def _register(self, b, key):
        if key in self.cache_index:
            return
        self.cache_index[key] = b
        self.block_key[b] = key

    # -- set-up -------------------------------------------------------------
    def set_free_order(self, order):
        """Replace the free list by `order` (blocks are taken from its end),
        as [P1] section 20, test 3 does to force a non-identity placement.
        Allowed only while no block is in use."""
        order = [int(b) for b in order]
        if self.block_tables or self.evict_queue or sorted(order) != list(range(self.num_blocks)):
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
        if self._available() < needed:
            return FAIL_NO_BLOCKS
        self.block_tables[seq] = [self._take() for _ in range(needed)]
        self.seq_lengths[seq] = num_tokens
        self.seq_tokens[seq] = None
        self.num_prompt_tokens += num_tokens
        return OK

    def enable_prefix_caching(self, enable=True):
        """Only while no sequence exists.  Switching off moves the queue to
        the free list, oldest first, and forgets every key."""
        if self.block_tables:
            return ERR_INVALID_ARG
        if not enable:
            for b in self.evict_queue:
                self.free_blocks.append(b)
            self.evict_queue.clear()
            self.cache_index.clear()
            self.block_key.clear()
        self.caching = bool(enable)
        return OK

    def allocate_tokens(self, seq, tokens):
        """New sequence with known prompt token ids.  Returns (status,
        number of leading positions found in the prefix cache)."""
        tokens = [int(t) for t in tokens]
        if seq in self.block_tables:
            return ERR_DUPLICATE_SEQ, 0
        if not tokens:
            return ERR_INVALID_ARG, 0
        B = self.block_size
        needed = -(-len(tokens) // B)
        full = len(tokens) // B
        keys = [tuple(tokens[:(i + 1) * B]) for i in range(full)]
        hits = []
        if self.caching:
            for key in keys:
                if key not in self.cache_index:
                    break
                hits.append(self.cache_index[key])
        from_queue = sum(1 for b in hits if b in self.evict_queue)
        if self._available() - from_queue < needed - len(hits):
            return FAIL_NO_BLOCKS, 0
        table = []
        for b in hits:
            self.evict_queue.pop(b, None)
            self.ref_counts[b] += 1
            table.append(b)
        for i in range(len(hits), needed):
            b = self._take()
            table.append(b)
            if self.caching and i < full:
                self._register(b, keys[i])
        self.block_tables[seq] = table
        self.seq_lengths[seq] = len(tokens)
        self.seq_tokens[seq] = tokens
        self.num_prompt_tokens += len(tokens)
        self.num_cached_tokens += len(hits) * B
        return OK, len(hits) * B

    def fork(self, parent, child):
        if parent not in self.block_tables:
            return ERR_UNKNOWN_SEQ
        if child in self.block_tables:
            return ERR_DUPLICATE_SEQ
        if parent in self.swapped:
            return ERR_SWAPPED
        for b in self.block_tables[parent]:
            self.ref_counts[b] += 1
        self.block_tables[child] = list(self.block_tables[parent])
        self.seq_lengths[child] = self.seq_lengths[parent]
        toks = self.seq_tokens.get(parent)
        self.seq_tokens[child] = None if toks is None else list(toks)
        return OK

    def append_slot(self, seq):
        """Plan one appended position.  Returns (status, slot, cow_src, cow_dst);
        slot is -1 and cow_src/cow_dst are -1 when there is nothing to do."""
        return self._append(seq, None)

    def append_token(self, seq, token):
        """append_slot for a position whose token id is known."""
        return self._append(seq, int(token))

    def _append(self, seq, token):
        if seq not in self.block_tables:
            return ERR_UNKNOWN_SEQ, -1, -1, -1
        if seq in self.swapped:
            return ERR_SWAPPED, -1, -1, -1
        B = self.block_size
        length = self.seq_lengths[seq]
        table = self.block_tables[seq]
        offset = length % B
        cow_src = cow_dst = -1
        if offset != 0:
            tail = table[-1]
            if self.ref_counts[tail] > 1:
                if not self._available():
                    return FAIL_NO_BLOCKS, -1, -1, -1
                new = self._take()
                self.ref_counts[tail] -= 1
                table[-1] = new
                cow_src, cow_dst = tail, new
                self.num_cow_copies += 1
                slot = new * B + offset
            else:
                slot = tail * B + offset
        else:
            if not self._available():
                return FAIL_NO_BLOCKS, -1, -1, -1
            new = self._take()
            table.append(new)
            slot = new * B
        self.seq_lengths[seq] = length + 1
        toks = self.seq_tokens.get(seq)
        if token is None or toks is None:
            self.seq_tokens[seq] = None
        else:
            toks.append(token)
            if self.caching and offset == B - 1:      # this position filled the block
                self._register(slot // B, tuple(toks))
        return OK, slot, cow_src, cow_dst

    def free(self, seq):
        if seq not in self.block_tables:
            return OK
        if seq in self.swapped:
            for h in self.block_tables[seq]:
                self.host_refs[h] -= 1
                if self.host_refs[h] == 0:
                    self.host_free.append(h)
            self.swapped.discard(seq)
            del self.block_tables[seq]
            del self.seq_lengths[seq]
            self.seq_tokens.pop(seq, None)
            return OK
        idle_cached = []
        for b in self.block_tables[seq]:
            self.ref_counts[b] -= 1
            if self.ref_counts[b] == 0:
                if b in self.block_key:
                    idle_cached.append(b)
                else:
                    self.free_blocks.append(b)
        for b in reversed(idle_cached):
            self.evict_queue[b] = None
        del self.block_tables[seq]
        del self.seq_lengths[seq]
        self.seq_tokens.pop(seq, None)
        return OK

    # -- queries --------------------------------------------------------------
    def slot_of(self, seq, i):
        """Pool slot of position i of a sequence ([P1] section 7)."""
        B = self.block_size
        return self.block_tables[seq][i // B] * B + i % B

    def num_free(self):
        return len(self.free_blocks)

    def enable_swap(self, num_host_blocks):
        if num_host_blocks < 0 or self.swapped:
            return ERR_INVALID_ARG
        self.host_free = list(reversed(range(num_host_blocks)))
        self.host_refs = [0] * num_host_blocks
        return OK

    def _swap_batch(self, seqs, from_swapped):
        """Check a swap batch; return (status, distinct blocks in first-appearance
        order, number of batch sequences using each)."""
        seen, blocks, counts = set(), [], {}
        for q in seqs:
            if q not in self.block_tables:
                return ERR_UNKNOWN_SEQ, None, None
            if (q in self.swapped) != from_swapped:
                return (ERR_INVALID_ARG if from_swapped else ERR_SWAPPED), None, None
            if q in seen:
                return ERR_INVALID_ARG, None, None
            seen.add(q)
            for b in self.block_tables[q]:
                if b not in counts:
                    counts[b] = 0
                    blocks.append(b)
                counts[b] += 1
        return OK, blocks, counts

    def swap_out(self, seqs):
        """Returns (status, [(device block, host block), ...])."""
        st, blocks, counts = self._swap_batch(seqs, False)
        if st != OK:
            return st, []
        if len(blocks) > len(self.host_free):
            return FAIL_NO_BLOCKS, []
        to_host = {}
        for b in blocks:
            h = self.host_free.pop()
            self.host_refs[h] = counts[b]
            to_host[b] = h
        for q in seqs:
            idle_cached = []
            for b in self.block_tables[q]:          # the device references go, as in free()
                self.ref_counts[b] -= 1
                if self.ref_counts[b] == 0:
                    if b in self.block_key:
                        idle_cached.append(b)
                    else:
                        self.free_blocks.append(b)
            for b in reversed(idle_cached):
                self.evict_queue[b] = None
            self.block_tables[q] = [to_host[b] for b in self.block_tables[q]]
            self.swapped.add(q)
        return OK, [(b, to_host[b]) for b in blocks]

    def swap_in(self, seqs):
        """Returns (status, [(host block, device block), ...])."""
        st, blocks, counts = self._swap_batch(seqs, True)
        if st != OK:
            return st, []
        if len(blocks) > self._available():
            return FAIL_NO_BLOCKS, []
        to_dev = {}
        for h in blocks:
            b = self._take()
            self.ref_counts[b] = counts[h]
            to_dev[h] = b
        for q in seqs:
            for h in self.block_tables[q]:
                self.host_refs[h] -= 1
                if self.host_refs[h] == 0:
                    self.host_free.append(h)
            self.block_tables[q] = [to_dev[h] for h in self.block_tables[q]]
            self.swapped.discard(q)
        return OK, [(h, to_dev[h]) for h in blocks]

    def num_cached(self):
        return len(self.evict_queue)

    def cached_list(self):
        """Zero-count cached blocks, next to be evicted first."""
        return list(self.evict_queue)
