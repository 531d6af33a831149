// Host block manager: free list, reference counts, fork, append with
// copy-on-write planning, release, and automatic prefix caching.
//
// Semantics follow "PagedAttention: Virtual Memory for the KV Cache"
// (sections 14-17 and the section 20 teaching model): the free list is a
// stack that initially hands out blocks 0, 1, 2, ...; a shared, partly
// filled tail block is cloned into a fresh block before the first write
// (copy-on-write); blocks return to the free list when their count reaches
// zero; running out of blocks changes nothing.  The payload is not kept
// here: the planned slot and copy pair drive pa_reshape_and_cache and
// pa_copy_blocks on the GPU.
//
// Swapping (same page, section 19, item 4): a batch of sequences can move
// to a pool of host blocks and back.  Every distinct device block of the
// batch gets one host block, referenced by as many sequences of the batch
// as shared it; the device blocks lose those references (and are freed or
// queued as usual).  Swapping in is the mirror image.  Both plan only: the
// returned (source, destination) pairs drive pa_swap_blocks.
//
// Prefix caching (same page, section 18; "PagedAttention in vLLM: scattered
// memory, exact attention", section 6; "PagedAttention and KV Memory"): a
// full block whose token ids are known is registered under a key made of its
// tokens and its parent's key, so two blocks match only when their whole
// prefix matches.  A registered block whose count drops to zero is not freed
// but kept, least recently released first, in an eviction queue; a later
// prompt with the same prefix revives it (count 0 -> 1) instead of writing
// it again.  Fresh blocks come from the free list first and only then by
// evicting the queue's oldest block.  The key of a block is exact: every
// distinct token prefix that ends on a block boundary is interned once as a
// node (its parent prefix's node id and the block's token ids), and two keys
// are equal only when they are the same node.  A 64-bit chained hash only
// buckets the nodes; a lookup compares the parent node id and the token ids,
// so a hash collision costs a comparison and can never reuse the wrong KV.
// A node lives while a registered block, a sequence or a child node holds it.

#include <algorithm>
#include <cstdint>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

constexpr uint64_t kRootKey = 0x9E3779B97F4A7C15ull;

uint64_t mix64(uint64_t x) {                 // splitmix64 finaliser
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

uint64_t block_key(uint64_t parent, const int32_t* tokens, int n) {
    uint64_t h = mix64(parent);
    for (int i = 0; i < n; ++i) h = mix64(h ^ (uint64_t)(uint32_t)tokens[i]);
    return h;
}

struct Sequence {
    std::vector<int32_t> table;   // logical block -> physical block (host block while swapped)
    bool swapped = false;
    int32_t length = 0;           // cached positions
    bool has_tokens = false;      // token ids known: full blocks can be registered
    std::vector<int32_t> tokens;  // token id of every position (when has_tokens)
    std::vector<int64_t> keys;    // prefix node of every full block (when has_tokens and caching)
};

// One interned prefix: the prefix of its parent node (0 = the empty prefix)
// followed by one block of token ids.
struct PrefixNode {
    int64_t parent;
    uint64_t hash;
    int64_t holders;              // registered blocks, sequences and child nodes holding it
    std::vector<int32_t> tokens;
};

}  // namespace

struct pa_alloc {
    int32_t num_blocks;
    int32_t block_size;
    std::vector<int32_t> free_stack;          // top = back()
    std::vector<int32_t> refs;
    std::unordered_map<int64_t, Sequence> seqs;
    int64_t num_cow_copies = 0;
    // prefix cache
    bool caching = false;
    std::unordered_map<int64_t, PrefixNode> nodes;      // node id -> interned prefix
    std::unordered_multimap<uint64_t, int64_t> by_hash; // bucket -> node ids
    int64_t next_node = 1;
    uint64_t hash_mask = ~0ull;                         // test hook: fewer bits, more collisions
    std::unordered_map<int64_t, int32_t> index;         // node -> registered block
    std::vector<char> registered;
    std::vector<int64_t> reg_node;
    std::list<int32_t> lru;                             // zero-count registered blocks, oldest first
    std::vector<std::list<int32_t>::iterator> lru_pos;
    std::vector<char> in_lru;
    int64_t prompt_tokens = 0, cached_tokens = 0;
    // swap space
    int32_t num_host_blocks = 0;
    std::vector<int32_t> host_free;                     // top = back()
    std::vector<int32_t> host_refs;
    int32_t num_swapped = 0;
    int64_t swap_outs = 0;                              // sequences swapped out since creation

    pa_alloc(int nb, int bs)
        : num_blocks(nb), block_size(bs), refs(nb, 0), registered(nb, 0), reg_node(nb, 0), lru_pos(nb),
          in_lru(nb, 0) {
        free_stack.reserve(nb);
        for (int b = nb - 1; b >= 0; --b) free_stack.push_back(b);
    }

    int64_t available() const { return (int64_t)free_stack.size() + (int64_t)lru.size(); }

    // The node of prefix `parent` + tokens[0 .. block_size), or -1.
    int64_t find_node(int64_t parent, const int32_t* tokens) const {
        const uint64_t h = block_key(parent ? nodes.at(parent).hash : kRootKey, tokens, block_size) & hash_mask;
        auto range = by_hash.equal_range(h);
        for (auto it = range.first; it != range.second; ++it) {
            const PrefixNode& n = nodes.at(it->second);
            if (n.parent == parent && std::equal(tokens, tokens + block_size, n.tokens.begin())) return it->second;
        }
        return -1;
    }

    // That node, created if new; the caller holds it (release with drop_node).
    int64_t intern(int64_t parent, const int32_t* tokens) {
        int64_t id = find_node(parent, tokens);
        if (id >= 0) {
            nodes.at(id).holders += 1;
            return id;
        }
        id = next_node++;
        PrefixNode n;
        n.parent = parent;
        n.hash = block_key(parent ? nodes.at(parent).hash : kRootKey, tokens, block_size);
        n.holders = 1;
        n.tokens.assign(tokens, tokens + block_size);
        by_hash.emplace(n.hash & hash_mask, id);
        nodes.emplace(id, std::move(n));
        if (parent) nodes.at(parent).holders += 1;
        return id;
    }

    void hold_node(int64_t id) {
        if (id) nodes.at(id).holders += 1;
    }

    // Let go of a node; one that nothing holds any more is forgotten, and so
    // is its parent in turn.
    void drop_node(int64_t id) {
        while (id) {
            auto it = nodes.find(id);
            if (--it->second.holders > 0) return;
            auto range = by_hash.equal_range(it->second.hash & hash_mask);
            for (auto h = range.first; h != range.second; ++h)
                if (h->second == id) {
                    by_hash.erase(h);
                    break;
                }
            const int64_t parent = it->second.parent;
            nodes.erase(it);
            id = parent;
        }
    }

    void drop_keys(Sequence& s) {
        for (int64_t k : s.keys) drop_node(k);
        s.keys.clear();
    }

    void unregister(int32_t b) {
        if (!registered[b]) return;
        auto it = index.find(reg_node[b]);
        if (it != index.end() && it->second == b) index.erase(it);
        registered[b] = 0;
        drop_node(reg_node[b]);
        reg_node[b] = 0;
    }

    void register_block(int32_t b, int64_t node) {
        if (index.count(node)) return;          // another block already holds this prefix
        index.emplace(node, b);
        registered[b] = 1;
        reg_node[b] = node;
        hold_node(node);
    }

    // Registered block holding this prefix node, or -1.
    int32_t lookup(int64_t node) const {
        if (node < 0) return -1;
        auto it = index.find(node);
        return it == index.end() ? -1 : it->second;
    }

    void lru_remove(int32_t b) {
        if (!in_lru[b]) return;
        lru.erase(lru_pos[b]);
        in_lru[b] = 0;
    }

    // A fresh block with count 1: from the free list, else the queue's oldest.
    int32_t take() {
        int32_t b;
        if (!free_stack.empty()) {
            b = free_stack.back();
            free_stack.pop_back();
        } else {
            b = lru.front();
            lru_remove(b);
            unregister(b);
        }
        refs[b] = 1;
        return b;
    }

    int append(int64_t seq, int64_t* slot, int32_t* src, int32_t* dst, const int32_t* token) {
        auto it = seqs.find(seq);
        if (it == seqs.end()) return PA_ERR_UNKNOWN_SEQ;
        Sequence& s = it->second;
        if (s.swapped) return PA_ERR_SWAPPED;
        const int32_t off = s.length % block_size;
        int32_t cs = -1, cd = -1, blk;
        if (off != 0) {
            const int32_t tail = s.table.back();
            if (refs[tail] > 1) {                       // shared tail: clone first
                if (available() == 0) return PA_FAIL_NO_BLOCKS;
                blk = take();
                refs[tail] -= 1;
                s.table.back() = blk;
                cs = tail;
                cd = blk;
                ++num_cow_copies;
            } else {
                blk = tail;                              // private tail: in place
            }
        } else {
            if (available() == 0) return PA_FAIL_NO_BLOCKS;
            blk = take();                                // tail full: new block
            s.table.push_back(blk);
        }
        *slot = (int64_t)blk * block_size + off;
        *src = cs;
        *dst = cd;
        s.length += 1;
        if (!token) {
            s.has_tokens = false;                        // content no longer known
            s.tokens.clear();
            drop_keys(s);
        } else if (s.has_tokens) {
            s.tokens.push_back(*token);
            if (caching && off == block_size - 1) {      // the block just became full
                const int64_t parent = s.keys.empty() ? 0 : s.keys.back();
                const int64_t node = intern(parent, s.tokens.data() + (s.length - block_size));
                s.keys.push_back(node);
                register_block(blk, node);
            }
        }
        return PA_OK;
    }

    // Drop one reference; a block that reaches zero goes to the free list, or
    // to the eviction queue when it is registered.
    void release_table(const std::vector<int32_t>& table) {
        std::vector<int32_t> to_queue;
        for (int32_t b : table) {
            refs[b] -= 1;
            if (refs[b] == 0) {
                if (registered[b])
                    to_queue.push_back(b);
                else
                    free_stack.push_back(b);
            }
        }
        // deeper blocks first, so that a chain is evicted from its tail end
        for (auto it = to_queue.rbegin(); it != to_queue.rend(); ++it) {
            lru.push_back(*it);
            lru_pos[*it] = std::prev(lru.end());
            in_lru[*it] = 1;
        }
    }
};

extern "C" {

pa_alloc_t* pa_alloc_create(int num_blocks, int block_size) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    return new (std::nothrow) pa_alloc(num_blocks, block_size);
}

void pa_alloc_destroy(pa_alloc_t* a) { delete a; }

int pa_alloc_set_free_order(pa_alloc_t* a, const int32_t* order, int n) {
    if (!a || !order || n != a->num_blocks || !a->seqs.empty() || !a->lru.empty()) return PA_ERR_INVALID_ARG;
    if ((int)a->free_stack.size() != a->num_blocks) return PA_ERR_INVALID_ARG;
    std::vector<char> seen(a->num_blocks, 0);
    for (int i = 0; i < n; ++i) {
        if (order[i] < 0 || order[i] >= a->num_blocks || seen[order[i]]) return PA_ERR_INVALID_ARG;
        seen[order[i]] = 1;
    }
    a->free_stack.assign(order, order + n);
    return PA_OK;
}

int pa_alloc_sequence(pa_alloc_t* a, int64_t seq, int num_tokens) {
    if (!a) return PA_ERR_INVALID_ARG;
    if (a->seqs.count(seq)) return PA_ERR_DUPLICATE_SEQ;
    if (num_tokens <= 0) return PA_ERR_INVALID_ARG;
    const int64_t need = ((int64_t)num_tokens + a->block_size - 1) / a->block_size;
    if (a->available() < need) return PA_FAIL_NO_BLOCKS;
    Sequence s;
    s.table.reserve(need);
    for (int64_t i = 0; i < need; ++i) s.table.push_back(a->take());
    s.length = num_tokens;
    a->seqs.emplace(seq, std::move(s));
    a->prompt_tokens += num_tokens;
    return PA_OK;
}

int pa_alloc_sequence_tokens(pa_alloc_t* a, int64_t seq, const int32_t* tokens, int num_tokens,
                             int* num_cached_tokens) {
    if (!a || !num_cached_tokens) return PA_ERR_INVALID_ARG;
    *num_cached_tokens = 0;
    if (a->seqs.count(seq)) return PA_ERR_DUPLICATE_SEQ;
    if (num_tokens <= 0 || !tokens) return PA_ERR_INVALID_ARG;
    const int B = a->block_size;
    const int64_t need = ((int64_t)num_tokens + B - 1) / B;
    const int full = num_tokens / B;
    // plan: the leading full blocks already cached (a registered block's
    // prefix node exists, so the walk stops at the first prefix without one)
    std::vector<int32_t> hits;
    int64_t revived_from_queue = 0;
    if (a->caching) {
        int64_t parent = 0;
        for (int i = 0; i < full; ++i) {
            const int64_t node = a->find_node(parent, tokens + (size_t)i * B);
            const int32_t b = a->lookup(node);
            if (b < 0) break;
            hits.push_back(b);
            revived_from_queue += a->in_lru[b] ? 1 : 0;
            parent = node;
        }
    }
    const int64_t fresh = need - (int64_t)hits.size();
    if (a->available() - revived_from_queue < fresh) return PA_FAIL_NO_BLOCKS;
    // apply
    Sequence s;
    s.table.reserve(need);
    for (int32_t b : hits) {
        a->lru_remove(b);                  // a cached block with count 0 comes back to 1
        a->refs[b] += 1;
        s.table.push_back(b);
    }
    for (int64_t i = (int64_t)hits.size(); i < need; ++i) s.table.push_back(a->take());
    if (a->caching) {                      // every full block's prefix node; fresh ones registered
        int64_t parent = 0;
        for (int i = 0; i < full; ++i) {
            parent = a->intern(parent, tokens + (size_t)i * B);
            s.keys.push_back(parent);
            if (i >= (int)hits.size()) a->register_block(s.table[i], parent);
        }
    }
    s.length = num_tokens;
    s.has_tokens = true;
    s.tokens.assign(tokens, tokens + num_tokens);
    a->seqs.emplace(seq, std::move(s));
    *num_cached_tokens = (int)hits.size() * B;
    a->prompt_tokens += num_tokens;
    a->cached_tokens += *num_cached_tokens;
    return PA_OK;
}

int pa_alloc_fork(pa_alloc_t* a, int64_t parent, int64_t child) {
    if (!a) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    if (a->seqs.count(child)) return PA_ERR_DUPLICATE_SEQ;
    if (it->second.swapped) return PA_ERR_SWAPPED;
    Sequence s = it->second;                 // copy before insert (rehash)
    for (int32_t b : s.table) a->refs[b] += 1;
    for (int64_t k : s.keys) a->hold_node(k);
    a->seqs.emplace(child, std::move(s));
    return PA_OK;
}

int pa_alloc_append_slot(pa_alloc_t* a, int64_t seq, int64_t* slot_out,
                         int32_t* cow_src, int32_t* cow_dst) {
    if (!a || !slot_out || !cow_src || !cow_dst) return PA_ERR_INVALID_ARG;
    return a->append(seq, slot_out, cow_src, cow_dst, nullptr);
}

int pa_alloc_append_token(pa_alloc_t* a, int64_t seq, int32_t token, int64_t* slot_out, int32_t* cow_src,
                          int32_t* cow_dst) {
    if (!a || !slot_out || !cow_src || !cow_dst) return PA_ERR_INVALID_ARG;
    return a->append(seq, slot_out, cow_src, cow_dst, &token);
}

int pa_alloc_append_slots(pa_alloc_t* a, const int64_t* seqs, int n, int64_t* slots_out,
                          int32_t* cow_pairs_out, int cow_capacity, int* num_cow, int* num_done) {
    if (!a || n < 0 || (n > 0 && (!seqs || !slots_out)) || !num_cow) return PA_ERR_INVALID_ARG;
    *num_cow = 0;
    if (num_done) *num_done = 0;
    for (int i = 0; i < n; ++i) {
        int32_t src, dst;
        if (*num_cow >= cow_capacity || !cow_pairs_out) {
            // A copy may be needed; refuse up front rather than lose a pair.
            const auto it = a->seqs.find(seqs[i]);
            if (it != a->seqs.end() && it->second.length % a->block_size != 0 &&
                a->refs[it->second.table.back()] > 1)
                return PA_ERR_INVALID_ARG;
        }
        int st = a->append(seqs[i], &slots_out[i], &src, &dst, nullptr);
        if (st != PA_OK) return st;
        if (src >= 0) {
            cow_pairs_out[2 * (*num_cow)] = src;
            cow_pairs_out[2 * (*num_cow) + 1] = dst;
            *num_cow += 1;
        }
        if (num_done) *num_done = i + 1;
    }
    return PA_OK;
}

int pa_alloc_free(pa_alloc_t* a, int64_t seq) {
    if (!a) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return PA_OK;
    if (it->second.swapped) {
        for (int32_t h : it->second.table)
            if (--a->host_refs[h] == 0) a->host_free.push_back(h);
        --a->num_swapped;
    } else {
        a->release_table(it->second.table);
    }
    a->drop_keys(it->second);
    a->seqs.erase(it);
    return PA_OK;
}

int pa_alloc_block_table(const pa_alloc_t* a, int64_t seq, int32_t* out, int cap, int* n_out) {
    if (!a || !n_out) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    const auto& t = it->second.table;
    *n_out = (int)t.size();
    if ((int)t.size() > cap || (!out && !t.empty())) return PA_ERR_INVALID_ARG;
    std::copy(t.begin(), t.end(), out);
    return PA_OK;
}

int pa_alloc_build_tables(const pa_alloc_t* a, const int64_t* seqs, int n, int32_t* tables,
                          int max_blocks, int32_t* context_lens) {
    if (!a || n < 0 || max_blocks < 0 || (n > 0 && (!seqs || !tables || !context_lens)))
        return PA_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seqs[i]);
        if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
        if (it->second.swapped) return PA_ERR_SWAPPED;
        const auto& t = it->second.table;
        if ((int)t.size() > max_blocks) return PA_ERR_INVALID_ARG;
        int32_t* row = tables + (size_t)i * max_blocks;
        std::copy(t.begin(), t.end(), row);
        std::fill(row + t.size(), row + max_blocks, -1);
        context_lens[i] = it->second.length;
    }
    return PA_OK;
}

int pa_alloc_slot_mapping(const pa_alloc_t* a, int64_t seq, int start, int n, int64_t* out) {
    if (!a || n < 0 || start < 0 || (n > 0 && !out)) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    const Sequence& s = it->second;
    if (s.swapped) return PA_ERR_SWAPPED;
    if ((int64_t)start + n > s.length) return PA_ERR_INVALID_ARG;
    const int B = a->block_size;
    for (int k = 0; k < n; ++k) {
        const int i = start + k;
        out[k] = (int64_t)s.table[i / B] * B + i % B;
    }
    return PA_OK;
}

int pa_alloc_seq_len(const pa_alloc_t* a, int64_t seq) {
    if (!a) return -1;
    auto it = a->seqs.find(seq);
    return it == a->seqs.end() ? -1 : it->second.length;
}

int pa_alloc_ref_count(const pa_alloc_t* a, int32_t block) {
    if (!a || block < 0 || block >= a->num_blocks) return -1;
    return a->refs[block];
}

int pa_alloc_num_free(const pa_alloc_t* a) { return a ? (int)a->free_stack.size() : -1; }

int pa_alloc_free_list(const pa_alloc_t* a, int32_t* out, int cap) {
    if (!a) return -1;
    const int n = (int)a->free_stack.size();
    if (out) std::copy(a->free_stack.begin(), a->free_stack.begin() + std::min(n, std::max(cap, 0)), out);
    return n;
}

int pa_alloc_get_stats(const pa_alloc_t* a, pa_alloc_stats_t* out) {
    if (!a || !out) return PA_ERR_INVALID_ARG;
    out->num_blocks = a->num_blocks;
    out->num_free = (int32_t)a->free_stack.size();
    out->num_cached = (int32_t)a->lru.size();
    out->num_used = a->num_blocks - out->num_free - out->num_cached;
    out->num_seqs = (int32_t)a->seqs.size();
    out->num_cow_copies = a->num_cow_copies;
    out->num_swapped = a->num_swapped;
    out->num_prompt_tokens = a->prompt_tokens;
    out->num_cached_tokens = a->cached_tokens;
    out->num_swap_outs = a->swap_outs;
    int64_t ctx = 0;
    for (const auto& kv : a->seqs) ctx += kv.second.length;
    out->num_context_tokens = ctx;
    return PA_OK;
}

int pa_alloc_enable_prefix_caching(pa_alloc_t* a, int enable) {
    if (!a || !a->seqs.empty()) return PA_ERR_INVALID_ARG;
    if (!enable) {                                  // forget the cache: queued blocks become free
        for (int32_t b : a->lru) {
            a->in_lru[b] = 0;
            a->free_stack.push_back(b);
        }
        a->lru.clear();
        for (int32_t b = 0; b < a->num_blocks; ++b) a->unregister(b);
        a->index.clear();
    }
    a->caching = enable != 0;
    return PA_OK;
}

int pa_alloc_set_key_mask(pa_alloc_t* a, uint64_t mask) {
    if (!a || !a->seqs.empty() || !a->nodes.empty()) return PA_ERR_INVALID_ARG;
    a->hash_mask = mask;
    return PA_OK;
}

int pa_alloc_num_prefix_nodes(const pa_alloc_t* a) { return a ? (int)a->nodes.size() : -1; }

int pa_alloc_num_cached(const pa_alloc_t* a) { return a ? (int)a->lru.size() : -1; }

int pa_alloc_enable_swap(pa_alloc_t* a, int num_host_blocks) {
    if (!a || num_host_blocks < 0 || a->num_swapped != 0) return PA_ERR_INVALID_ARG;
    a->num_host_blocks = num_host_blocks;
    a->host_refs.assign(num_host_blocks, 0);
    a->host_free.clear();
    for (int b = num_host_blocks - 1; b >= 0; --b) a->host_free.push_back(b);
    return PA_OK;
}

int pa_alloc_num_free_host(const pa_alloc_t* a) { return a ? (int)a->host_free.size() : -1; }

int pa_alloc_is_swapped(const pa_alloc_t* a, int64_t seq) {
    if (!a) return -1;
    auto it = a->seqs.find(seq);
    return it == a->seqs.end() ? -1 : (it->second.swapped ? 1 : 0);
}

// Shared by swap_out and swap_in: check the batch (known, distinct, all in
// state `from_swapped`), collect its distinct blocks in first-appearance
// order with the number of batch sequences referencing each.
static int swap_plan(pa_alloc_t* a, const int64_t* seqs, int n, bool from_swapped, std::vector<int32_t>& blocks,
                     std::vector<int32_t>& counts) {
    if (n < 0 || (n > 0 && !seqs)) return PA_ERR_INVALID_ARG;
    std::unordered_map<int32_t, int32_t> index;
    std::unordered_map<int64_t, char> seen;
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seqs[i]);
        if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
        if (it->second.swapped != from_swapped) return from_swapped ? PA_ERR_INVALID_ARG : PA_ERR_SWAPPED;
        if (seen.count(seqs[i])) return PA_ERR_INVALID_ARG;
        seen.emplace(seqs[i], 1);
        for (int32_t b : it->second.table) {
            auto f = index.find(b);
            if (f == index.end()) {
                index.emplace(b, (int32_t)blocks.size());
                blocks.push_back(b);
                counts.push_back(1);
            } else {
                counts[f->second] += 1;
            }
        }
    }
    return PA_OK;
}

int pa_alloc_swap_out(pa_alloc_t* a, const int64_t* seqs, int n, int32_t* pairs_out, int pair_capacity,
                      int* num_pairs) {
    if (!a || !num_pairs) return PA_ERR_INVALID_ARG;
    *num_pairs = 0;
    std::vector<int32_t> blocks, counts;
    int st = swap_plan(a, seqs, n, false, blocks, counts);
    if (st != PA_OK) return st;
    *num_pairs = (int)blocks.size();
    if ((int)blocks.size() > pair_capacity || (!pairs_out && !blocks.empty())) return PA_ERR_INVALID_ARG;
    if (blocks.size() > a->host_free.size()) return PA_FAIL_NO_BLOCKS;
    std::unordered_map<int32_t, int32_t> to_host;
    for (size_t i = 0; i < blocks.size(); ++i) {
        const int32_t hb = a->host_free.back();
        a->host_free.pop_back();
        a->host_refs[hb] = counts[i];
        to_host.emplace(blocks[i], hb);
        pairs_out[2 * i] = blocks[i];
        pairs_out[2 * i + 1] = hb;
    }
    for (int i = 0; i < n; ++i) {
        Sequence& s = a->seqs.find(seqs[i])->second;
        a->release_table(s.table);            // device references go (blocks freed or queued at 0)
        for (int32_t& b : s.table) b = to_host[b];
        s.swapped = true;
        ++a->num_swapped;
        ++a->swap_outs;
    }
    return PA_OK;
}

int pa_alloc_swap_in(pa_alloc_t* a, const int64_t* seqs, int n, int32_t* pairs_out, int pair_capacity,
                     int* num_pairs) {
    if (!a || !num_pairs) return PA_ERR_INVALID_ARG;
    *num_pairs = 0;
    std::vector<int32_t> blocks, counts;
    int st = swap_plan(a, seqs, n, true, blocks, counts);
    if (st != PA_OK) return st;
    *num_pairs = (int)blocks.size();
    if ((int)blocks.size() > pair_capacity || (!pairs_out && !blocks.empty())) return PA_ERR_INVALID_ARG;
    if ((int64_t)blocks.size() > a->available()) return PA_FAIL_NO_BLOCKS;
    std::unordered_map<int32_t, int32_t> to_dev;
    for (size_t i = 0; i < blocks.size(); ++i) {
        const int32_t db = a->take();
        a->refs[db] = counts[i];
        to_dev.emplace(blocks[i], db);
        pairs_out[2 * i] = blocks[i];
        pairs_out[2 * i + 1] = db;
    }
    for (int i = 0; i < n; ++i) {
        Sequence& s = a->seqs.find(seqs[i])->second;
        for (int32_t& h : s.table) {
            if (--a->host_refs[h] == 0) a->host_free.push_back(h);
            h = to_dev[h];
        }
        s.swapped = false;
        --a->num_swapped;
    }
    return PA_OK;
}

int pa_alloc_cached_list(const pa_alloc_t* a, int32_t* out, int cap) {
    if (!a) return -1;
    int i = 0;
    for (int32_t b : a->lru) {
        if (out && i < cap) out[i] = b;
        ++i;
    }
    return i;
}

}  // extern "C"
