// Host block manager: free list, reference counts, fork, append with
// copy-on-write planning, release.
//
// Semantics follow "PagedAttention: Virtual Memory for the KV Cache"
// (sections 14-17 and the section 20 teaching model): the free list is a
// stack that initially hands out blocks 0, 1, 2, ...; a shared, partly
// filled tail block is cloned into a fresh block before the first write
// (copy-on-write); blocks return to the free list when their count reaches
// zero; running out of blocks changes nothing.  The payload is not kept
// here: the planned slot and copy pair drive pa_reshape_and_cache and
// pa_copy_blocks on the GPU.

#include <algorithm>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

struct Sequence {
    std::vector<int32_t> table;   // logical block -> physical block
    int32_t length = 0;           // cached positions
};

}  // namespace

struct pa_alloc {
    int32_t num_blocks;
    int32_t block_size;
    std::vector<int32_t> free_stack;          // top = back()
    std::vector<int32_t> refs;
    std::unordered_map<int64_t, Sequence> seqs;
    int64_t num_cow_copies = 0;

    pa_alloc(int nb, int bs) : num_blocks(nb), block_size(bs), refs(nb, 0) {
        free_stack.reserve(nb);
        for (int b = nb - 1; b >= 0; --b) free_stack.push_back(b);
    }

    int32_t take() {
        int32_t b = free_stack.back();
        free_stack.pop_back();
        refs[b] = 1;
        return b;
    }

    int append(int64_t seq, int64_t* slot, int32_t* src, int32_t* dst) {
        auto it = seqs.find(seq);
        if (it == seqs.end()) return PA_ERR_UNKNOWN_SEQ;
        Sequence& s = it->second;
        const int32_t off = s.length % block_size;
        int32_t cs = -1, cd = -1, blk;
        if (off != 0) {
            const int32_t tail = s.table.back();
            if (refs[tail] > 1) {                       // shared tail: clone first
                if (free_stack.empty()) return PA_FAIL_NO_BLOCKS;
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
            if (free_stack.empty()) return PA_FAIL_NO_BLOCKS;
            blk = take();                                // tail full: new block
            s.table.push_back(blk);
        }
        *slot = (int64_t)blk * block_size + off;
        *src = cs;
        *dst = cd;
        s.length += 1;
        return PA_OK;
    }
};

extern "C" {

pa_alloc_t* pa_alloc_create(int num_blocks, int block_size) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    return new (std::nothrow) pa_alloc(num_blocks, block_size);
}

void pa_alloc_destroy(pa_alloc_t* a) { delete a; }

int pa_alloc_set_free_order(pa_alloc_t* a, const int32_t* order, int n) {
    if (!a || !order || n != a->num_blocks || !a->seqs.empty()) return PA_ERR_INVALID_ARG;
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
    if ((int64_t)a->free_stack.size() < need) return PA_FAIL_NO_BLOCKS;
    Sequence s;
    s.table.reserve(need);
    for (int64_t i = 0; i < need; ++i) s.table.push_back(a->take());
    s.length = num_tokens;
    a->seqs.emplace(seq, std::move(s));
    return PA_OK;
}

int pa_alloc_fork(pa_alloc_t* a, int64_t parent, int64_t child) {
    if (!a) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end()) return PA_ERR_UNKNOWN_SEQ;
    if (a->seqs.count(child)) return PA_ERR_DUPLICATE_SEQ;
    Sequence s = it->second;                 // copy before insert (rehash)
    for (int32_t b : s.table) a->refs[b] += 1;
    a->seqs.emplace(child, std::move(s));
    return PA_OK;
}

int pa_alloc_append_slot(pa_alloc_t* a, int64_t seq, int64_t* slot_out,
                         int32_t* cow_src, int32_t* cow_dst) {
    if (!a || !slot_out || !cow_src || !cow_dst) return PA_ERR_INVALID_ARG;
    return a->append(seq, slot_out, cow_src, cow_dst);
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
        int st = a->append(seqs[i], &slots_out[i], &src, &dst);
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
    for (int32_t b : it->second.table) {
        a->refs[b] -= 1;
        if (a->refs[b] == 0) a->free_stack.push_back(b);
    }
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
    out->num_used = a->num_blocks - out->num_free;
    out->num_seqs = (int32_t)a->seqs.size();
    out->num_cow_copies = a->num_cow_copies;
    return PA_OK;
}

}  // extern "C"
