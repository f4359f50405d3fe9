// Host KV block manager: free list, reference counts, on-demand allocation,
// fork, and copy-on-write of the last shared block.
//
// Follows the wywy.jp notes ("KV cache manager", "Reference count",
// "Copy-on-write" and the parallel-sampling walkthrough: a write into a last
// logical block whose physical block is shared allocates a new block, has the
// block engine copy the old one, and drops the old count by one; the last
// holder writes in place) and the zhaifeiyue.github.io detail page's Memory
// Management table (Allocate when the previous logical block is full; Free the
// whole request; Copy-on-Write one block when its count exceeds one).  Slots
// follow the ricepunchb garden's section 3.2: table[pos / B] * B + pos mod B.
//
// The pages leave the free-list order open.  Here it starts as a seeded
// permutation (Fisher-Yates over SplitMix64), allocation takes the front and a
// freed block goes to the back, so block tables are reproducible.
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv_internal.h"

namespace {

struct SplitMix64 {
    uint64_t state;
    uint64_t next() {
        state += 0x9E3779B97F4A7C15ull;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        return z ^ (z >> 31);
    }
};

struct Sequence {
    std::vector<int32_t> table;   // GPU block ids, or CPU block ids while swapped out
    int32_t ctx = 0;
    bool swapped = false;
};

std::vector<int32_t> seeded_permutation(int64_t n, uint64_t seed) {
    std::vector<int32_t> perm((size_t)n);
    for (int64_t i = 0; i < n; ++i) perm[(size_t)i] = (int32_t)i;
    SplitMix64 rng{seed};
    for (int64_t i = n - 1; i > 0; --i) {
        const int64_t j = (int64_t)(rng.next() % (uint64_t)(i + 1));
        const int32_t t = perm[(size_t)i];
        perm[(size_t)i] = perm[(size_t)j];
        perm[(size_t)j] = t;
    }
    return perm;
}

}  // namespace

struct pkv_bm {
    int64_t num_blocks;
    int B;
    std::deque<int32_t> free_list;
    std::vector<int32_t> ref;
    std::unordered_map<int64_t, Sequence> seqs;
    // CPU swap pool (empty until pkv_bm_add_cpu_pool)
    int64_t num_cpu_blocks = 0;
    std::deque<int32_t> cpu_free;
    std::vector<int32_t> cpu_ref;

    int64_t slot_of(const Sequence& sq, int64_t pos) const {
        return (int64_t)sq.table[pos / B] * B + pos % B;
    }
    int32_t take() {
        const int32_t b = free_list.front();
        free_list.pop_front();
        ref[b] = 1;
        return b;
    }
    // Blocks one append of `sq` consumes: a fresh block at a block boundary,
    // a copy-on-write block when the partial last block is shared, else none.
    int blocks_for_append(const Sequence& sq) const {
        if (sq.ctx % B == 0) return 1;
        return ref[sq.table.back()] > 1 ? 1 : 0;
    }
    void append(Sequence& sq, int64_t* slot, int32_t* src, int32_t* dst) {
        const int64_t pos = sq.ctx;
        *src = -1;
        *dst = -1;
        if (pos % B == 0) {
            sq.table.push_back(take());
        } else {
            const int32_t last = sq.table.back();
            if (ref[last] > 1) {
                const int32_t fresh = take();
                ref[last] -= 1;
                sq.table.back() = fresh;
                *src = last;
                *dst = fresh;
            }
        }
        sq.ctx = (int32_t)(pos + 1);
        *slot = slot_of(sq, pos);
    }
};

extern "C" {

pkv_status pkv_bm_create(int64_t num_blocks, int block_size, uint64_t seed, pkv_bm** out) {
    if (!out) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_create: out is NULL");
    *out = nullptr;
    if (num_blocks < 1 || num_blocks > INT32_MAX)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_create: num_blocks must be in [1, 2^31)");
    if (block_size < 1) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_create: block_size must be >= 1");
    pkv_bm* bm = new (std::nothrow) pkv_bm;
    if (!bm) return pkv::fail(PKV_ERR_OOM, "pkv_bm_create: host allocation failed");
    bm->num_blocks = num_blocks;
    bm->B = block_size;
    std::vector<int32_t> perm = seeded_permutation(num_blocks, seed);
    bm->free_list.assign(perm.begin(), perm.end());
    bm->ref.assign((size_t)num_blocks, 0);
    *out = bm;
    return PKV_OK;
}

void pkv_bm_destroy(pkv_bm* bm) { delete bm; }

pkv_status pkv_bm_add_sequence(pkv_bm* bm, int64_t seq_id, int32_t prompt_len,
                               int64_t* slots_out) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_add_sequence: NULL manager");
    if (prompt_len < 0) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_add_sequence: negative length");
    if (bm->seqs.count(seq_id))
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_add_sequence: sequence %lld exists",
                         (long long)seq_id);
    const int64_t need = ((int64_t)prompt_len + bm->B - 1) / bm->B;
    if (need > (int64_t)bm->free_list.size())
        return pkv::fail(PKV_ERR_OOM, "pkv_bm_add_sequence: %lld blocks needed, %zu free",
                         (long long)need, bm->free_list.size());
    Sequence sq;
    sq.table.reserve((size_t)need);
    for (int64_t i = 0; i < need; ++i) sq.table.push_back(bm->take());
    sq.ctx = prompt_len;
    if (slots_out)
        for (int64_t p = 0; p < prompt_len; ++p) slots_out[p] = bm->slot_of(sq, p);
    bm->seqs.emplace(seq_id, std::move(sq));
    return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_bm* bm, int64_t parent, int64_t child) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_fork: NULL manager");
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end() || bm->seqs.count(child))
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_fork: unknown parent or existing child");
    if (it->second.swapped)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_fork: parent is swapped out");
    Sequence sq = it->second;
    for (int32_t b : sq.table) bm->ref[b] += 1;
    bm->seqs.emplace(child, std::move(sq));
    return PKV_OK;
}

pkv_status pkv_bm_append_slot(pkv_bm* bm, int64_t seq_id, int64_t* slot, int32_t* cow_src,
                              int32_t* cow_dst) {
    if (!bm || !slot || !cow_src || !cow_dst)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_append_slot: NULL argument");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_append_slot: unknown sequence %lld",
                         (long long)seq_id);
    if (it->second.ctx == INT32_MAX || it->second.swapped)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_append_slot: sequence full or swapped out");
    if (bm->blocks_for_append(it->second) > (int)bm->free_list.size())
        return pkv::fail(PKV_ERR_OOM, "pkv_bm_append_slot: no free block");
    bm->append(it->second, slot, cow_src, cow_dst);
    return PKV_OK;
}

pkv_status pkv_bm_append_slots(pkv_bm* bm, const int64_t* seq_ids, int n, int64_t* slots,
                               int32_t* pairs, int32_t* num_pairs) {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots || !pairs)) || !num_pairs)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_append_slots: bad argument");
    // Check first (all-or-nothing): known, distinct sequences, and enough blocks.
    std::unordered_map<int64_t, int> seen;
    int64_t need = 0;
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() || seen.count(seq_ids[i]) || it->second.ctx == INT32_MAX ||
            it->second.swapped)
            return pkv::fail(PKV_ERR_INVALID,
                             "pkv_bm_append_slots: unknown, repeated, full or swapped-out "
                             "sequence %lld",
                             (long long)seq_ids[i]);
        seen[seq_ids[i]] = i;
    }
    // Appends are applied in order, and a copy-on-write by an earlier sequence
    // can lower the count a later one sees, so count on a scratch copy.
    {
        std::unordered_map<int32_t, int32_t> refd;
        for (int i = 0; i < n; ++i) {
            const Sequence& sq = bm->seqs.find(seq_ids[i])->second;
            if (sq.ctx % bm->B == 0) {
                need += 1;
                continue;
            }
            const int32_t last = sq.table.back();
            auto r = refd.find(last);
            const int32_t cnt = r == refd.end() ? bm->ref[last] : r->second;
            if (cnt > 1) {
                need += 1;
                refd[last] = cnt - 1;
            }
        }
    }
    if (need > (int64_t)bm->free_list.size())
        return pkv::fail(PKV_ERR_OOM, "pkv_bm_append_slots: %lld blocks needed, %zu free",
                         (long long)need, bm->free_list.size());
    int32_t np = 0;
    for (int i = 0; i < n; ++i) {
        int32_t src, dst;
        bm->append(bm->seqs.find(seq_ids[i])->second, &slots[i], &src, &dst);
        if (src >= 0) {
            pairs[2 * np] = src;
            pairs[2 * np + 1] = dst;
            ++np;
        }
    }
    *num_pairs = np;
    return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_bm* bm, int64_t seq_id) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_free_sequence: NULL manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_free_sequence: unknown sequence %lld",
                         (long long)seq_id);
    if (it->second.swapped) {
        for (int32_t b : it->second.table)
            if (--bm->cpu_ref[b] == 0) bm->cpu_free.push_back(b);
    } else {
        for (int32_t b : it->second.table)
            if (--bm->ref[b] == 0) bm->free_list.push_back(b);
    }
    bm->seqs.erase(it);
    return PKV_OK;
}

pkv_status pkv_bm_block_table(const pkv_bm* bm, int64_t seq_id, int32_t* out, int32_t cap,
                              int32_t* n) {
    if (!bm || !n) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_block_table: NULL argument");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_block_table: unknown sequence %lld",
                         (long long)seq_id);
    const std::vector<int32_t>& t = it->second.table;
    *n = (int32_t)t.size();
    if ((int64_t)t.size() > cap || (!out && !t.empty()))
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_block_table: capacity %d < %zu", cap, t.size());
    if (!t.empty()) std::memcpy(out, t.data(), t.size() * sizeof(int32_t));
    return PKV_OK;
}

pkv_status pkv_bm_context_len(const pkv_bm* bm, int64_t seq_id, int32_t* n) {
    if (!bm || !n) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_context_len: NULL argument");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_context_len: unknown sequence %lld",
                         (long long)seq_id);
    *n = it->second.ctx;
    return PKV_OK;
}

pkv_status pkv_bm_export(const pkv_bm* bm, const int64_t* seq_ids, int n, int32_t* tables,
                         int32_t max_blocks, int32_t* context_lens) {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !tables || !context_lens)) || max_blocks < 1)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_export: bad argument");
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end())
            return pkv::fail(PKV_ERR_INVALID, "pkv_bm_export: unknown sequence %lld",
                             (long long)seq_ids[i]);
        if ((int64_t)it->second.table.size() > max_blocks)
            return pkv::fail(PKV_ERR_INVALID, "pkv_bm_export: table longer than max_blocks");
        if (it->second.swapped)
            return pkv::fail(PKV_ERR_INVALID, "pkv_bm_export: sequence %lld is swapped out",
                             (long long)seq_ids[i]);
    }
    for (int i = 0; i < n; ++i) {
        const Sequence& sq = bm->seqs.find(seq_ids[i])->second;
        int32_t* row = tables + (int64_t)i * max_blocks;
        const size_t len = sq.table.size();
        if (len) std::memcpy(row, sq.table.data(), len * sizeof(int32_t));
        for (int64_t j = (int64_t)len; j < max_blocks; ++j) row[j] = -1;
        context_lens[i] = sq.ctx;
    }
    return PKV_OK;
}

pkv_status pkv_bm_add_cpu_pool(pkv_bm* bm, int64_t num_cpu_blocks, uint64_t seed) {
    if (!bm) return pkv::fail(PKV_ERR_INVALID, "pkv_bm_add_cpu_pool: NULL manager");
    if (bm->num_cpu_blocks != 0)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_add_cpu_pool: the manager has a CPU pool");
    if (num_cpu_blocks < 1 || num_cpu_blocks > INT32_MAX)
        return pkv::fail(PKV_ERR_INVALID, "pkv_bm_add_cpu_pool: num_cpu_blocks out of range");
    std::vector<int32_t> perm = seeded_permutation(num_cpu_blocks, seed);
    bm->cpu_free.assign(perm.begin(), perm.end());
    bm->cpu_ref.assign((size_t)num_cpu_blocks, 0);
    bm->num_cpu_blocks = num_cpu_blocks;
    return PKV_OK;
}

// Swap a group of sequences between the pools (out: GPU -> CPU, in: CPU -> GPU).
// All of their blocks move together (all-or-nothing eviction); a block shared
// with a sequence outside the group cannot move.  Distinct blocks are taken in
// first-seen order (group order, then table order); each gets a fresh block in
// the other pool with the same reference count; the old blocks are freed in
// the same order.
static pkv_status swap_group(pkv_bm* bm, const int64_t* seq_ids, int n, int32_t* pairs,
                             int32_t cap, int32_t* num_pairs, bool out, const char* fn) {
    if (!bm || n < 0 || (n > 0 && !seq_ids) || !num_pairs || cap < 0 || (cap > 0 && !pairs))
        return pkv::fail(PKV_ERR_INVALID, "%s: bad argument", fn);
    if (bm->num_cpu_blocks == 0) return pkv::fail(PKV_ERR_INVALID, "%s: no CPU pool", fn);
    std::unordered_map<int64_t, int> seen;
    std::vector<int32_t> order;                        // distinct blocks, first-seen order
    std::unordered_map<int32_t, int32_t> uses;         // references from within the group
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() || seen.count(seq_ids[i]) || it->second.swapped == out)
            return pkv::fail(PKV_ERR_INVALID, "%s: unknown, repeated or %s sequence %lld", fn,
                             out ? "already swapped-out" : "resident", (long long)seq_ids[i]);
        seen[seq_ids[i]] = i;
        for (int32_t b : it->second.table) {
            if (uses[b]++ == 0) order.push_back(b);
        }
    }
    const std::vector<int32_t>& from_ref = out ? bm->ref : bm->cpu_ref;
    for (int32_t b : order)
        if (from_ref[(size_t)b] != uses[b])
            return pkv::fail(PKV_ERR_INVALID, "%s: block %d is shared outside the group", fn, b);
    std::deque<int32_t>& to_free = out ? bm->cpu_free : bm->free_list;
    if ((int64_t)order.size() > (int64_t)to_free.size())
        return pkv::fail(PKV_ERR_OOM, "%s: %zu blocks needed, %zu free", fn, order.size(),
                         to_free.size());
    if ((int64_t)order.size() > cap)
        return pkv::fail(PKV_ERR_INVALID, "%s: %zu pairs, capacity %d", fn, order.size(), cap);
    std::vector<int32_t>& fref = out ? bm->ref : bm->cpu_ref;
    std::vector<int32_t>& tref = out ? bm->cpu_ref : bm->ref;
    std::deque<int32_t>& from_free = out ? bm->free_list : bm->cpu_free;
    std::unordered_map<int32_t, int32_t> moved;
    for (size_t k = 0; k < order.size(); ++k) {
        const int32_t b = order[k];
        const int32_t nb = to_free.front();
        to_free.pop_front();
        tref[(size_t)nb] = fref[(size_t)b];
        moved[b] = nb;
        pairs[2 * k] = b;
        pairs[2 * k + 1] = nb;
    }
    for (int32_t b : order) {
        fref[(size_t)b] = 0;
        from_free.push_back(b);
    }
    for (int i = 0; i < n; ++i) {
        Sequence& sq = bm->seqs.find(seq_ids[i])->second;
        for (int32_t& b : sq.table) b = moved[b];
        sq.swapped = out;
    }
    *num_pairs = (int32_t)order.size();
    return PKV_OK;
}

pkv_status pkv_bm_swap_out(pkv_bm* bm, const int64_t* seq_ids, int n, int32_t* pairs,
                           int32_t cap, int32_t* num_pairs) {
    return swap_group(bm, seq_ids, n, pairs, cap, num_pairs, true, "pkv_bm_swap_out");
}

pkv_status pkv_bm_swap_in(pkv_bm* bm, const int64_t* seq_ids, int n, int32_t* pairs, int32_t cap,
                          int32_t* num_pairs) {
    return swap_group(bm, seq_ids, n, pairs, cap, num_pairs, false, "pkv_bm_swap_in");
}

int32_t pkv_bm_is_swapped(const pkv_bm* bm, int64_t seq_id) {
    if (!bm) return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : (it->second.swapped ? 1 : 0);
}

int32_t pkv_bm_cpu_refcount(const pkv_bm* bm, int32_t block) {
    if (!bm || block < 0 || block >= bm->num_cpu_blocks) return -1;
    return bm->cpu_ref[(size_t)block];
}

int64_t pkv_bm_num_free_cpu(const pkv_bm* bm) { return bm ? (int64_t)bm->cpu_free.size() : -1; }

int32_t pkv_bm_refcount(const pkv_bm* bm, int32_t block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    return bm->ref[(size_t)block];
}

int64_t pkv_bm_num_free(const pkv_bm* bm) { return bm ? (int64_t)bm->free_list.size() : -1; }

}  // extern "C"
