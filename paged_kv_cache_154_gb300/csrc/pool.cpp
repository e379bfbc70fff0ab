// Host block pool: free list, per-sequence block tables, refcounts and
// copy-on-write. Restates the block manager of "KV Cache ... PagedAttention"
// (devpress.csdn.net) §七 -- free list popped from its end, ceil(n/16)
// blocks per sequence, a new block exactly when the token count reaches the
// capacity, release back to the list -- and adds the refcounts and
// copy-on-write that "LLM推理优化深度实战" (ybb.press) §2.1 describes for
// best-of-N sharing (copy a shared block only when it is modified).
#include <algorithm>
#include <new>
#include <vector>

#include "pa_internal.h"

struct pa_pool {
    int32_t num_blocks;
    int32_t block_size;
    std::vector<int32_t> free_list;            // taken from / returned to the back
    std::vector<int32_t> ref;                  // per physical block
    std::vector<std::vector<int32_t>> tables;  // per sequence id
    std::vector<int32_t> lens;                 // tokens per sequence id
    std::vector<uint8_t> live;                 // sequence id still alive
};

namespace {

pa_status check_seq(const pa_pool* p, int32_t seq) {
    if (seq < 0 || seq >= (int32_t)p->live.size() || !p->live[seq])
        return pa::fail(PA_ERR_INVALID_ARG, "unknown or freed sequence id %d", seq);
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_pool_create(int32_t num_blocks, int32_t block_size,
                                    const int32_t* free_order, pa_pool** out) {
    if (!out) return pa::fail(PA_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (num_blocks < 0) return pa::fail(PA_ERR_INVALID_ARG, "num_blocks < 0");
    if (block_size != 16)
        return pa::fail(PA_ERR_UNSUPPORTED, "block_size %d (only 16 is supported)", block_size);
    pa_pool* p = new (std::nothrow) pa_pool();
    if (!p) return pa::fail(PA_ERR_INVALID_ARG, "host allocation failed");
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->ref.assign(num_blocks, 0);
    p->free_list.resize(num_blocks);
    if (free_order) {
        std::vector<uint8_t> seen(num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete p;
                return pa::fail(PA_ERR_INVALID_ARG,
                                "free_order is not a permutation of 0..%d", num_blocks - 1);
            }
            seen[b] = 1;
            p->free_list[i] = b;
        }
    } else {
        for (int32_t i = 0; i < num_blocks; ++i) p->free_list[i] = i;
    }
    *out = p;
    return PA_OK;
}

extern "C" void pa_pool_destroy(pa_pool* pool) { delete pool; }

extern "C" pa_status pa_seq_create(pa_pool* p, int32_t* seq_id) {
    if (!p || !seq_id) return pa::fail(PA_ERR_INVALID_ARG, "NULL argument");
    *seq_id = (int32_t)p->tables.size();
    p->tables.emplace_back();
    p->lens.push_back(0);
    p->live.push_back(1);
    return PA_OK;
}

extern "C" pa_status pa_seq_fork(pa_pool* p, int32_t parent, int32_t* child) {
    if (!p || !child) return pa::fail(PA_ERR_INVALID_ARG, "NULL argument");
    if (pa_status s = check_seq(p, parent)) return s;
    int32_t c = (int32_t)p->tables.size();
    p->tables.push_back(p->tables[parent]);
    p->lens.push_back(p->lens[parent]);
    p->live.push_back(1);
    for (int32_t b : p->tables[c]) p->ref[b] += 1;
    *child = c;
    return PA_OK;
}

extern "C" pa_status pa_seq_append_slots(pa_pool* p, int32_t seq, int32_t n_tokens,
                                         int64_t* slots_out, int32_t* cow_pair_out,
                                         int32_t* n_cow) {
    if (!p || !n_cow) return pa::fail(PA_ERR_INVALID_ARG, "NULL argument");
    if (pa_status s = check_seq(p, seq)) return s;
    if (n_tokens < 0) return pa::fail(PA_ERR_INVALID_ARG, "n_tokens < 0");
    *n_cow = 0;
    if (n_tokens == 0) return PA_OK;
    if (!slots_out) return pa::fail(PA_ERR_INVALID_ARG, "slots_out is NULL");
    std::vector<int32_t>& table = p->tables[seq];
    const int64_t bs = p->block_size;
    const int64_t L = p->lens[seq];
    const bool cow = (L % bs != 0) && p->ref[table.back()] > 1;
    const int64_t new_blocks = (L + n_tokens + bs - 1) / bs - (int64_t)table.size();
    const int64_t need = new_blocks + (cow ? 1 : 0);
    if (need > (int64_t)p->free_list.size())
        return pa::fail(PA_ERR_OUT_OF_BLOCKS, "append of %d tokens needs %lld blocks, %zu free",
                        n_tokens, (long long)need, p->free_list.size());
    if (cow && !cow_pair_out)
        return pa::fail(PA_ERR_INVALID_ARG, "append needs a block copy but cow_pair_out is NULL");
    if (L + n_tokens > INT32_MAX) return pa::fail(PA_ERR_INVALID_ARG, "sequence too long");
    if (cow) {
        int32_t src = table.back();
        int32_t dst = p->free_list.back();
        p->free_list.pop_back();
        p->ref[src] -= 1;
        p->ref[dst] = 1;
        table.back() = dst;
        cow_pair_out[0] = src;
        cow_pair_out[1] = dst;
        *n_cow = 1;
    }
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t pos = L + i;
        if (pos >= (int64_t)table.size() * bs) {
            int32_t b = p->free_list.back();
            p->free_list.pop_back();
            p->ref[b] = 1;
            table.push_back(b);
        }
        slots_out[i] = (int64_t)table[pos / bs] * bs + pos % bs;
    }
    p->lens[seq] = (int32_t)(L + n_tokens);
    return PA_OK;
}

extern "C" pa_status pa_seq_free(pa_pool* p, int32_t seq) {
    if (!p) return pa::fail(PA_ERR_INVALID_ARG, "NULL pool");
    if (pa_status s = check_seq(p, seq)) return s;
    std::vector<int32_t>& table = p->tables[seq];
    for (int32_t b : table)
        if (p->ref[b] <= 0)
            return pa::fail(PA_ERR_BAD_REFCOUNT, "refcount underflow on block %d", b);
    for (int32_t b : table) {
        p->ref[b] -= 1;
        if (p->ref[b] == 0) p->free_list.push_back(b);
    }
    table.clear();
    table.shrink_to_fit();
    p->lens[seq] = 0;
    p->live[seq] = 0;
    return PA_OK;
}

extern "C" pa_status pa_seq_len(pa_pool* p, int32_t seq, int32_t* len) {
    if (!p || !len) return pa::fail(PA_ERR_INVALID_ARG, "NULL argument");
    if (pa_status s = check_seq(p, seq)) return s;
    *len = p->lens[seq];
    return PA_OK;
}

extern "C" pa_status pa_pool_block_tables(pa_pool* p, const int32_t* seqs, int32_t n,
                                          int32_t max_blocks, int32_t* tables_out,
                                          int32_t* lens_out) {
    if (!p || (n > 0 && (!seqs || !tables_out)) || n < 0 || max_blocks < 0)
        return pa::fail(PA_ERR_INVALID_ARG, "bad argument");
    for (int32_t i = 0; i < n; ++i) {
        if (pa_status s = check_seq(p, seqs[i])) return s;
        if ((int32_t)p->tables[seqs[i]].size() > max_blocks)
            return pa::fail(PA_ERR_INVALID_ARG, "sequence %d holds %zu blocks > max_blocks %d",
                            seqs[i], p->tables[seqs[i]].size(), max_blocks);
    }
    for (int32_t i = 0; i < n; ++i) {
        const std::vector<int32_t>& t = p->tables[seqs[i]];
        int32_t* row = tables_out + (int64_t)i * max_blocks;
        std::copy(t.begin(), t.end(), row);
        std::fill(row + t.size(), row + max_blocks, -1);
        if (lens_out) lens_out[i] = p->lens[seqs[i]];
    }
    return PA_OK;
}

extern "C" pa_status pa_pool_stats(pa_pool* p, int32_t* free_blocks, int32_t* used,
                                   int32_t* shared) {
    if (!p) return pa::fail(PA_ERR_INVALID_ARG, "NULL pool");
    int32_t u = 0, s = 0;
    for (int32_t r : p->ref) {
        u += r > 0;
        s += r > 1;
    }
    if (free_blocks) *free_blocks = (int32_t)p->free_list.size();
    if (used) *used = u;
    if (shared) *shared = s;
    return PA_OK;
}

extern "C" pa_status pa_pool_refcount(pa_pool* p, int32_t block, int32_t* ref) {
    if (!p || !ref) return pa::fail(PA_ERR_INVALID_ARG, "NULL argument");
    if (block < 0 || block >= p->num_blocks)
        return pa::fail(PA_ERR_INVALID_ARG, "block %d outside the pool", block);
    *ref = p->ref[block];
    return PA_OK;
}

// Groups of adjacent sequences (in the order given) that hold the same first
// physical block -- forks of one prompt -- and the number of tokens at the
// front that every member holds in the same physical blocks and that precede
// every query of the member: whole blocks only, at most (L - r + 1) / 16 of
// them for a member with L tokens and a query run of r. A group of one gets
// prefix 0 (reading it once is reading it once per sequence).
extern "C" pa_status pa_pool_prefix_groups(pa_pool* p, const int32_t* seqs, int32_t n,
                                           const int32_t* q_lens, int32_t* group_start_out,
                                           int32_t* prefix_len_out, int32_t* num_groups_out) {
    if (!p || n < 0 || (n > 0 && (!seqs || !group_start_out || !prefix_len_out)) ||
        !num_groups_out)
        return pa::fail(PA_ERR_INVALID_ARG, "bad argument");
    for (int32_t i = 0; i < n; ++i) {
        if (pa_status s = check_seq(p, seqs[i])) return s;
        const int32_t r = q_lens ? q_lens[i] : 1;
        if (r < 1 || r > p->lens[seqs[i]])
            return pa::fail(PA_ERR_INVALID_ARG, "sequence %d: query run %d, %d tokens", seqs[i], r,
                            p->lens[seqs[i]]);
    }
    const int32_t bs = p->block_size;
    int32_t ng = 0, i = 0;
    while (i < n) {
        const std::vector<int32_t>& t0 = p->tables[seqs[i]];
        int32_t j = i + 1;
        while (j < n && !t0.empty() && !p->tables[seqs[j]].empty() &&
               p->tables[seqs[j]][0] == t0[0])
            ++j;
        int32_t k = 0;
        if (j - i > 1) {
            k = (int32_t)t0.size();
            for (int32_t m = i; m < j; ++m) {
                const std::vector<int32_t>& t = p->tables[seqs[m]];
                const int32_t r = q_lens ? q_lens[m] : 1;
                int32_t c = 0;
                const int32_t lim = std::min<int32_t>((int32_t)t.size(), k);
                while (c < lim && t[c] == t0[c]) ++c;
                k = std::min(c, (p->lens[seqs[m]] - r + 1) / bs);
            }
        }
        group_start_out[ng] = i;
        prefix_len_out[ng] = k * bs;
        ++ng;
        i = j;
    }
    if (n > 0) group_start_out[ng] = n;
    *num_groups_out = ng;
    return PA_OK;
}
