// Host block pool: free list, per-sequence block tables, refcounts and
// copy-on-write. Restates the block manager of "KV Cache ... PagedAttention"
// (devpress.csdn.net) §七 -- free list popped from its end, ceil(n/16)
// blocks per sequence, a new block exactly when the token count reaches the
// capacity, release back to the list -- and adds the refcounts and
// copy-on-write that "LLM推理优化深度实战" (ybb.press) §2.1 describes for
// best-of-N sharing (copy a shared block only when it is modified).
//
// Prefix cache ("大模型推理优化全攻略" §2.4 and "KV Cache ... PagedAttention":
// requests that share a prefix reuse its KV blocks, found by a hash of the
// prefix tokens, with least-recently-used eviction). Restated at block
// granularity: a full block is identified by the whole token prefix that
// ends with it, kept as a trie of prefix nodes -- node = (parent node, the
// block's 16 token ids), looked up through a hash of that pair and then
// compared token by token, so a hash collision can never hand out the wrong
// KV. A block filled through pa_seq_append_tokens is registered under its
// node; pa_seq_create_with_prefix takes the longest chain of registered
// blocks for a new request. Registered blocks that no sequence holds any
// more wait in an LRU list (at most max_cached_blocks of them); allocation
// takes the free list first and then evicts the oldest cached block.
#include <algorithm>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_internal.h"

namespace {

constexpr int kPB = 16;   // tokens per block

struct PrefixNode {
    int64_t parent;       // node of the prefix one block shorter; -1 at the root
    int32_t tokens[kPB];
    int32_t block;        // registered physical block holding this prefix, or -1
    int32_t children;     // child nodes that exist
};

}  // namespace

struct pa_pool {
    int32_t num_blocks;
    int32_t block_size;
    std::vector<int32_t> free_list;            // taken from / returned to the back
    std::vector<int32_t> ref;                  // per physical block
    std::vector<std::vector<int32_t>> tables;  // per sequence id
    std::vector<int32_t> lens;                 // tokens per sequence id
    std::vector<uint8_t> live;                 // sequence id still alive
    // prefix cache (off unless enabled)
    bool pc_on = false;
    int32_t pc_max = 0;                                   // unreferenced blocks kept
    std::unordered_map<int64_t, PrefixNode> nodes;
    std::unordered_map<uint64_t, std::vector<int64_t>> edges;   // hash -> candidate nodes
    int64_t next_node = 0;
    std::vector<int64_t> block_node;                      // per block: its node, or -1
    std::list<int32_t> lru;                               // oldest first
    std::vector<std::list<int32_t>::iterator> lru_pos;
    std::vector<uint8_t> in_lru;
    std::vector<std::vector<int64_t>> seq_nodes;          // per sequence: node of each full block
    std::vector<std::vector<int32_t>> seq_tail;           // tokens of the partial last block
    std::vector<uint8_t> seq_known;                       // all tokens known (append_tokens only)
    int64_t hits = 0, lookups = 0;
};

namespace {

pa_status check_seq(const pa_pool* p, int32_t seq) {
    if (seq < 0 || seq >= (int32_t)p->live.size() || !p->live[seq])
        return pa::fail(PA_ERR_INVALID_ARG, "unknown or freed sequence id %d", seq);
    return PA_OK;
}

uint64_t mix64(uint64_t z) {   // a 64-bit finaliser (xor-shift-multiply rounds)
    z ^= z >> 33;
    z *= 0xff51afd7ed558ccdull;
    z ^= z >> 33;
    z *= 0xc4ceb9fe1a85ec53ull;
    z ^= z >> 33;
    return z;
}

uint64_t edge_hash(int64_t parent, const int32_t* t) {
    uint64_t h = mix64((uint64_t)parent + 0x9e3779b97f4a7c15ull);
    for (int i = 0; i < kPB; ++i) h = mix64(h ^ ((uint64_t)(uint32_t)t[i] + (uint64_t)i * 0x100000001ull));
    return h;
}

int64_t find_edge(const pa_pool* p, int64_t parent, const int32_t* t) {
    auto it = p->edges.find(edge_hash(parent, t));
    if (it == p->edges.end()) return -1;
    for (int64_t id : it->second) {
        const PrefixNode& n = p->nodes.at(id);
        if (n.parent == parent && std::equal(t, t + kPB, n.tokens)) return id;
    }
    return -1;
}

int64_t make_node(pa_pool* p, int64_t parent, const int32_t* t) {
    const int64_t id = p->next_node++;
    PrefixNode n;
    n.parent = parent;
    std::copy(t, t + kPB, n.tokens);
    n.block = -1;
    n.children = 0;
    p->nodes.emplace(id, n);
    p->edges[edge_hash(parent, t)].push_back(id);
    if (parent >= 0) p->nodes.at(parent).children += 1;
    return id;
}

// A node that holds no block and has no children is dropped, and so is its
// parent if that leaves it the same.
void drop_dead_nodes(pa_pool* p, int64_t id) {
    while (id >= 0) {
        auto it = p->nodes.find(id);
        if (it == p->nodes.end() || it->second.block >= 0 || it->second.children > 0) return;
        const int64_t parent = it->second.parent;
        std::vector<int64_t>& bucket = p->edges[edge_hash(parent, it->second.tokens)];
        bucket.erase(std::find(bucket.begin(), bucket.end(), id));
        if (bucket.empty()) p->edges.erase(edge_hash(parent, it->second.tokens));
        p->nodes.erase(it);
        if (parent >= 0) p->nodes.at(parent).children -= 1;
        id = parent;
    }
}

void unregister_block(pa_pool* p, int32_t b) {
    const int64_t id = p->block_node[b];
    if (id < 0) return;
    p->block_node[b] = -1;
    p->nodes.at(id).block = -1;
    drop_dead_nodes(p, id);
}

int64_t available(const pa_pool* p) { return (int64_t)p->free_list.size() + (int64_t)p->lru.size(); }

// A block for a new use: the free list first, else the least recently
// released cached block (evicted from the prefix cache).
int32_t take_block(pa_pool* p) {
    if (!p->free_list.empty()) {
        const int32_t b = p->free_list.back();
        p->free_list.pop_back();
        return b;
    }
    const int32_t b = p->lru.front();
    p->lru.pop_front();
    p->in_lru[b] = 0;
    unregister_block(p, b);
    return b;
}

// The last holder let go of block b: a registered block waits in the LRU
// list (evicting the oldest past max_cached_blocks), any other block is free.
void release_block(pa_pool* p, int32_t b) {
    if (p->block_node.empty() || p->block_node[b] < 0) {
        p->free_list.push_back(b);
        return;
    }
    p->lru_pos[b] = p->lru.insert(p->lru.end(), b);
    p->in_lru[b] = 1;
    if ((int64_t)p->lru.size() > p->pc_max) {
        const int32_t old = p->lru.front();
        p->lru.pop_front();
        p->in_lru[old] = 0;
        unregister_block(p, old);
        p->free_list.push_back(old);
    }
}

// A cached block taken back into use by a prefix hit.
void revive_block(pa_pool* p, int32_t b) {
    if (p->in_lru[b]) {
        p->lru.erase(p->lru_pos[b]);
        p->in_lru[b] = 0;
    }
}

void new_seq_info(pa_pool* p) {
    p->seq_nodes.emplace_back();
    p->seq_tail.emplace_back();
    p->seq_known.push_back(1);
}

// Token bookkeeping after an append of n tokens starting at position L: the
// tail fills up, and every block that becomes full is registered under the
// node of its prefix (unless that prefix already has a block).
void record_tokens(pa_pool* p, int32_t seq, const int32_t* tokens, int64_t L, int64_t n) {
    if (!p->seq_known[seq]) return;
    std::vector<int32_t>& tail = p->seq_tail[seq];
    std::vector<int64_t>& chain = p->seq_nodes[seq];
    for (int64_t i = 0; i < n; ++i) {
        tail.push_back(tokens[i]);
        if ((int)tail.size() < kPB) continue;
        const int64_t b = (L + i) / kPB;                 // the block just filled
        const int64_t parent = b == 0 ? -1 : chain[b - 1];
        if (parent >= 0 && !p->nodes.count(parent)) {   // its prefix node is gone
            p->seq_known[seq] = 0;
            return;
        }
        int64_t id = find_edge(p, parent, tail.data());
        if (id < 0) id = make_node(p, parent, tail.data());
        chain.push_back(id);
        PrefixNode& node = p->nodes.at(id);
        const int32_t blk = p->tables[seq][b];
        if (node.block < 0 && p->block_node[blk] < 0) {
            node.block = blk;
            p->block_node[blk] = id;
        }
        tail.clear();
    }
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
    new_seq_info(p);
    return PA_OK;
}

extern "C" pa_status pa_seq_fork(pa_pool* p, int32_t parent, int32_t* child) {
    if (!p || !child) return pa::fail(PA_ERR_INVALID_ARG, "NULL argument");
    if (pa_status s = check_seq(p, parent)) return s;
    int32_t c = (int32_t)p->tables.size();
    p->tables.push_back(p->tables[parent]);
    p->lens.push_back(p->lens[parent]);
    p->live.push_back(1);
    p->seq_nodes.push_back(p->seq_nodes[parent]);
    p->seq_tail.push_back(p->seq_tail[parent]);
    p->seq_known.push_back(p->seq_known[parent]);
    for (int32_t b : p->tables[c]) p->ref[b] += 1;
    *child = c;
    return PA_OK;
}

namespace {

// Reserve n token slots of a sequence (copy-on-write of a shared partial tail
// first); all or nothing.
pa_status append(pa_pool* p, int32_t seq, int32_t n_tokens, int64_t* slots_out,
                 int32_t* cow_pair_out, int32_t* n_cow) {
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
    if (need > available(p))
        return pa::fail(PA_ERR_OUT_OF_BLOCKS, "append of %d tokens needs %lld blocks, %lld free",
                        n_tokens, (long long)need, (long long)available(p));
    if (cow && !cow_pair_out)
        return pa::fail(PA_ERR_INVALID_ARG, "append needs a block copy but cow_pair_out is NULL");
    if (L + n_tokens > INT32_MAX) return pa::fail(PA_ERR_INVALID_ARG, "sequence too long");
    if (cow) {
        int32_t src = table.back();
        int32_t dst = take_block(p);
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
            int32_t b = take_block(p);
            p->ref[b] = 1;
            table.push_back(b);
        }
        slots_out[i] = (int64_t)table[pos / bs] * bs + pos % bs;
    }
    p->lens[seq] = (int32_t)(L + n_tokens);
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_seq_append_slots(pa_pool* p, int32_t seq, int32_t n_tokens,
                                         int64_t* slots_out, int32_t* cow_pair_out,
                                         int32_t* n_cow) {
    if (pa_status s = append(p, seq, n_tokens, slots_out, cow_pair_out, n_cow)) return s;
    if (n_tokens > 0) p->seq_known[seq] = 0;   // tokens unknown: nothing more to register
    return PA_OK;
}

extern "C" pa_status pa_seq_append_slots_batch(pa_pool* p, const int32_t* seqs,
                                               const int32_t* n_tokens, int32_t n,
                                               int64_t* slots_out, int32_t* cow_pairs_out,
                                               int32_t* n_cow) {
    if (!p) return pa::fail(PA_ERR_INVALID_ARG, "NULL pool");
    if (n < 0 || (n > 0 && (!seqs || !n_tokens)))
        return pa::fail(PA_ERR_INVALID_ARG, "batch of %d sequences without arrays", n);
    if (!n_cow) return pa::fail(PA_ERR_INVALID_ARG, "n_cow is NULL");
    *n_cow = 0;
    int64_t off = 0;
    for (int32_t i = 0; i < n; ++i) {
        // without cow_pairs_out the single call refuses a copy before it changes anything
        int32_t pair[2], one = 0;
        if (pa_status s = pa_seq_append_slots(p, seqs[i], n_tokens[i], slots_out + off,
                                              cow_pairs_out ? pair : nullptr, &one))
            return s;   // the sequences before i keep their reservations
        off += n_tokens[i] > 0 ? n_tokens[i] : 0;
        if (one) {
            cow_pairs_out[2 * *n_cow] = pair[0];
            cow_pairs_out[2 * *n_cow + 1] = pair[1];
            ++*n_cow;
        }
    }
    return PA_OK;
}

extern "C" pa_status pa_seq_append_tokens(pa_pool* p, int32_t seq, const int32_t* token_ids,
                                          int32_t n_tokens, int64_t* slots_out,
                                          int32_t* cow_pair_out, int32_t* n_cow) {
    if (p && !p->pc_on) return pa::fail(PA_ERR_INVALID_ARG, "the prefix cache is not enabled");
    if (n_tokens > 0 && !token_ids) return pa::fail(PA_ERR_INVALID_ARG, "token_ids is NULL");
    const int64_t L = (p && seq >= 0 && seq < (int32_t)p->lens.size()) ? p->lens[seq] : 0;
    if (pa_status s = append(p, seq, n_tokens, slots_out, cow_pair_out, n_cow)) return s;
    record_tokens(p, seq, token_ids, L, n_tokens);
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
        if (p->ref[b] == 0) release_block(p, b);
    }
    table.clear();
    table.shrink_to_fit();
    p->lens[seq] = 0;
    p->live[seq] = 0;
    p->seq_nodes[seq].clear();
    p->seq_nodes[seq].shrink_to_fit();
    p->seq_tail[seq].clear();
    p->seq_known[seq] = 0;
    return PA_OK;
}

extern "C" pa_status pa_pool_enable_prefix_cache(pa_pool* p, int32_t max_cached_blocks) {
    if (!p) return pa::fail(PA_ERR_INVALID_ARG, "NULL pool");
    if (max_cached_blocks < 0) return pa::fail(PA_ERR_INVALID_ARG, "max_cached_blocks < 0");
    if (!p->pc_on) {
        p->block_node.assign(p->num_blocks, -1);
        p->lru_pos.resize(p->num_blocks);
        p->in_lru.assign(p->num_blocks, 0);
        p->pc_on = true;
    }
    p->pc_max = max_cached_blocks;
    while ((int64_t)p->lru.size() > p->pc_max) {   // a smaller limit evicts at once
        const int32_t old = p->lru.front();
        p->lru.pop_front();
        p->in_lru[old] = 0;
        unregister_block(p, old);
        p->free_list.push_back(old);
    }
    return PA_OK;
}

extern "C" pa_status pa_seq_create_with_prefix(pa_pool* p, const int32_t* token_ids,
                                               int32_t n_tokens, int32_t* seq_out,
                                               int32_t* n_cached_out) {
    if (!p || !seq_out || !n_cached_out || (n_tokens > 0 && !token_ids))
        return pa::fail(PA_ERR_INVALID_ARG, "NULL argument");
    if (!p->pc_on) return pa::fail(PA_ERR_INVALID_ARG, "the prefix cache is not enabled");
    if (n_tokens < 0) return pa::fail(PA_ERR_INVALID_ARG, "n_tokens < 0");
    int32_t seq;
    pa_seq_create(p, &seq);
    std::vector<int32_t>& table = p->tables[seq];
    std::vector<int64_t>& chain = p->seq_nodes[seq];
    int64_t parent = -1;
    // whole blocks only, and at least one token left to compute
    for (int64_t b = 0; (b + 1) * kPB <= (int64_t)n_tokens - 1; ++b) {
        p->lookups += 1;
        const int64_t id = find_edge(p, parent, token_ids + b * kPB);
        if (id < 0 || p->nodes.at(id).block < 0) break;
        const int32_t blk = p->nodes.at(id).block;
        if (p->ref[blk] == 0) revive_block(p, blk);
        p->ref[blk] += 1;
        table.push_back(blk);
        chain.push_back(id);
        p->hits += 1;
        parent = id;
    }
    p->lens[seq] = (int32_t)(table.size() * kPB);
    *seq_out = seq;
    *n_cached_out = p->lens[seq];
    return PA_OK;
}

extern "C" pa_status pa_pool_prefix_stats(pa_pool* p, int32_t* cached_free, int32_t* registered,
                                          int64_t* hit_blocks, int64_t* lookup_blocks) {
    if (!p) return pa::fail(PA_ERR_INVALID_ARG, "NULL pool");
    int32_t reg = 0;
    for (int64_t id : p->block_node) reg += id >= 0;
    if (cached_free) *cached_free = (int32_t)p->lru.size();
    if (registered) *registered = reg;
    if (hit_blocks) *hit_blocks = p->hits;
    if (lookup_blocks) *lookup_blocks = p->lookups;
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
