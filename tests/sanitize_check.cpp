// Host block pool and CPU oracle under AddressSanitizer and
// UndefinedBehaviorSanitizer (built and run by tests/test_sanitize.py).
//
// The pool source is compiled into this program as it is into the library;
// the oracle (plain C) is linked in. Seeded random traces drive every pool
// call -- sequences created, forked, appended to (by slots and by token ids,
// with the prefix cache off and on, at several LRU sizes), freed; block
// tables, statistics, refcounts, fork groups; argument errors -- and after
// each operation the pool's own counts are checked against each other:
//   * every block is free, held (refcount > 0) or cached, exactly once;
//   * the refcounts add up to the block-table entries of the live sequences;
//   * a sequence holds ceil(len / 16) blocks.
// Then the oracle's attention, quantiser, appends and block copies run on
// small random paged caches of every element type. Any sanitizer finding
// aborts the program; "ok" on stdout means every check passed.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "pool.cpp"   // the library's host pool, built here with the sanitizers

namespace pa {
// the library reports argument errors through this (capi.cu in the library)
pa_status fail(pa_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    return s;
}
}  // namespace pa

extern "C" {
int orc_attend(double* out_o, double* out_m, double* out_l, const double* q,
               const void* k_cache, const void* v_cache, int kv_dtype, const float* k_scale,
               const float* v_scale, const int8_t* k_zp, const int8_t* v_zp,
               const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
               const int32_t* query_start_loc, int num_seqs, int num_heads, int num_kv_heads,
               int head_dim, int block_size, double scale, int64_t t_begin, int64_t t_end,
               int threads);
void orc_quantize_row(const float* x, int d, int8_t* codes, float* scale_out, int8_t* zp_out);
void orc_append(uint16_t* cache, const uint16_t* src, const int64_t* slots, int64_t num_tokens,
                int num_kv_heads, int head_dim, int block_size);
void orc_append_int8(int8_t* codes, float* scales, int8_t* zps, const uint16_t* src, int src_bf16,
                     const int64_t* slots, int64_t num_tokens, int num_kv_heads, int head_dim,
                     int block_size);
void orc_append_fp8(uint8_t* codes, const float* head_scale, const uint16_t* src, int src_bf16,
                    const int64_t* slots, int64_t num_tokens, int num_kv_heads, int head_dim,
                    int block_size);
void orc_copy_blocks(uint8_t* base, int64_t bytes_per_block, const int32_t* pairs, int n_pairs);
}

namespace {

uint64_t g_rng = 0x9e3779b97f4a7c15ull;
uint32_t rnd() {
    g_rng ^= g_rng << 13;
    g_rng ^= g_rng >> 7;
    g_rng ^= g_rng << 17;
    return (uint32_t)(g_rng >> 11);
}
int rnd(int n) { return n > 0 ? (int)(rnd() % (uint32_t)n) : 0; }

int g_failures = 0;
long g_oob = 0, g_cow = 0, g_hit_tokens = 0, g_ops = 0;   // paths the traces reached
#define CHECK(c)                                                               \
    do {                                                                       \
        if (!(c)) {                                                            \
            std::printf("check failed at line %d: %s\n", __LINE__, #c);        \
            if (++g_failures > 20) std::exit(1);                               \
        }                                                                      \
    } while (0)

// The pool's counts, checked against each other.
void check_pool(pa_pool* p, int nb, const std::vector<int>& live) {
    int32_t fr = -1, used = -1, shared = -1, cached = 0, reg = 0;
    int64_t hits = 0, looks = 0;
    CHECK(pa_pool_stats(p, &fr, &used, &shared) == PA_OK);
    CHECK(pa_pool_prefix_stats(p, &cached, &reg, &hits, &looks) == PA_OK);
    CHECK(fr + used + cached == nb);
    CHECK(shared <= used && hits <= looks && cached <= reg);
    int64_t refs = 0;
    int held = 0;
    for (int b = 0; b < nb; ++b) {
        int32_t r = -1;
        CHECK(pa_pool_refcount(p, b, &r) == PA_OK);
        CHECK(r >= 0);
        refs += r;
        held += r > 0;
    }
    CHECK(held == used);
    int64_t entries = 0;
    if (!live.empty()) {
        int maxb = 1;
        for (int s : live) {
            int32_t L = -1;
            CHECK(pa_seq_len(p, s, &L) == PA_OK);
            maxb = std::max(maxb, (L + 15) / 16);
        }
        std::vector<int32_t> tables((size_t)live.size() * maxb), lens(live.size());
        CHECK(pa_pool_block_tables(p, live.data(), (int)live.size(), maxb, tables.data(),
                                   lens.data()) == PA_OK);
        for (size_t i = 0; i < live.size(); ++i) {
            const int nbs = (lens[i] + 15) / 16;
            for (int j = 0; j < maxb; ++j) {
                const int32_t e = tables[i * maxb + j];
                if (j < nbs) CHECK(e >= 0 && e < nb);
                else CHECK(e == -1);
            }
            entries += nbs;
        }
    }
    CHECK(refs == entries);
}

// A seeded trace of pool operations; with max_cached >= 0 the prefix cache is on.
void pool_trace(int nb, int ops, int max_cached) {
    pa_pool* p = nullptr;
    std::vector<int32_t> order(nb);
    for (int i = 0; i < nb; ++i) order[i] = i;
    for (int i = nb - 1; i > 0; --i) std::swap(order[i], order[rnd(i + 1)]);
    CHECK(pa_pool_create(nb, 16, order.data(), &p) == PA_OK);
    if (max_cached >= 0) CHECK(pa_pool_enable_prefix_cache(p, max_cached) == PA_OK);
    // a few shared prompts, so that prefixes repeat
    std::vector<std::vector<int32_t>> prompts(4);
    for (auto& pr : prompts) {
        pr.resize(16 + rnd(120));
        for (auto& t : pr) t = rnd(50);
    }
    std::vector<int> live;
    std::vector<char> by_tokens;   // the sequence was only ever appended by token ids
    std::vector<int64_t> slots(256);
    for (int op = 0; op < ops; ++op) {
        const int k = rnd(100);
        int32_t pair[2], ncow = 0, sid = -1;
        if (k < 12 || live.empty()) {
            if (max_cached >= 0 && rnd(2)) {
                std::vector<int32_t> toks = prompts[rnd(4)];
                const int extra = rnd(40);
                for (int i = 0; i < extra; ++i) toks.push_back(rnd(50));
                int32_t got = -1;
                const pa_status st =
                    pa_seq_create_with_prefix(p, toks.data(), (int)toks.size(), &sid, &got);
                CHECK(st == PA_OK);
                if (st == PA_OK) {
                    CHECK(got % 16 == 0 && got < (int)toks.size());
                    g_hit_tokens += got;
                    live.push_back(sid);
                    by_tokens.push_back(1);
                    const pa_status a = pa_seq_append_tokens(p, sid, toks.data() + got,
                                                             (int)toks.size() - got, slots.data(),
                                                             pair, &ncow);
                    CHECK(a == PA_OK || a == PA_ERR_OUT_OF_BLOCKS);
                }
            } else {
                CHECK(pa_seq_create(p, &sid) == PA_OK);
                live.push_back(sid);
                by_tokens.push_back(0);
            }
        } else if (k < 24) {
            const int i = rnd((int)live.size());
            if (pa_seq_fork(p, live[i], &sid) == PA_OK) {
                live.push_back(sid);
                by_tokens.push_back(by_tokens[i]);
            }
        } else if (k < 60) {
            const int i = rnd((int)live.size());
            const int n = rnd(48);
            pa_status st;
            if (max_cached >= 0 && by_tokens[i] && rnd(2)) {
                std::vector<int32_t> toks(n);
                for (auto& t : toks) t = rnd(50);
                st = pa_seq_append_tokens(p, live[i], toks.data(), n, slots.data(), pair, &ncow);
            } else {
                st = pa_seq_append_slots(p, live[i], n, slots.data(), pair, &ncow);
                by_tokens[i] = 0;
            }
            CHECK(st == PA_OK || st == PA_ERR_OUT_OF_BLOCKS || st == PA_ERR_INVALID_ARG);
            g_oob += st == PA_ERR_OUT_OF_BLOCKS;
            g_cow += st == PA_OK && ncow;
            if (st == PA_OK) {
                for (int t = 0; t < n; ++t) CHECK(slots[t] >= 0 && slots[t] < (int64_t)nb * 16);
                if (ncow) CHECK(pair[0] != pair[1] && pair[0] >= 0 && pair[1] < nb);
            }
        } else if (k < 66) {
            // a decode step's reservations in one call over a run of live sequences
            const int n = 1 + rnd((int)live.size());
            std::vector<int32_t> cnt(n), prs(2 * n);
            int64_t total = 0;
            for (auto& c : cnt) total += (c = rnd(5));
            std::vector<int64_t> sl(total + 1);
            int32_t nc = -1;
            const pa_status st = pa_seq_append_slots_batch(p, live.data(), cnt.data(), n,
                                                           sl.data(), prs.data(), &nc);
            CHECK(st == PA_OK || st == PA_ERR_OUT_OF_BLOCKS);
            CHECK(nc >= 0 && nc <= n);
            g_oob += st == PA_ERR_OUT_OF_BLOCKS;
            g_cow += nc;
            if (st == PA_OK)
                for (int64_t t = 0; t < total; ++t) CHECK(sl[t] >= 0 && sl[t] < (int64_t)nb * 16);
            for (int c = 0; c < nc; ++c)
                CHECK(prs[2 * c] != prs[2 * c + 1] && prs[2 * c] >= 0 && prs[2 * c + 1] < nb);
            for (int i = 0; i < n; ++i) by_tokens[i] = 0;
        } else if (k < 80) {
            const int i = rnd((int)live.size());
            CHECK(pa_seq_free(p, live[i]) == PA_OK);
            CHECK(pa_seq_free(p, live[i]) == PA_ERR_INVALID_ARG);   // a second free is refused
            live.erase(live.begin() + i);
            by_tokens.erase(by_tokens.begin() + i);
        } else if (k < 88) {
            // fork groups of a random run of live sequences (query runs of 1..3)
            const int n = 1 + rnd((int)live.size());
            std::vector<int32_t> seqs(live.begin(), live.begin() + n), ql(n), gs(n + 1), pl(n);
            bool ok_runs = true;
            for (int i = 0; i < n; ++i) {
                int32_t L = 0;
                pa_seq_len(p, seqs[i], &L);
                ql[i] = L >= 1 ? 1 + rnd(std::min(3, (int)L)) : 1;
                ok_runs &= L >= 1;
            }
            int32_t ng = -1;
            const pa_status st =
                pa_pool_prefix_groups(p, seqs.data(), n, ql.data(), gs.data(), pl.data(), &ng);
            if (ok_runs) {
                CHECK(st == PA_OK);
                if (st == PA_OK) {
                    CHECK(ng >= 1 && ng <= n && gs[0] == 0 && gs[ng] == n);
                    for (int g = 0; g < ng; ++g) CHECK(gs[g + 1] > gs[g] && pl[g] % 16 == 0);
                }
            }
        } else if (k < 94) {
            // argument errors: unknown ids, negative sizes, NULL outputs
            CHECK(pa_seq_free(p, 1 << 30) == PA_ERR_INVALID_ARG);
            CHECK(pa_seq_fork(p, -1, &sid) == PA_ERR_INVALID_ARG);
            CHECK(pa_seq_append_slots(p, live[0], -1, slots.data(), pair, &ncow) ==
                  PA_ERR_INVALID_ARG);
            CHECK(pa_seq_append_slots(p, live[0], 3, nullptr, pair, &ncow) == PA_ERR_INVALID_ARG);
            const int32_t bad_n[1] = {-2};
            CHECK(pa_seq_append_slots_batch(p, live.data(), bad_n, 1, slots.data(), nullptr,
                                            &ncow) == PA_ERR_INVALID_ARG && ncow == 0);
            CHECK(pa_seq_append_slots_batch(p, live.data(), nullptr, 1, slots.data(), nullptr,
                                            &ncow) == PA_ERR_INVALID_ARG);
            CHECK(pa_seq_append_slots_batch(p, nullptr, nullptr, 0, nullptr, nullptr, &ncow) ==
                  PA_OK && ncow == 0);
            int32_t r;
            CHECK(pa_pool_refcount(p, nb, &r) == PA_ERR_INVALID_ARG);
            int32_t t1[1];
            int32_t L = 0;
            pa_seq_len(p, live[0], &L);
            if (L > 16) CHECK(pa_pool_block_tables(p, live.data(), 1, 1, t1, nullptr) ==
                              PA_ERR_INVALID_ARG);
        } else if (max_cached >= 0) {
            CHECK(pa_pool_enable_prefix_cache(p, rnd(nb)) == PA_OK);   // resize the LRU
        }
        check_pool(p, nb, live);
        ++g_ops;
        if (g_failures) break;
    }
    for (int s : live) CHECK(pa_seq_free(p, s) == PA_OK);
    check_pool(p, nb, {});
    pa_pool_destroy(p);
}

uint16_t f32_to_bf16(float x) {
    uint32_t u;
    std::memcpy(&u, &x, 4);
    return (uint16_t)((u + 0x7fff + ((u >> 16) & 1)) >> 16);
}

// The oracle's functions on small random paged caches.
void oracle_calls() {
    const int S = 3, Hq = 8, Hkv = 2, d = 64, bs = 16, maxb = 8, nb = 32;
    const int lens[S] = {1, 47, 128};
    const int qsl[S + 1] = {0, 1, 4, 6};   // query runs of 1, 3 and 2 tokens
    std::vector<int32_t> tables(S * maxb, -1);
    std::vector<int32_t> perm(nb);
    for (int i = 0; i < nb; ++i) perm[i] = i;
    for (int i = nb - 1; i > 0; --i) std::swap(perm[i], perm[rnd(i + 1)]);
    int used = 0;
    for (int s = 0; s < S; ++s)
        for (int b = 0; b < (lens[s] + bs - 1) / bs; ++b) tables[s * maxb + b] = perm[used++];
    const size_t elems = (size_t)nb * Hkv * bs * d;
    std::vector<uint16_t> k16(elems), v16(elems);
    for (size_t i = 0; i < elems; ++i) {
        k16[i] = f32_to_bf16((float)(rnd(2001) - 1000) / 500.f);
        v16[i] = f32_to_bf16((float)(rnd(2001) - 1000) / 500.f);
    }
    const int nq = qsl[S];
    std::vector<double> q((size_t)nq * Hq * d), o((size_t)nq * Hq * d), m(nq * Hq), l(nq * Hq);
    for (auto& x : q) x = (double)(rnd(2001) - 1000) / 700.0;
    CHECK(orc_attend(o.data(), m.data(), l.data(), q.data(), k16.data(), v16.data(), 1, nullptr,
                     nullptr, nullptr, nullptr, tables.data(), maxb, lens, qsl, S, Hq, Hkv, d, bs,
                     0.125, 0, 1 << 20, 1) == 0);
    for (double x : o) CHECK(std::isfinite(x));
    // split range [16, 64): rows with no visible key there have l = 0
    CHECK(orc_attend(o.data(), m.data(), l.data(), q.data(), k16.data(), v16.data(), 1, nullptr,
                     nullptr, nullptr, nullptr, tables.data(), maxb, lens, qsl, S, Hq, Hkv, d, bs,
                     0.125, 16, 64, 1) == 0);
    // an invalid query run is reported, not read past
    const int bad_qsl[S + 1] = {0, 2, 3, 4};   // 2 query tokens for a 1-token sequence
    CHECK(orc_attend(o.data(), m.data(), l.data(), q.data(), k16.data(), v16.data(), 1, nullptr,
                     nullptr, nullptr, nullptr, tables.data(), maxb, lens, bad_qsl, S, Hq, Hkv, d,
                     bs, 0.125, 0, 1 << 20, 1) != 0);
    // appends, quantisers, block copies
    const int T = 5;
    std::vector<int64_t> slots = {(int64_t)perm[0] * bs + 3, -1, (int64_t)perm[5] * bs + 15,
                                  (int64_t)perm[2] * bs, (int64_t)perm[9] * bs + 7};
    std::vector<uint16_t> src((size_t)T * Hkv * d);
    for (auto& x : src) x = f32_to_bf16((float)(rnd(2001) - 1000) / 300.f);
    orc_append(k16.data(), src.data(), slots.data(), T, Hkv, d, bs);
    std::vector<int8_t> codes(elems), zps((size_t)nb * Hkv * bs);
    std::vector<float> scales((size_t)nb * Hkv * bs);
    orc_append_int8(codes.data(), scales.data(), zps.data(), src.data(), 1, slots.data(), T, Hkv,
                    d, bs);
    std::vector<uint8_t> fp8(elems);
    const float hs[Hkv] = {0.01f, 0.02f};
    orc_append_fp8(fp8.data(), hs, src.data(), 1, slots.data(), T, Hkv, d, bs);
    std::vector<float> row(d);
    int8_t zp;
    float sc;
    for (int rep = 0; rep < 200; ++rep) {
        for (auto& x : row) x = (float)(rnd(20001) - 10000) / (float)(1 + rnd(5000));
        orc_quantize_row(row.data(), d, codes.data(), &sc, &zp);
        CHECK(sc > 0.f && std::isfinite(sc));
    }
    const int32_t pairs[4] = {perm[0], perm[20], perm[1], perm[21]};
    orc_copy_blocks(reinterpret_cast<uint8_t*>(k16.data()), (int64_t)Hkv * bs * d * 2, pairs, 2);
    CHECK(std::memcmp(&k16[(size_t)perm[0] * Hkv * bs * d], &k16[(size_t)perm[20] * Hkv * bs * d],
                      (size_t)Hkv * bs * d * 2) == 0);
    // the quantised caches through the attention
    CHECK(orc_attend(o.data(), m.data(), l.data(), q.data(), codes.data(), codes.data(), 3,
                     scales.data(), scales.data(), zps.data(), zps.data(), tables.data(), maxb, lens,
                     qsl, S, Hq, Hkv, d, bs, 0.125, 0, 1 << 20, 1) == 0);
    CHECK(orc_attend(o.data(), m.data(), l.data(), q.data(), fp8.data(), fp8.data(), 4, hs, hs,
                     nullptr, nullptr, tables.data(), maxb, lens, qsl, S, Hq, Hkv, d, bs, 0.125, 0,
                     1 << 20, 1) == 0);
}

}  // namespace

int main(int argc, char** argv) {
    const int ops = argc > 1 ? std::atoi(argv[1]) : 1500;
    pool_trace(64, ops, -1);     // prefix cache off, a small pool (appends run out of blocks)
    pool_trace(512, ops, -1);
    pool_trace(256, ops, 0);     // prefix cache on, nothing kept
    pool_trace(256, ops, 16);    // a small LRU
    pool_trace(512, ops, 512);   // an LRU as large as the pool
    oracle_calls();
    if (g_failures) return 1;
    std::printf("ok: %ld pool operations, %ld appends out of blocks, %ld copy-on-write appends, "
                "%ld prompt tokens found in the prefix cache\n", g_ops, g_oob, g_cow, g_hit_tokens);
    return 0;
}
