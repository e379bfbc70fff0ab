// Host check of the in-kernel split-KV merge's bookkeeping, on the real
// schedule arithmetic of csrc/balanced.cuh (share_count, share_start,
// share_of, blocks_in, cut_piece), over random call shapes.
//
// For every share, the pieces it writes are found the way the decode kernel
// finds them: a head piece when the share's first segment began before the
// share and ends inside it, a tail piece when the share does not hold its
// last segment whole. Each piece is counted in with cut_piece's counter and
// total. The check then asserts:
//   - every counter belongs to one segment;
//   - every counter's arrivals add up to exactly its total, so exactly one
//     piece completes it;
//   - every fold reads, for each share, the slot that share's piece was
//     written to, and each group partial overwrites its own group's slot;
//   - the second-level total equals the number of groups.
// Prints "ok" and exits 0, or prints the first failure and exits 1.
#include <cstdio>
#include <cstdlib>
#include <map>
#include <random>
#include <vector>

#include "balanced.cuh"

using pa::sched::CutPiece;
using pa::sched::Params;
using pa::sched::blocks_in;
using pa::sched::cut_piece;
using pa::sched::kCounterRegion;
using pa::sched::kMergeFanIn;
using pa::sched::share_count;
using pa::sched::share_of;
using pa::sched::share_start;

static unsigned int g_counters[3 * kCounterRegion];

#define CHECK(cond, ...)                                              \
    do {                                                              \
        if (!(cond)) {                                                \
            std::printf("FAIL %s:%d: ", __FILE__, __LINE__);          \
            std::printf(__VA_ARGS__);                                 \
            std::printf("\n");                                        \
            std::exit(1);                                             \
        }                                                             \
    } while (0)

struct Written {
    int64_t seg;    // segment of the piece
    int64_t slot;   // slot index it was written to
};

static void run_case(std::mt19937_64& rng, int64_t workers, const std::vector<int>& seg_len) {
    std::vector<int64_t> start(seg_len.size() + 1, 0);
    for (size_t i = 0; i < seg_len.size(); ++i) start[i + 1] = start[i] + seg_len[i];
    const int64_t B = start.back();
    Params p{};
    p.workers = (int)workers;
    p.arrivals = g_counters;
    const int64_t W = share_count(p, B);
    CHECK(W >= 1 && W <= B && W <= workers, "share count %lld for B %lld", (long long)W,
          (long long)B);
    auto seg_of = [&](int64_t f) {   // the segment holding virtual block f
        size_t lo = 0, hi = seg_len.size();
        while (hi - lo > 1) {
            const size_t mid = (lo + hi) / 2;
            if (start[mid] <= f) lo = mid;
            else hi = mid;
        }
        return (int64_t)lo;
    };
    std::map<int64_t, int64_t> counter_seg;   // counter index -> segment
    std::map<int64_t, int64_t> counter_sum;   // counter index -> blocks counted in
    std::map<int64_t, int64_t> counter_total;
    std::map<int64_t, Written> share_slot;    // (2 * share + k) -> piece written there
    std::map<int64_t, CutPiece> any_piece;    // segment -> one of its pieces
    std::map<int64_t, std::vector<int64_t>> seg_shares;
    auto count_in = [&](const CutPiece& x, int64_t seg) {
        const int64_t idx = x.cnt - g_counters;
        CHECK(idx >= 0 && idx < 3 * kCounterRegion, "counter index %lld", (long long)idx);
        auto it = counter_seg.find(idx);
        CHECK(it == counter_seg.end() || it->second == seg,
              "counter %lld shared by segments %lld and %lld", (long long)idx,
              (long long)it->second, (long long)seg);
        counter_seg[idx] = seg;
        counter_sum[idx] += x.pb;
        auto t = counter_total.find(idx);
        CHECK(t == counter_total.end() || t->second == x.total, "counter %lld totals differ",
              (long long)idx);
        counter_total[idx] = x.total;
        any_piece[seg] = x;
    };
    for (int64_t w = 0; w < W; ++w) {
        const int64_t f0 = share_start(w, B, W), f1 = share_start(w + 1, B, W);
        const int n = (int)(f1 - f0);
        CHECK(n >= 1, "empty share %lld", (long long)w);
        const int64_t s_first = seg_of(f0), s_last = seg_of(f1 - 1);
        // head: the first segment began before the share and ends inside it
        // (before the share's last block)
        const int64_t hb = f0 - start[s_first];
        const int hnbs = seg_len[s_first];
        if (hb > 0 && hnbs - hb < n) {
            const CutPiece x = cut_piece(p, B, w, start[s_first], (int)(hnbs - hb), hnbs,
                                         (int)s_first, 0, 0, 0, 1, -1, 0, w);
            count_in(x, s_first);
            share_slot[2 * w] = Written{s_first, 2 * w};
            seg_shares[s_first].push_back(w);
        }
        // tail: the last segment, unless the share holds it whole
        const int64_t seg_b0 = s_last == s_first ? f0 - start[s_last] : 0;
        const int64_t done = f1 - start[s_last];
        const bool whole = seg_b0 == 0 && done == seg_len[s_last];
        if (!whole) {
            const int64_t fs = start[s_last];
            const CutPiece x = cut_piece(p, B, w, fs, (int)(done - seg_b0), seg_len[s_last],
                                         (int)s_last, 0, 0, 0, 1, fs >= f0 ? w : -1, f0, -1);
            count_in(x, s_last);
            const int64_t slot = 2 * w + (s_last == s_first ? 0 : 1);
            share_slot[slot] = Written{s_last, slot};
            seg_shares[s_last].push_back(w);
        }
    }
    for (const auto& kv : counter_sum)
        CHECK(kv.second == counter_total[kv.first], "counter %lld: %lld blocks of %lld",
              (long long)kv.first, (long long)kv.second, (long long)counter_total[kv.first]);
    // every cut segment: the pieces the folds read are the ones written
    for (const auto& kv : any_piece) {
        const int64_t seg = kv.first;
        const CutPiece& x = kv.second;
        CHECK(x.fs == start[seg] && x.nbs == seg_len[seg], "segment %lld geometry",
              (long long)seg);
        CHECK(x.wa == share_of(x.fs, B, W) && x.wb == share_of(x.fs + x.nbs - 1, B, W),
              "segment %lld: shares %lld..%lld", (long long)seg, (long long)x.wa,
              (long long)x.wb);
        CHECK((int64_t)seg_shares[seg].size() == x.wb - x.wa + 1,
              "segment %lld: %zu pieces over shares %lld..%lld", (long long)seg,
              seg_shares[seg].size(), (long long)x.wa, (long long)x.wb);
        int64_t blocks = 0;
        for (int64_t sh = x.wa; sh <= x.wb; ++sh) {
            const int64_t b = blocks_in(B, W, x.fs, x.nbs, x.wb, sh, 1);
            CHECK(b >= 1, "segment %lld: share %lld holds none of it", (long long)seg,
                  (long long)sh);
            blocks += b;
            const int64_t slot = 2 * sh + (sh == x.wa ? x.first_slot : 0);
            auto it = share_slot.find(slot);
            CHECK(it != share_slot.end() && it->second.seg == seg,
                  "segment %lld: fold reads slot %lld of share %lld, not its piece",
                  (long long)seg, (long long)slot, (long long)sh);
        }
        CHECK(blocks == x.nbs, "segment %lld: pieces hold %lld of %d blocks", (long long)seg,
              (long long)blocks, x.nbs);
        if (x.wb - x.wa + 1 > kMergeFanIn) {
            CHECK(x.two_level, "segment %lld should merge in two levels", (long long)seg);
            const int64_t np = x.wb - x.wa + 1;
            const int64_t groups = (np + kMergeFanIn - 1) / kMergeFanIn;
            int64_t gsum = 0;
            for (int64_t j = 0; j < groups; ++j) {
                const int64_t g0 = x.wa + j * kMergeFanIn;
                const int64_t part = 2 * g0 + (g0 == x.wa ? x.first_slot : 0);
                CHECK(share_slot.count(part) && share_slot[part].seg == seg,
                      "segment %lld: group %lld partial over another segment's slot",
                      (long long)seg, (long long)j);
                const int64_t idx = j == 0 ? x.wa : kCounterRegion + g0;
                CHECK(counter_sum.count(idx) && counter_sum[idx] == counter_total[idx],
                      "segment %lld: group %lld counter incomplete", (long long)seg,
                      (long long)j);
                gsum += blocks_in(B, W, x.fs, x.nbs, x.wb, g0, kMergeFanIn);
            }
            CHECK(gsum == x.nbs, "segment %lld: groups hold %lld of %d blocks", (long long)seg,
                  (long long)gsum, x.nbs);
        } else {
            CHECK(!x.two_level, "segment %lld should merge in one level", (long long)seg);
            CHECK(counter_total[x.wa] == x.nbs, "segment %lld: one-level total",
                  (long long)seg);
        }
    }
    (void)rng;
}

int main(int argc, char** argv) {
    const int cases = argc > 1 ? std::atoi(argv[1]) : 3000;
    std::mt19937_64 rng(1540);
    int two_level = 0;
    for (int t = 0; t < cases; ++t) {
        const int kind = t % 4;
        std::vector<int> seg;
        const int nseg = 1 + (int)(rng() % (kind == 3 ? 4 : 300));
        for (int i = 0; i < nseg; ++i) {
            int len;
            if (kind == 0) len = 1 + (int)(rng() % 8);                 // short segments
            else if (kind == 1) len = 32 + (int)(rng() % 225);         // decode-like
            else if (kind == 2) len = 1 + (int)(rng() % 600);          // mixed
            else len = 500 + (int)(rng() % 8000);                      // few long ones
            seg.push_back(len);
        }
        int64_t B = 0;
        for (int l : seg) B += l;
        const int64_t workers = 1 + (int64_t)(rng() % 2048);
        run_case(rng, workers, seg);
        // count the calls with a two-level merge, to be sure they are exercised
        Params p{};
        p.workers = (int)workers;
        const int64_t W = share_count(p, B);
        int64_t f = 0;
        for (int l : seg) {
            if (share_of(f + l - 1, B, W) - share_of(f, B, W) + 1 > kMergeFanIn) {
                ++two_level;
                break;
            }
            f += l;
        }
    }
    std::printf("ok: %d call shapes, %d with two-level merges\n", cases, two_level);
    return two_level > 0 ? 0 : 1;
}
