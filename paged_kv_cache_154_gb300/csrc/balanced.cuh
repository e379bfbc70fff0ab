// The balanced decode schedule, shared by the 16-bit, INT8 and FP8 kernels.
//
// Work space. Each sequence s has nb_s = ceil(L_s / 16) blocks and R_s = G *
// r_s query rows per KV head (G q heads per KV head, r_s query tokens). Rows
// are served in tiles of RT (16 or 32); a sequence has C_s = ceil(R_s / RT)
// row chunks. A *segment* is (sequence, kv head, chunk); segments are laid
// out in order s, then kv head, then chunk, each as nb_s consecutive
// "virtual blocks". Chunks of one (sequence, kv head) read the same KV, and
// sit next to each other, so the workers that stream them do so at about
// the same time and the repeated reads mostly hit L2.
//
// Shares. The B virtual blocks are cut into W equal contiguous shares, one
// per worker warp: share w = [w*B/W, (w+1)*B/W). A segment that a share holds
// whole is written as final output by that warp. Where share boundaries cut
// a segment, every piece is written as a partial (m, l, O) to a slot -- slot
// 2w for the first segment of share w, 2w+1 for its last -- and the reduce
// kernel merges the pieces with the log-sum-exp rule.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>

#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {
namespace sched {

constexpr int kBS = 16;            // tokens per block
constexpr int kWorkerWarps = 4;    // warps per CTA

struct Params {
    void* out;
    const void* q;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* qsl;            // may be null: one query token per sequence
    int32_t* cum_out;              // workspace copy of the prefix sums [num_seqs + 1]
    uint8_t* slots;                // partial slots [2 * workers][slot_bytes]
    unsigned int* err;
    int max_blocks;
    int num_heads;
    int num_kv_heads;
    int group;                     // q heads per kv head
    int num_seqs;
    int num_blocks;
    int workers;
    int rows_per_tile;             // RT
    int slot_bytes;
    float scale_log2;              // softmax scale * log2(e)
    int out_f32;
    const int32_t* ctx_start;      // may be null; else sequence s attends tokens [ctx_start[s], L)
                                   // (a multiple of 16)
    float* lse_out;                // may be null; else [num_q_tokens][num_heads] base-2 log-sum-exp
                                   // of each output row, in scale * log2(e) units
    int unmasked;                  // 1: every query row sees every key < L (no causal offset)
    unsigned int* arrivals;        // may be null; else one counter per worker, zero on entry
                                   // and on exit: the decode kernel merges cut segments itself
};

// First block a sequence attends (0 unless ctx_start is given).
__device__ __forceinline__ int first_block(const Params& p, int s) {
    return p.ctx_start ? __ldg(p.ctx_start + s) / kBS : 0;
}


// A partial slot: int32 {seq, kv head, chunk, first token, end token, 0, 0, 0},
// then fp32 m[RT] (base-2 units), l[RT], O[RT][D] (not normalised). Row j of a
// slot is query row chunk*RT + j of the (sequence, kv head).
struct Slot {
    int32_t* hdr;
    float* m;
    float* l;
    float* o;
    __device__ __forceinline__ Slot(uint8_t* base, int rt) {
        hdr = reinterpret_cast<int32_t*>(base);
        m = reinterpret_cast<float*>(base + 32);
        l = m + rt;
        o = l + rt;
    }
};

__host__ __device__ __forceinline__ int64_t slot_bytes(int rt, int d) {
    return (32 + 4 * (int64_t)rt * (d + 2) + 15) / 16 * 16;
}

__device__ __forceinline__ int query_run(const int32_t* qsl, int s, int* q0) {
    if (!qsl) {
        *q0 = s;
        return 1;
    }
    *q0 = __ldg(qsl + s);
    return __ldg(qsl + s + 1) - *q0;
}

__device__ __forceinline__ int chunks_of(const Params& p, int s) {
    int q0;
    const int r = query_run(p.qsl, s, &q0);
    return (p.group * r + p.rows_per_tile - 1) / p.rows_per_tile;
}

// Causal block skipping: row chunk c of a sequence (L tokens, a query run of
// r, query i at position L - r + i) attends blocks first_block .. end - 1,
// where end is the block holding the last key that the chunk's last query
// row sees (all blocks with unmasked rows). A chunk of early queries of a
// long run -- a prefill -- thus skips the blocks no row of it can see.
__device__ __forceinline__ int chunk_blocks(const Params& p, int L, int r, int sb, int c) {
    const int nb = (L + kBS - 1) / kBS;
    int end = nb;
    if (!p.unmasked) {
        const int jmax = min(r - 1, ((c + 1) * p.rows_per_tile - 1) / p.group);
        end = min(nb, (L - r + jmax) / kBS + 1);
    }
    return max(0, end - sb);
}

// Blocks of every row chunk of sequence s together (one kv head).
__device__ __forceinline__ int seq_blocks(const Params& p, int s, int C) {
    int q0;
    const int L = __ldg(p.context_lens + s), r = query_run(p.qsl, s, &q0), sb = first_block(p, s);
    int total = 0;
    for (int c = 0; c < C; ++c) total += chunk_blocks(p, L, r, sb, c);
    return total;
}

// Blocks of segment (s, c); a single-chunk sequence reads it off the prefix sums.
__device__ __forceinline__ int segment_blocks(const Params& p, const int32_t* cum,
                                              const uint8_t* chunks, int s, int c) {
    if (chunks[s] == 1) return (cum[s + 1] - cum[s]) / p.num_kv_heads;
    int q0;
    const int r = query_run(p.qsl, s, &q0);
    return chunk_blocks(p, __ldg(p.context_lens + s), r, first_block(p, s), c);
}

__host__ __device__ __forceinline__ int64_t share_start(int64_t w, int64_t B, int64_t W) {
    return w * B / W;
}

// Shares the B virtual blocks are cut into: one per worker, but never more
// than there are blocks, so that every share holds at least one block
// (workers past the count get no share).
__host__ __device__ __forceinline__ int64_t share_count(const Params& p, int64_t B) {
    return max((int64_t)1, min((int64_t)p.workers, B));
}

// Shared-memory header of a balanced kernel: per-warp mbarriers, then
// cum[num_seqs + 1] (virtual blocks before each sequence) and chunks[num_seqs].
__host__ __device__ __forceinline__ int header_bytes(int num_seqs, int stages) {
    return ((kWorkerWarps * stages * 8 + (num_seqs + 1) * 4 + num_seqs) + 1023) / 1024 * 1024;
}

// cum[s] = num_kv_heads * (blocks of all row chunks of the sequences before
// s) and chunks[s] = C_s, by one CTA; CTA 0 also copies cum to the workspace
// for the reduce kernel.
static __device__ void build_prefix(int32_t* cum, uint8_t* chunks, const Params& p) {
    __shared__ int32_t warp_tot[32];
    pa::grid_dependents_launch();   // the reduce kernel may be scheduled early
    pa::grid_dependency_wait();     // inputs written by the previous kernel are visible
    const int n = p.num_seqs;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (n + nt - 1) / nt;
    const int a = min(n, tid * per), b = min(n, a + per);
    int32_t local = 0;
    for (int i = a; i < b; ++i) {
        const int c = chunks_of(p, i);
        chunks[i] = (uint8_t)c;
        local += p.num_kv_heads * seq_blocks(p, i, c);
    }
    const int lane = tid & 31, warp = tid >> 5;
    int32_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = nt >> 5;
        int32_t t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < nw) warp_tot[lane] = t;
    }
    __syncthreads();
    int32_t run = x - local + (warp > 0 ? warp_tot[warp - 1] : 0);
    for (int i = a; i < b; ++i) {
        cum[i] = run;
        run += p.num_kv_heads * seq_blocks(p, i, chunks[i]);
    }
    if (tid == nt - 1) cum[n] = run;
    __syncthreads();
    if (blockIdx.x == 0 && p.cum_out)
        for (int i = tid; i <= n; i += nt) p.cum_out[i] = cum[i];
}

// Position of virtual block f: sequence, kv head, chunk, block.
struct Pos {
    int s, g, c, b, nbs, C;
};

// Virtual blocks of a sequence are laid out kv head by kv head, and within a
// kv head chunk by chunk, each chunk's blocks in order.
__device__ __forceinline__ Pos locate(const Params& p, const int32_t* cum, const uint8_t* chunks,
                                      int64_t f) {
    const int n = p.num_seqs;
    int lo = 0, hi = n;   // largest s with cum[s] <= f
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid] <= f) lo = mid;
        else hi = mid;
    }
    Pos q;
    q.s = lo;
    q.C = chunks[lo];
    const int span = (cum[lo + 1] - cum[lo]) / p.num_kv_heads;   // one kv head's blocks
    const int local = (int)(f - cum[lo]);
    q.g = local / span;
    int rem = local - q.g * span;
    if (q.C == 1) {
        q.c = 0;
        q.nbs = span;
    } else {
        int q0;
        const int L = __ldg(p.context_lens + lo), r = query_run(p.qsl, lo, &q0);
        const int sb = first_block(p, lo);
        for (q.c = 0;; ++q.c) {
            q.nbs = chunk_blocks(p, L, r, sb, q.c);
            if (rem < q.nbs || q.c == q.C - 1) break;
            rem -= q.nbs;
        }
    }
    q.b = rem;
    return q;
}

// The next segment after (s, g, c) that has blocks.
__device__ __forceinline__ void next_segment(const Params& p, Pos& q, const int32_t* cum,
                                             const uint8_t* chunks) {
    q.b = 0;
    for (;;) {
        if (++q.c >= q.C) {
            q.c = 0;
            if (++q.g >= p.num_kv_heads) {
                q.g = 0;
                if (++q.s >= p.num_seqs) {
                    q.nbs = 0;
                    return;
                }
                q.C = chunks[q.s];
            }
        }
        q.nbs = segment_blocks(p, cum, chunks, q.s, q.c);
        if (q.nbs > 0) return;
    }
}

template <typename T>
__device__ __forceinline__ void store_out(void* out, int64_t idx, float v, int out_f32) {
    if (out_f32) static_cast<float*>(out)[idx] = v;
    else if constexpr (sizeof(T) == 2) {
        if constexpr (std::is_same<T, __half>::value)
            static_cast<__half*>(out)[idx] = __float2half_rn(v);
        else
            static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    }
}

// Merge records. A segment that share boundaries cut has its first piece in
// the share where it starts (share wa); that share's worker owns the merge.
// Every worker writes, on every call, words 5..7 of its second slot's header:
// {1, wb, slot of the first piece} for an owner (wb = the share holding the
// segment's last block), {0, 0, 0} otherwise; an owner also writes words 5, 6
// of its first slot's header: the segment's first query token and its rows in
// the tile. With the first piece's own header {sequence, kv head, chunk, ..}
// this is all the reduce needs, in one round of loads.
__device__ __forceinline__ void write_merge_record(const Params& p, int64_t wid, int owner,
                                                   int64_t wb, int first_slot, int q0 = 0,
                                                   int rows = 0) {
    if (wid >= p.workers) return;
    int32_t* h1 = reinterpret_cast<int32_t*>(p.slots + (2 * wid + 1) * (int64_t)p.slot_bytes);
    h1[5] = owner;
    h1[6] = (int32_t)wb;
    h1[7] = first_slot;
    if (owner) {
        int32_t* h0 = reinterpret_cast<int32_t*>(p.slots + 2 * wid * (int64_t)p.slot_bytes);
        h0[5] = q0;
        h0[6] = rows;
    }
}

// Called at the end of a share: is its last segment cut after the share (not
// all of its blocks done) and did it start in this share (its first piece
// here)? Then this worker owns the merge; wb = the share holding its last
// block, at virtual index f1 + (blocks left) - 1.
__device__ __forceinline__ void record_last_segment(const Params& p, int64_t wid, int64_t f1,
                                                    int64_t B, bool seg_done, int seg_b0,
                                                    int blocks_left, bool seg_first, int q0,
                                                    int rows) {
    if (!seg_done && seg_b0 == 0) {
        const int64_t fb = f1 + blocks_left;                 // one past the segment's end
        write_merge_record(p, wid, 1, (fb * share_count(p, B) - 1) / B, seg_first ? 0 : 1, q0,
                           rows);
    }
}

// The share holding virtual block f: the largest w with share_start(w) <= f.
__host__ __device__ __forceinline__ int64_t share_of(int64_t f, int64_t B, int64_t W) {
    return ((f + 1) * W - 1) / B;
}

// In-kernel merge of cut segments. The pieces of a cut segment are merged by
// whichever piece finishes last, so no reduce kernel runs after the decode
// kernel and merges overlap other warps' streaming. After writing its slot,
// a piece's warp adds its block count to a counter; the warp whose addition
// completes the count knows that every piece it covers is written, merges
// them, and resets the counter to zero for the next call. A segment of at
// most kMergeFanIn shares is merged in one level (counter: by the share
// where the segment starts). A longer one -- a long sequence cut by many
// shares -- in two: the shares are grouped kMergeFanIn at a time, the last
// piece of a group folds the group into one partial (m, l, O) written over
// the slot of the group's first piece, and the last group to finish merges
// the group partials. Counters live in three regions of kBalancedMaxWorkers
// each, so no two levels or segments share one: group 0 (or a whole short
// segment) by the segment's first share, groups 1.. by their first share (a
// middle share of the segment, which no other segment's group can start
// at), and the second level by the segment's first share.
constexpr int kMergeFanIn = 8;
constexpr int kCounterRegion = pa::kBalancedMaxWorkers;   // counters per region

// Release: the warp barrier orders every lane's stores before lane 0's
// acq_rel atomic (cumulative, as a CTA barrier before a thread's release);
// acquire: the same atomic, then a warp barrier before the lanes read the
// pieces (through L2, ld.global.cg). A count past the total, before or
// after the addition, means the counters were not zero on entry.
__device__ __forceinline__ bool arrive(const Params& p, unsigned int* cnt, int add, int total,
                                       int lane) {
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        unsigned int old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                     : "=r"(old)
                     : "l"(cnt), "r"((unsigned int)add)
                     : "memory");
        const unsigned int now = old + (unsigned int)add;
        // a clean counter never exceeds its total: checking the old value as
        // well catches a dirty one that the addition wrapped around
        if ((old > (unsigned int)total || now > (unsigned int)total) && p.err)
            atomicOr(p.err, pa::ERR_WORKSPACE);
        last = now == (unsigned int)total;
        if (last) atomicExch(cnt, 0u);   // no other piece counts here in this launch
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    __syncwarp();
    return last != 0;
}

// Blocks of segment [fs, fs + nbs) held by shares sh .. min(sh + span - 1, wb).
__host__ __device__ __forceinline__ int64_t blocks_in(int64_t B, int64_t W, int64_t fs, int nbs,
                                             int64_t wb, int64_t sh, int span) {
    const int64_t b0 = max(fs, share_start(sh, B, W));
    const int64_t b1 = min(fs + nbs, share_start(min(sh + span - 1, wb) + 1, B, W));
    return max((int64_t)0, b1 - b0);
}

// Partials staged in shared memory at a time by fold_partials, and the
// shared memory it needs for them (four rows of D fp32 each).
constexpr int kFoldBatch = 8;
__host__ __device__ constexpr int fold_stage_bytes(int d) { return kFoldBatch * 4 * d * 4; }

// Folds, row by row, the partials at shares s0, s0 + step, .. <= s1 of the
// segment of nbs blocks from virtual block fs, held by shares wa .. wb (the
// piece in wa in slot first_slot, the others in slot 0); with step 1 the
// pieces themselves, with step kMergeFanIn the group partials. A share (or
// group) holding no block of the segment wrote nothing and is skipped. Four
// rows at a time: the rows of kFoldBatch partials are copied at once into
// the warp's free staging buffer (cp.async, one round trip for the batch),
// then every lane folds its D / 8 columns of one row with the log-sum-exp
// rule. The result goes to slot `part` as a partial (m = M, l = sum
// 2^(m_i - M) l_i, O = sum 2^(m_i - M) O_i) with the header of a piece
// covering the shares s0 .. s1, or, with part null, to the output as O / l
// (row j of the tile is query row c * RT + j of sequence s, first query
// token q0, kv head g).
template <typename T, int D>
__device__ __forceinline__ void fold_partials(const Params& p, int64_t B, int64_t fs, int nbs,
                                              int64_t wa, int64_t wb, int first_slot, int64_t s0,
                                              int64_t s1, int step, int rows, uint8_t* part, int s,
                                              int g, int c, int q0, uint32_t stage, int lane) {
    constexpr int EPL = D / 8;
    constexpr int kRowBytes = D * 4;
    constexpr int kPerLane = 4 * kRowBytes / 16 / 32;   // 16-byte chunks a lane copies per partial
    const int64_t W = share_count(p, B);
    const int RT = p.rows_per_tile, G = p.group;
    const int cp = lane & 7;
    // with at least as many blocks as shares every share holds one: no
    // share (nor group) of the segment is empty, and no division is needed
    const bool may_be_empty = B < W;
    if (part && lane == 0) {
        // tokens of the blocks of the segment in shares s0 .. s1
        const int64_t b0 = max(fs, share_start(s0, B, W));
        const int64_t b1 = min(fs + nbs, share_start(s1 + 1, B, W));
        const int sb = first_block(p, s);
        int32_t* hdr = reinterpret_cast<int32_t*>(part);
        hdr[0] = s;
        hdr[1] = g;
        hdr[2] = c;
        hdr[3] = (sb + (int)(b0 - fs)) * kBS;
        hdr[4] = min((sb + (int)(b1 - fs)) * kBS, __ldg(p.context_lens + s));
    }
    // the staging buffer was last written by the tensor-copy engine
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int r0 = 0; r0 < rows; r0 += 4) {
        const int row = r0 + (lane >> 3);
        const bool on = row < rows;
        float M = -INFINITY, den = 0.f, acc[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
        for (int64_t x0 = s0; x0 <= s1; x0 += (int64_t)step * kFoldBatch) {
            float mv[kFoldBatch], lv[kFoldBatch];
            __syncwarp();   // every lane is done with the previous batch in the buffer
#pragma unroll
            for (int j = 0; j < kFoldBatch; ++j) {
                const int64_t sh = x0 + (int64_t)j * step;
                lv[j] = 0.f;
                mv[j] = -INFINITY;
                if (sh > s1 || (may_be_empty && blocks_in(B, W, fs, nbs, wb, sh, step) == 0))
                    continue;                                               // warp-uniform
                Slot sl(p.slots + (2 * sh + (sh == wa ? first_slot : 0)) * (int64_t)p.slot_bytes, RT);
                if (on) {
                    lv[j] = __ldcg(sl.l + row);
                    mv[j] = __ldcg(sl.m + row);
                }
                // rows r0 .. r0 + 3 of the partial (r0 + 4 <= RT: in the slot)
                const char* src = reinterpret_cast<const char*>(sl.o + (int64_t)r0 * D);
#pragma unroll
                for (int i = 0; i < kPerLane; ++i) {
                    const int ch = lane + 32 * i;
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                     stage + (uint32_t)(j * 4 * kRowBytes + ch * 16)),
                                 "l"(src + ch * 16)
                                 : "memory");
                }
            }
            asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
            __syncwarp();
#pragma unroll
            for (int j = 0; j < kFoldBatch; ++j) {
                if (!(lv[j] > 0.f)) continue;          // no partial, or no visible key in it
                const float Mn = fmaxf(M, mv[j]);
                const float a = exp2f(M - Mn), b = exp2f(mv[j] - Mn);
                den = den * a + b * lv[j];
                const uint32_t at = stage + (uint32_t)(j * 4 * kRowBytes + (row - r0) * kRowBytes +
                                                       cp * EPL * 4);
#pragma unroll
                for (int e = 0; e < EPL / 4; ++e) {
                    float x, y, z, w;
                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(x), "=f"(y), "=f"(z), "=f"(w)
                                 : "r"(at + 16 * e));
                    acc[4 * e + 0] = acc[4 * e + 0] * a + b * x;
                    acc[4 * e + 1] = acc[4 * e + 1] * a + b * y;
                    acc[4 * e + 2] = acc[4 * e + 2] * a + b * z;
                    acc[4 * e + 3] = acc[4 * e + 3] * a + b * w;
                }
                M = Mn;
            }
        }
        if (part) {
            if (on) {
                Slot sl(part, RT);
                if (cp == 0) {
                    sl.m[row] = M;
                    sl.l[row] = den;
                }
                float4* dst = reinterpret_cast<float4*>(sl.o + (int64_t)row * D + cp * EPL);
#pragma unroll
                for (int e = 0; e < EPL / 4; ++e)
                    dst[e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
            }
            continue;
        }
        if (!on) continue;
        const int grow = c * RT + row;
        const int64_t orow = (int64_t)(q0 + grow / G) * p.num_heads + g * G + grow % G;
        const int64_t base = orow * D + cp * EPL;
        const float inv = 1.f / den;
        if (p.lse_out && cp == 0) p.lse_out[orow] = M + log2f(den);
        if (p.out_f32) {
#pragma unroll
            for (int e = 0; e < EPL / 4; ++e)
                reinterpret_cast<float4*>(static_cast<float*>(p.out) + base)[e] =
                    make_float4(acc[4 * e] * inv, acc[4 * e + 1] * inv, acc[4 * e + 2] * inv,
                                acc[4 * e + 3] * inv);
        } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) store_out<T>(p.out, base + e, acc[e] * inv, 0);
        }
    }
}

// A piece of a cut segment, as the warp that wrote it sees it: pb of the
// segment's nbs blocks (from virtual block fs, held by shares wa .. wb, its
// first piece in slot first_slot of share wa) of (sequence s, kv head g, row
// chunk c; first query token q0, rows rows of the tile); the counter it
// counts its blocks into and the total that completes that counter; for a
// segment of more than kMergeFanIn shares, the group g0 .. g1 it belongs to.
struct CutPiece {
    int64_t fs, wa, wb, g0, g1;
    unsigned int* cnt;
    int pb, nbs, s, g, c, q0, rows, first_slot, total;
    bool two_level;
};

// wa_known / wb_known: the first / last share of the segment when the caller
// knows it (-1 otherwise), which spares a 64-bit division each; f_wa: the
// first block of share wa when wa_known.
__host__ __device__ __forceinline__ CutPiece cut_piece(const Params& p, int64_t B, int64_t wme, int64_t fs,
                                              int pb, int nbs, int s, int g, int c, int q0,
                                              int rows, int64_t wa_known, int64_t f_wa,
                                              int64_t wb_known) {
    const int64_t W = share_count(p, B);
    CutPiece x;
    x.fs = fs;
    x.pb = pb;
    x.nbs = nbs;
    x.s = s;
    x.g = g;
    x.c = c;
    x.q0 = q0;
    x.rows = rows;
    x.wa = wa_known >= 0 ? wa_known : share_of(fs, B, W);
    x.wb = wb_known >= 0 ? wb_known : share_of(fs + nbs - 1, B, W);
    x.first_slot = (wa_known >= 0 ? f_wa : share_start(x.wa, B, W)) == fs ? 0 : 1;
    x.two_level = x.wb - x.wa + 1 > kMergeFanIn;
    if (!x.two_level) {
        x.g0 = x.wa;
        x.g1 = x.wb;
        x.cnt = p.arrivals + x.wa;
        x.total = nbs;
    } else {
        const int64_t j = (wme - x.wa) / kMergeFanIn;
        x.g0 = x.wa + j * kMergeFanIn;
        x.g1 = min(x.g0 + kMergeFanIn - 1, x.wb);
        x.cnt = j == 0 ? p.arrivals + x.wa : p.arrivals + kCounterRegion + x.g0;
        x.total = (int)blocks_in(B, W, fs, nbs, x.wb, x.g0, kMergeFanIn);
    }
    return x;
}

// Counts up to two pieces of a warp in at once (lane 0 the first, lane 1 the
// second: one round trip for both); bit 0 / bit 1 of the result: that piece
// completed its counter. Ordering as in arrive().
__device__ __forceinline__ int arrive_pair(const Params& p, const CutPiece& a, bool has_a,
                                           const CutPiece& b, bool has_b, int lane) {
    __syncwarp();
    int last = 0;
    if ((lane == 0 && has_a) || (lane == 1 && has_b)) {
        unsigned int* cnt = lane == 0 ? a.cnt : b.cnt;
        const int add = lane == 0 ? a.pb : b.pb, total = lane == 0 ? a.total : b.total;
        unsigned int old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                     : "=r"(old)
                     : "l"(cnt), "r"((unsigned int)add)
                     : "memory");
        const unsigned int now = old + (unsigned int)add;
        // a clean counter never exceeds its total: checking the old value as
        // well catches a dirty one that the addition wrapped around
        if ((old > (unsigned int)total || now > (unsigned int)total) && p.err)
            atomicOr(p.err, pa::ERR_WORKSPACE);
        last = now == (unsigned int)total;
        if (last) atomicExch(cnt, 0u);   // no other piece counts here in this launch
    }
    const int la = __shfl_sync(0xffffffffu, last, 0), lb = __shfl_sync(0xffffffffu, last, 1);
    __syncwarp();
    return la | (lb << 1);
}

// After x completed its counter: merge the segment (one level), or fold the
// group into its partial and, if that completes the segment's groups, merge
// the group partials (stage: fold_stage_bytes(D) bytes of this warp's
// shared memory, free).
template <typename T, int D>
__device__ __forceinline__ void merge_cut(const Params& p, int64_t B, const CutPiece& x,
                                          uint32_t stage, int lane) {
    const int64_t W = share_count(p, B);
    if (!x.two_level) {
        fold_partials<T, D>(p, B, x.fs, x.nbs, x.wa, x.wb, x.first_slot, x.wa, x.wb, 1, x.rows,
                            nullptr, x.s, x.g, x.c, x.q0, stage, lane);
        return;
    }
    uint8_t* part =
        p.slots + (2 * x.g0 + (x.g0 == x.wa ? x.first_slot : 0)) * (int64_t)p.slot_bytes;
    fold_partials<T, D>(p, B, x.fs, x.nbs, x.wa, x.wb, x.first_slot, x.g0, x.g1, 1, x.rows, part,
                        x.s, x.g, x.c, x.q0, stage, lane);
    // groups that hold blocks (with more shares than blocks, whole groups can be empty)
    const int64_t np = x.wb - x.wa + 1;
    int groups = (int)((np + kMergeFanIn - 1) / kMergeFanIn);
    if (B < W) {
        groups = 0;
        for (int64_t y = x.wa + (int64_t)lane * kMergeFanIn; y <= x.wb; y += 32 * kMergeFanIn)
            groups += blocks_in(B, W, x.fs, x.nbs, x.wb, y, kMergeFanIn) > 0;
        groups = __reduce_add_sync(0xffffffffu, groups);
    }
    if (arrive(p, p.arrivals + 2 * kCounterRegion + x.wa, 1, groups, lane))
        fold_partials<T, D>(p, B, x.fs, x.nbs, x.wa, x.wb, x.first_slot, x.wa, x.wb, kMergeFanIn,
                            x.rows, nullptr, x.s, x.g, x.c, x.q0, stage, lane);
}

// Merges the pieces of every cut segment: CTAs of kReduceWarps warps over
// (worker, group of kReduceWarps rows), reading the worker's two slot headers
// in one round; a non-owner (or a row group past the segment's rows) returns
// at once. A row with its own warp (or, with fewer rows than warps, wpr warps
// that split its pieces and meet in shared memory) is merged in two passes: the
// lanes take the pieces' (m, l) 32 at a time for the row's largest m and the
// denominator sum 2^(m - M) l; then, the weights known, every lane adds its
// D / 32 columns of every piece with independent loads (no chain through
// the running maximum): out = sum 2^(m - M) O / sum 2^(m - M) l.
template <typename T, int D, int kReduceWarps>
__global__ void __launch_bounds__(32 * kReduceWarps, 32 / kReduceWarps) segment_reduce_kernel(
    const Params p, int row_groups) {
    constexpr int EPL = D / 32;
    constexpr int kUnroll = 4;                      // pieces whose loads are in flight together
    __shared__ int32_t hdr[17];                     // slot 0 words 0..7, slot 1 words 0..7, B
    __shared__ float part[kReduceWarps][D + 2];
    pa::grid_dependency_wait();     // the decode kernel's partials must be complete
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t w = blockIdx.x / row_groups;
    const int rg = (int)(blockIdx.x % row_groups);
    if (w >= p.workers) return;
    if (threadIdx.x < 16)
        hdr[threadIdx.x] = __ldg(reinterpret_cast<const int32_t*>(
                                     p.slots + (2 * w + (threadIdx.x >> 3)) *
                                                   (int64_t)p.slot_bytes) +
                                 (threadIdx.x & 7));
    else if (threadIdx.x == 16)
        hdr[16] = __ldg(p.cum_out + p.num_seqs);
    __syncthreads();
    if (hdr[8 + 5] != 1) return;                    // not the owner of a cut segment
    const int64_t wb = hdr[8 + 6];
    const int first_slot = hdr[8 + 7];
    const int32_t* piece = hdr + 8 * first_slot;
    const int g = piece[1], c = piece[2];
    const int q0 = hdr[5], rows_all = hdr[6];
    const int row0 = rg * kReduceWarps;
    if (row0 >= rows_all) return;
    const int rows = min(kReduceWarps, rows_all - row0);
    const int RT = p.rows_per_tile, G = p.group;
    const int64_t B = hdr[16];
    const int64_t W = share_count(p, B);
    const bool may_be_empty = B < W;                 // only then can a share hold no block
    // warps per row: the largest power of two with wpr x rows <= kReduceWarps (one round)
    int wpr = 1;
    while (2 * wpr * rows <= kReduceWarps) wpr *= 2;
    const int row = row0 + warp / wpr, sub = warp % wpr;
    const bool active = warp / wpr < rows;
    const int64_t np = wb - w + 1;                    // pieces of the segment (shares w .. wb)
    auto slot_of = [&](int64_t x) {                   // the piece of share w + x, or null
        const int64_t sh = w + x;
        if (may_be_empty && sh != w && share_start(sh, B, W) == share_start(sh + 1, B, W))
            return (uint8_t*)nullptr;
        // later shares start inside the segment: their piece is in slot 0
        return p.slots + (2 * sh + (sh == w ? first_slot : 0)) * (int64_t)p.slot_bytes;
    };
    float M = -INFINITY, den = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    if (active) {
        // pass 1: the row's largest m over this warp's pieces (sub, sub + wpr, ...)
        for (int64_t x = sub + (int64_t)wpr * lane; x < np; x += (int64_t)wpr * 32) {
            const uint8_t* sp = slot_of(x);
            if (!sp) continue;
            Slot sl(const_cast<uint8_t*>(sp), RT);
            if (__ldg(sl.l + row) > 0.f) M = fmaxf(M, __ldg(sl.m + row));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        // pass 2: weights 2^(m - M), the denominator and the columns
        if (M != -INFINITY) {
            for (int64_t x0 = sub; x0 < np; x0 += (int64_t)wpr * kUnroll) {
                float wv[kUnroll], lv[kUnroll], ov[kUnroll][EPL];
#pragma unroll
                for (int j = 0; j < kUnroll; ++j) {
                    const int64_t x = x0 + (int64_t)j * wpr;
                    wv[j] = 0.f;
                    lv[j] = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) ov[j][e] = 0.f;
                    const uint8_t* sp = x < np ? slot_of(x) : nullptr;
                    if (sp) {
                        Slot sl(const_cast<uint8_t*>(sp), RT);
                        lv[j] = __ldg(sl.l + row);
                        wv[j] = __ldg(sl.m + row);
                        const float* src = sl.o + (int64_t)row * D + lane * EPL;
                        if constexpr (EPL == 4) {
                            const float4 t = __ldg(reinterpret_cast<const float4*>(src));
                            ov[j][0] = t.x; ov[j][1] = t.y; ov[j][2] = t.z; ov[j][3] = t.w;
                        } else {
                            const float2 t = __ldg(reinterpret_cast<const float2*>(src));
                            ov[j][0] = t.x; ov[j][1] = t.y;
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < kUnroll; ++j) {
                    const float wgt = lv[j] > 0.f ? exp2f(wv[j] - M) : 0.f;
                    den += wgt * lv[j];
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[e] += wgt * ov[j][e];
                }
            }
        }
    }
    if (wpr > 1) {
        // the row's warps meet in shared memory; the first of them folds
#pragma unroll
        for (int e = 0; e < EPL; ++e) part[warp][lane * EPL + e] = acc[e];
        if (lane == 0) {
            part[warp][D] = M;
            part[warp][D + 1] = den;
        }
        __syncthreads();
        if (active && sub == 0) {
            float Mt = -INFINITY;
            for (int j = 0; j < wpr; ++j)
                if (part[warp + j][D + 1] > 0.f) Mt = fmaxf(Mt, part[warp + j][D]);
            float dt = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
            for (int j = 0; j < wpr; ++j) {
                const float wgt = part[warp + j][D + 1] > 0.f ? exp2f(part[warp + j][D] - Mt) : 0.f;
                dt += wgt * part[warp + j][D + 1];
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[e] += wgt * part[warp + j][lane * EPL + e];
            }
            M = Mt;
            den = dt;
        }
    }
    if (!active || sub != 0) return;
    const int grow = c * RT + row;
    const int64_t orow = (int64_t)(q0 + grow / G) * p.num_heads + g * G + grow % G;
    const int64_t base = orow * D + lane * EPL;
    const float inv = 1.f / den;
    if (p.lse_out && lane == 0) p.lse_out[orow] = M + log2f(den);
    if constexpr (EPL == 4) {
        if (p.out_f32) {
            *reinterpret_cast<float4*>(static_cast<float*>(p.out) + base) =
                make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
            return;
        }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) store_out<T>(p.out, base + e, acc[e] * inv, p.out_f32);
}

// Merges the pieces of every cut segment, one warp per (sequence, kv head,
// chunk, query row) -- a flat grid of 4-warp CTAs over num_seqs x num_kv_heads
// x max_chunks x row_slots items (row_slots = the most rows a chunk can have)
// -- so the items that exist run in about one wave. A lane owns D / 32
// columns. Pieces are read eight at a time (independent loads), then folded
// into an online log-sum-exp: out = sum 2^(m - M) O / sum 2^(m - M) l.
template <typename T, int D>
__global__ void __launch_bounds__(128) segment_reduce_rows_kernel(const Params p, int max_chunks,
                                                             int row_slots) {
    constexpr int EPL = D / 32;
    constexpr int kBatch = 8;
    pa::grid_dependency_wait();     // the decode kernel's partials must be complete
    const int lane = threadIdx.x & 31;
    int64_t item = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int row = (int)(item % row_slots);
    item /= row_slots;
    const int gc = (int)(item % (p.num_kv_heads * max_chunks));
    const int s = (int)(item / (p.num_kv_heads * max_chunks));
    if (s >= p.num_seqs) return;
    const int C = chunks_of(p, s);
    const int g = gc / C, c = gc - (gc / C) * C;
    if (g >= p.num_kv_heads) return;
    int q0;
    const int r = query_run(p.qsl, s, &q0);
    const int G = p.group, RT = p.rows_per_tile;
    if (row >= min(RT, G * r - c * RT)) return;    // before any 64-bit division
    const int L = __ldg(p.context_lens + s), sb = first_block(p, s);
    const int nbs = chunk_blocks(p, L, r, sb, c);
    if (nbs == 0) return;                          // nothing attended: no output row
    const int64_t B = __ldg(p.cum_out + p.num_seqs);
    const int64_t W = share_count(p, B);
    int before = 0;                                // blocks of the chunks before c
    for (int cc = 0; cc < c; ++cc) before += chunk_blocks(p, L, r, sb, cc);
    const int span = (__ldg(p.cum_out + s + 1) - __ldg(p.cum_out + s)) / p.num_kv_heads;
    const int64_t fa = __ldg(p.cum_out + s) + (int64_t)g * span + before;
    const int64_t fb = fa + nbs;
    const int64_t wa = ((fa + 1) * W - 1) / B;     // share holding virtual block fa
    const int64_t wb = (fb * W - 1) / B;           // share holding virtual block fb - 1
    if (wa == wb) return;                          // written whole by that share
    // share wa holds the segment's first piece in its second slot unless the
    // segment starts exactly where the share does; later shares hold their
    // piece in their first slot (they start inside the segment)
    const int first_slot = share_start(wa, B, W) < fa ? 1 : 0;
    const bool may_be_empty = B < W;               // only then can a share hold no block
    float M = -INFINITY, den = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    for (int64_t w0 = wa; w0 <= wb; w0 += kBatch) {
        float lv[kBatch], mv[kBatch], ov[kBatch][EPL];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int64_t w = w0 + j;
            bool ok = w <= wb;
            if (ok && may_be_empty) ok = share_start(w, B, W) != share_start(w + 1, B, W);
            lv[j] = 0.f;
            mv[j] = -INFINITY;
#pragma unroll
            for (int e = 0; e < EPL; ++e) ov[j][e] = 0.f;
            if (ok) {
                const int slot = w == wa ? first_slot : 0;
                Slot sl(p.slots + (2 * w + slot) * (int64_t)p.slot_bytes, RT);
                lv[j] = __ldg(sl.l + row);
                mv[j] = __ldg(sl.m + row);
                const float* src = sl.o + (int64_t)row * D + lane * EPL;
                if constexpr (EPL == 4) {
                    const float4 t = __ldg(reinterpret_cast<const float4*>(src));
                    ov[j][0] = t.x; ov[j][1] = t.y; ov[j][2] = t.z; ov[j][3] = t.w;
                } else {
                    const float2 t = __ldg(reinterpret_cast<const float2*>(src));
                    ov[j][0] = t.x; ov[j][1] = t.y;
                }
            }
        }
        float Mb = M;
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (lv[j] > 0.f) Mb = fmaxf(Mb, mv[j]);
        if (Mb == -INFINITY) continue;                 // no piece of this batch saw a key
        const float a = exp2f(M - Mb);
        den *= a;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] *= a;
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const float wgt = lv[j] > 0.f ? exp2f(mv[j] - Mb) : 0.f;
            den += wgt * lv[j];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] += wgt * ov[j][e];
        }
        M = Mb;
    }
    const int grow = c * RT + row;
    const int64_t base =
        ((int64_t)(q0 + grow / G) * p.num_heads + g * G + grow % G) * D + lane * EPL;
    const float inv = 1.f / den;
    if (p.lse_out && lane == 0)
        p.lse_out[(int64_t)(q0 + grow / G) * p.num_heads + g * G + grow % G] = M + log2f(den);
    if constexpr (EPL == 4) {
        if (p.out_f32) {
            *reinterpret_cast<float4*>(static_cast<float*>(p.out) + base) =
                make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
            return;
        }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) store_out<T>(p.out, base + e, acc[e] * inv, p.out_f32);
}

// Launch the reduce for a balanced decode call (PDL, after the decode kernel).
// One CTA per worker by default: only the owners of cut segments do any work,
// reading the merge records the decode kernel left. The phases of a read-once
// shared-prefix call (the ones that write log-sum-exp rows) merge long
// fork-group prefixes cut into many pieces with up to G x forks rows each;
// there one warp per (sequence, kv head, chunk, row) item merges its own row
// in parallel, while there are at most 64K items.
template <typename T, int D>
cudaError_t launch_segment_reduce(const Params& prm, int max_chunks, int row_slots,
                                  cudaStream_t stream) {
    const int64_t items = (int64_t)prm.num_seqs * prm.num_kv_heads * max_chunks * row_slots;
    if (prm.lse_out && items <= (1 << 16))
        return pa::launch_pdl(segment_reduce_rows_kernel<T, D>, dim3((unsigned)((items + 3) / 4)),
                              dim3(128), 0, stream, prm, max_chunks, row_slots);
    // CTAs over (worker, group of rows) of the most rows a chunk holds: four
    // warps (and rows) a CTA when segments are cut into few pieces (workers
    // per segment, on average, at most 8); eight when few long segments are
    // each cut into many pieces, which the warps of a row then share.
    const int64_t segments = (int64_t)prm.num_seqs * prm.num_kv_heads * max_chunks;
    if (prm.workers <= 8 * segments) {
        const int row_groups = (row_slots + 3) / 4;
        return pa::launch_pdl(segment_reduce_kernel<T, D, 4>, dim3((unsigned)(prm.workers * row_groups)),
                              dim3(128), 0, stream, prm, row_groups);
    }
    const int row_groups = (row_slots + 7) / 8;
    return pa::launch_pdl(segment_reduce_kernel<T, D, 8>, dim3((unsigned)(prm.workers * row_groups)),
                          dim3(256), 0, stream, prm, row_groups);
}

}  // namespace sched
}  // namespace pa
