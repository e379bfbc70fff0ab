// Paged decode attention over an INT8 cache on the 5th-generation tensor
// cores (tcgen05, TMEM), for calls averaging at least 64 query rows per KV
// head (MQA or GQA verify steps) at head_dim 128.
//
// The cache holds codes x_q with one fp32 scale and int8 zero point per
// (token, kv head); a value is (x_q - zp) * scale ("cs336 lecture 10",
// Quantization). The attention, softmax(Q K^T / sqrt(d)) V ("KV Cache ...
// PagedAttention" §二), is computed with the cached tokens in the M dimension
// of the products, so that one CTA converts each code once for every query
// row of its (sequence, kv head) and the softmax runs one thread per token.
// Per tile of 128 tokens (eight 16-token blocks) and a chunk of at most 96
// query rows, with fp16 operands and fp32 accumulators in TMEM:
//
//   S^T = Kc Q^T     M 128 tokens x N rows x K 128 dims. Kc = K codes - zp,
//                    an exact integer in fp16, written by the converter warps
//                    straight into TMEM (token t in lane t) and read from
//                    there as the A operand; Q in shared memory (K-major),
//                    each row scaled by a power of two so that its fp16 copy
//                    is exact and uses the whole fp16 range.
//   softmax          one thread per token: s = S^T * k_scale * (row scale)
//                    in base-2 units; online softmax per column (query row)
//                    whose running max is moved only when a tile raises it by
//                    more than 2^8 -- then the tile's column maxima come from
//                    a transposing warp reduction and shared memory.
//   O^T += V' P^T    M 128 dims x N x K 128 tokens. V' = (V codes - zp) *
//                    v_scale / 2^e in shared memory (MN-major A), 2^e a
//                    running power-of-two reference (the largest V scale
//                    seen, rounded up; O is rescaled by an exact power of two
//                    when it grows), P (fp16, K-major B) from the softmax.
//   l   += 1 P^T     the same B against an all-ones A: every TMEM lane of l
//                    holds the column sums of P, so the denominators need no
//                    column reduction.
//
// Work split: the segments of the balanced schedule (balanced.cuh) with row
// chunks of 96, cut into one share per CTA (one CTA per SM) by cost rather
// than by blocks (see "Shares balanced by cost" below); segments cut by share
// boundaries go to partial slots that segment_reduce_kernel merges. Roles:
// warp 0 streams the code tiles (TMA, one 16-token block per lane) into a
// 4-stage ring; warps 1-4 convert (one token per thread, its scales and zero
// point by plain loads one tile ahead); warps 5-8 run the softmax and the
// epilogue; warp 9 issues the MMAs. Every wait is bounded; a wait that gives
// up sets an error bit, after which every other wait of the call returns at
// once, and the roles run out their loops without further copies or
// products.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <float.h>
#include <math.h>

#include <algorithm>

#include "balanced.cuh"
#include "pa_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace {

using pa::sched::kBS;
using pa::sched::Pos;
constexpr int D = 128;
constexpr int kTok = 128;                   // tokens per tile (TMEM lanes, MMA M)
constexpr int kTileBlocks = kTok / kBS;     // 8
constexpr int kRT = 96;                     // query rows per chunk (MMA N at most)
constexpr int kStages = 4;                  // code staging ring
constexpr int kThreads = 320;               // producer, 4 converter warps, 4 softmax warps, MMA
constexpr int kMaxSeqs = 1536;              // sequences per call (prefix sums in shared memory)
constexpr float kLazyMax = 8.f;             // base-2 headroom before the running max moves
constexpr uint32_t kMagic = 0x64646464u;

// shared memory, offsets from a 1024-byte aligned base
constexpr int kCodes = kTok * D;            // one tile of K (or V) codes
// A stage: K codes, then V codes (128-byte swizzled rows, token t in row t).
// The converters overwrite it in place with V' (fp16, dims 0-63 over the K
// codes once those are in TMEM, dims 64-127 over the V codes a thread has
// read), which the O product reads; the stage is free again once that
// product is done.
constexpr int kStageBytes = 2 * kCodes;
constexpr int kHalfV = kTok * 128;          // one 64-dim half of V' (= kCodes)
constexpr int kQOff = kStages * kStageBytes; // Q fp16 [2 dim halves][96 rows][128 B]
constexpr int kHalfQ = kRT * 128;
constexpr int kPOff = kQOff + 2 * kHalfQ;   // P fp16, 2 buffers of [2 token halves][96 rows][128 B]
constexpr int kPBuf = 2 * kHalfQ;
constexpr int kOnesOff = kPOff + 2 * kPBuf; // 128 x 16 fp16 ones, no swizzle (4 KB)
constexpr int kInfoOff = kOnesOff + 4096;
constexpr int kInfoBytes = 1024;            // per tile (2 entries): ks[128], rm[96], vfix, vref
constexpr int kInfoRm = 128, kInfoVfix = 224, kInfoVref = 225;   // float indices
constexpr int kRedOff = kInfoOff + 2 * kInfoBytes;   // vmax[2][4]; then colmax[4][96], mr, mu,
constexpr int kRedBytes = 4096;                      // alpha, bound, zero [96]
constexpr int kBarOff = kRedOff + kRedBytes;
constexpr int kHdrOff = kBarOff + 256;
static_assert(kHalfV == kCodes, "V' halves over the code halves");
static_assert(kQOff % 1024 == 0 && kPOff % 1024 == 0 && kOnesOff % 1024 == 0 && kHalfQ % 1024 == 0,
              "128-byte swizzle atoms");
static_assert(64 + 9 * kRT * 4 <= kRedBytes, "reduction area");
static_assert(kHdrOff + ((kMaxSeqs + 1) * 4 + kMaxSeqs + 15) / 16 * 16 + 1024 + 256 <= 227 * 1024,
              "shared memory per CTA");

// mbarriers (pairs are indexed by tile parity, stages by tile mod kStages)
enum : int {
    kFull = 0,                       // codes of a stage landed (producer + copies)
    kEmpty = kFull + kStages,        // a stage's O product done: the stage is free
    kKReady = kEmpty + kStages,      // [2] Kc in TMEM and the tile's info written
    kInfoFree = kKReady + 2,         // [2] softmax done with a tile's Kc buffer and info
    kSFull = kInfoFree + 2,          // [2] S^T of a tile computed
    kSFree = kSFull + 2,             // [2] softmax done reading an S buffer
    kVReady = kSFree + 2,            // V' of a stage written (per stage: the converters may run
                                     // two tiles past the oldest O product not yet issued)
    kPFull = kVReady + kStages,      // [2] P of a tile written (O, l rescaled if needed)
    kODone = kPFull + 2,             // [2] a tile's O and l products done (its P buffer free)
    kOFree = kODone + 2,             // epilogue of a piece done reading O and l
    kFin = kOFree + 1,               // every product of the CTA done
    kNumBars = kFin + 1
};
static_assert(8 * kNumBars + 16 <= 256, "barrier area");

// TMEM columns: two S buffers of up to 96, O, l, two Kc buffers of 64
constexpr uint32_t kColS = 0, kColO = 2 * kRT, kColL = 3 * kRT, kColK = 4 * kRT;
constexpr uint32_t kTmemCols = 512;
static_assert(kColK + 2 * 64 <= kTmemCols, "TMEM columns");

// Non-blocking probe: has phase `parity` of the barrier completed?
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared-memory matrix descriptor without swizzling (core matrices of 8
// rows x 16 bytes; lbo / sbo: byte distance between core matrices along K /
// along M or N; descriptor version 1, layout type 0).
__device__ __forceinline__ uint64_t smem_desc_noswizzle(uint32_t saddr, uint32_t lbo_bytes,
                                                        uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3fff);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3fff) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3fff) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

// fp16 pair (1152 + z, 1152 + z): what 1024 + (code ^ 0x80) = 1152 + code
// must lose to leave code - z exactly
__device__ __forceinline__ uint32_t zp_bias(int z) {
    const __half h = __int2half_rn(1152 + z);
    return (uint32_t)__half_as_ushort(h) * 0x10001u;
}

// smallest e with 2^e >= x, for a positive finite x (x = 0 gives -126)
__device__ __forceinline__ int ceil_log2(float x) {
    const uint32_t b = __float_as_uint(x);
    const int e = (int)((b >> 23) & 0xff) - 127;
    if (e < -126) return -126;
    return (b & 0x7fffff) ? e + 1 : e;
}
__device__ __forceinline__ float exp2i(int e) {   // 2^e for e in [-126, 127]
    e = max(-126, min(127, e));
    return __uint_as_float((uint32_t)(e + 127) << 23);
}

// byte offset of 16-byte chunk c (0..7) of row `row` in a 128-byte-wide,
// 128-byte-swizzled matrix (8-row atoms of 1024 bytes)
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return row * 128 + ((c ^ (row & 7)) << 4);
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}
__device__ __forceinline__ void sts16(uint32_t a, unsigned short v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(v) : "memory");
}

// Named barrier over `n` threads that also ORs a predicate across them.
__device__ __forceinline__ bool bar_red_or(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Column maxima of a warp's 32 x 32 values (lane = row, v[j] = column j):
// five exchange rounds halve the columns a lane keeps, so that lane l ends
// with the maximum of column l over all 32 lanes.
__device__ __forceinline__ float colmax32(float (&v)[32], int lane) {
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) {
        const bool hi = (lane & k) != 0;
#pragma unroll
        for (int i = 0; i < k; ++i) {
            const float send = hi ? v[i] : v[i + k];
            const float keep = hi ? v[i + k] : v[i];
            v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, k));
        }
    }
    return v[0];
}

struct Extra {
    const float* k_scale;   // [num_blocks][num_kv_heads][16]
    const float* v_scale;
    const int8_t* k_zp;
    const int8_t* v_zp;
};

// Shares balanced by cost, not by blocks. The blocks of a segment
// (sequence, kv head, row chunk) cost block_cost(rows) units each -- a tile's
// softmax grows with its rows -- and a segment's start costs kSegCost more
// (its epilogue, the next Q and the exact maxima of its first tile come to
// about two 32-row tiles). Segments are laid out as in the balanced schedule
// (sequence, then kv head, then chunk); the total B of units is cut into W
// equal ranges, and a block belongs to the share whose range holds its first
// unit. Every share holds at least kMinShareUnits units, so every share
// holds the first unit of some block.
constexpr int kSegCost = 48;
constexpr int kMinShareUnits = kSegCost + 8 * 5;
__host__ __device__ __forceinline__ int block_cost(int rows) { return 2 + ((rows + 31) >> 5); }

__device__ __forceinline__ int chunk_rows(const pa::sched::Params& p, int r, int c) {
    return min(kRT, p.group * r - c * kRT);
}

// units of chunk c of a sequence (L tokens, query run r); its blocks in *nbs
__device__ __forceinline__ int seg_units(const pa::sched::Params& p, int L, int r, int c, int* nbs) {
    *nbs = pa::sched::chunk_blocks(p, L, r, 0, c);
    return *nbs > 0 ? kSegCost + *nbs * block_cost(chunk_rows(p, r, c)) : 0;
}

__device__ __forceinline__ int seq_units(const pa::sched::Params& p, int s, int C) {
    int q0, nbs, u = 0;
    const int L = __ldg(p.context_lens + s), r = pa::sched::query_run(p.qsl, s, &q0);
    for (int c = 0; c < C; ++c) u += seg_units(p, L, r, c, &nbs);
    return u;
}

// cum[s] = units of the sequences before s (every kv head), chunks[s] = C_s,
// by one CTA (a block-wide scan); CTA 0 copies cum for the reduce kernel.
__device__ void build_cost_prefix(int32_t* cum, uint8_t* chunks, const pa::sched::Params& p) {
    __shared__ int32_t warp_tot[32];
    pa::grid_dependents_launch();   // the reduce kernel may be scheduled early
    pa::grid_dependency_wait();     // inputs written by the previous kernel are visible
    const int n = p.num_seqs;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (n + nt - 1) / nt;
    const int a = min(n, tid * per), b = min(n, a + per);
    int32_t local = 0;
    for (int i = a; i < b; ++i) {
        const int c = pa::sched::chunks_of(p, i);
        chunks[i] = (uint8_t)c;
        local += p.num_kv_heads * seq_units(p, i, c);
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
        run += p.num_kv_heads * seq_units(p, i, chunks[i]);
    }
    if (tid == nt - 1) cum[n] = run;
    __syncthreads();
    if (blockIdx.x == 0 && p.cum_out)
        for (int i = tid; i <= n; i += nt) p.cum_out[i] = cum[i];
}

// The tiles of a share in order: up to 8 blocks at a time of the current
// segment, never past the segment's end or the share's last block. Every
// role walks its own copy.
struct Cursor {
    Pos cur;            // sequence, kv head, chunk, block, blocks, chunks of the sequence
    int64_t u0;         // first unit of the segment (its block 0)
    int w;              // units per block of the segment
    int64_t f1;         // end of the share's units
    int lim;            // blocks of the segment in this share or before it
    bool done, cut;     // past the share's last block; its last segment continues after it
    int seg_b0;         // the segment's block where this share's piece starts
    bool seg_first;     // the piece is the share's first
    int L, r, q0, rows; // of the current segment

    __device__ __forceinline__ int64_t start(int bb) const {
        return bb == 0 ? u0 : u0 + kSegCost + (int64_t)bb * w;
    }
    // this segment's blocks whose first unit lies before f1
    __device__ __forceinline__ int limit() const {
        if (f1 <= u0) return 0;
        const int64_t over = f1 - u0 - kSegCost;   // start(bb) < f1 <=> bb * w < over (bb >= 1)
        const int64_t more = over > 0 ? (over + w - 1) / w - 1 : 0;
        return (int)min((int64_t)cur.nbs, 1 + max((int64_t)0, more));
    }
    __device__ __forceinline__ void load(const pa::sched::Params& p) {
        L = __ldg(p.context_lens + cur.s);
        r = pa::sched::query_run(p.qsl, cur.s, &q0);
        rows = chunk_rows(p, r, cur.c);
        w = block_cost(rows);
    }
    // from segment (s, g, c) starting at unit u, the first one with blocks;
    // false past the last sequence
    __device__ bool settle(const pa::sched::Params& p, const uint8_t* chunks) {
        for (;;) {
            int q0_, nbs;
            const int Ls = __ldg(p.context_lens + cur.s);
            const int rs = pa::sched::query_run(p.qsl, cur.s, &q0_);
            seg_units(p, Ls, rs, cur.c, &nbs);
            if (nbs > 0) {
                cur.nbs = nbs;
                load(p);
                return true;
            }
            if (++cur.c >= cur.C) {
                cur.c = 0;
                if (++cur.g >= p.num_kv_heads) {
                    cur.g = 0;
                    if (++cur.s >= p.num_seqs) return false;
                    cur.C = chunks[cur.s];
                }
            }
        }
    }
    __device__ void init(const pa::sched::Params& p, const int32_t* cum, const uint8_t* chunks,
                         int64_t fa, int64_t fb) {
        f1 = fb;
        done = cut = false;
        seg_first = true;
        // the sequence holding unit fa, then its kv head and chunk
        int lo = 0, hi = p.num_seqs;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cum[mid] <= fa) lo = mid;
            else hi = mid;
        }
        cur.s = lo;
        cur.C = chunks[lo];
        const int64_t span = (cum[lo + 1] - cum[lo]) / p.num_kv_heads;
        cur.g = (int)((fa - cum[lo]) / span);
        u0 = cum[lo] + (int64_t)cur.g * span;
        int q0_, nbs;
        const int Ls = __ldg(p.context_lens + lo), rs = pa::sched::query_run(p.qsl, lo, &q0_);
        for (cur.c = 0; cur.c < cur.C; ++cur.c) {
            const int un = seg_units(p, Ls, rs, cur.c, &nbs);
            if (fa < u0 + un) break;
            u0 += un;
        }
        cur.nbs = nbs;
        load(p);
        // the first block whose first unit is at or after fa
        const int64_t rem = fa - u0;
        int b0 = 0;
        if (rem > 0) b0 = (int)max((int64_t)1, (rem - kSegCost + w - 1) / w);
        if (b0 >= cur.nbs) {
            u0 += kSegCost + (int64_t)cur.nbs * w;
            cur.b = 0;
            if (++cur.c >= cur.C) {
                cur.c = 0;
                if (++cur.g >= p.num_kv_heads) {
                    cur.g = 0;
                    if (++cur.s >= p.num_seqs) {
                        done = true;
                        return;
                    }
                    cur.C = chunks[cur.s];
                }
            }
            if (!settle(p, chunks)) {
                done = true;
                return;
            }
            b0 = 0;
        }
        cur.b = b0;
        seg_b0 = b0;
        lim = limit();
        done = cur.b >= lim;
    }
    __device__ __forceinline__ bool more() const { return !done; }
    __device__ __forceinline__ int blocks() const { return min(kTileBlocks, lim - cur.b); }
    __device__ __forceinline__ bool piece_first() const { return cur.b == seg_b0; }
    __device__ __forceinline__ bool piece_last(int nb) const { return cur.b + nb == lim; }
    __device__ __forceinline__ int cols() const { return (rows + 31) & ~31; }   // MMA N
    __device__ void advance(const pa::sched::Params& p, const int32_t* cum, const uint8_t* chunks,
                            int nb) {
        cur.b += nb;
        if (cur.b < lim) return;
        if (lim < cur.nbs) {            // the segment continues in the next share
            done = cut = true;
            return;
        }
        // the next segment with blocks, if it starts in this share
        const int64_t next_u0 = u0 + kSegCost + (int64_t)cur.nbs * w;
        const Pos keep = cur;
        if (++cur.c >= cur.C) {
            cur.c = 0;
            if (++cur.g >= p.num_kv_heads) {
                cur.g = 0;
                if (++cur.s >= p.num_seqs) {
                    cur = keep;
                    done = true;
                    return;
                }
                cur.C = chunks[cur.s];
            }
        }
        if (next_u0 >= f1 || !settle(p, chunks)) {
            cur = keep;
            done = true;
            return;
        }
        u0 = next_u0;
        cur.b = 0;
        seg_b0 = 0;
        seg_first = false;
        lim = limit();
    }
};

template <typename TQ>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_int8_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                const __grid_constant__ CUtensorMap tmap_v,
                                const pa::sched::Params p, const Extra x) {
    namespace tc = pa::tc;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = pa::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bars = base + kBarOff;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(smem + kBarOff + 8 * kNumBars);
    int32_t* const cum = reinterpret_cast<int32_t*>(smem + kHdrOff);
    uint8_t* const chunks = reinterpret_cast<uint8_t*>(cum + p.num_seqs + 1);

    build_cost_prefix(cum, chunks, p);             // every thread; waits for the previous kernel
    const int64_t B = cum[p.num_seqs];
    const int64_t wid = blockIdx.x;
    const int64_t W = max((int64_t)1, min((int64_t)p.workers, B / kMinShareUnits));
    const int64_t f0 = pa::sched::share_start(wid, B, W);
    const int64_t f1 = pa::sched::share_start(wid + 1, B, W);
    if (threadIdx.x == 0) pa::sched::write_merge_record(p, wid, 0, 0, 0);   // none unless set later
    if (wid >= W || f1 <= f0) return;              // uniform over the CTA

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            // arrivals: one per converter or softmax warp, else the producer or a commit
            const bool four = (i >= kKReady && i < kSFull) || (i >= kSFree && i < kODone) ||
                              i == kOFree;
            pa::mbar_init(bar(i), four ? 4 : 1);
        }
        pa::fence_barrier_init();
        pa::prefetch_tensormap(&tmap_k);
        pa::prefetch_tensormap(&tmap_v);
    }
    if (warp == 9) {
        tc::tmem_alloc(pa::smem_addr(tmem_holder), kTmemCols);
        tc::tmem_relinquish();
    }
    // the all-ones A operand of the denominator products (fp16 1.0 = 0x3C00)
    for (int i = threadIdx.x; i < 4096 / 16; i += kThreads)
        sts128(base + kOnesOff + 16 * i, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    const int G = p.group;
    auto wait_w = [&](uint32_t b, uint32_t parity, unsigned int code) -> bool {
        return __all_sync(0xffffffffu, pa::mbar_wait(b, parity, p.err, code));
    };

    if (warp == 0) {
        // ---------------- producer: the code tiles ----------------
        Cursor it;
        it.init(p, cum, chunks, f0, f1);
        const uint64_t pol_once = pa::policy_evict_first(), pol_again = pa::policy_evict_normal();
        int u = 0;
        bool ok = true;
        for (; it.more(); ++u) {
            const int nb = it.blocks();
            const int st = u % kStages;
            // the tile's block ids load while the stage is waited for
            int tile = 0;
            if (lane < nb) {
                int blk = __ldg(p.block_tables + (int64_t)it.cur.s * p.max_blocks + it.cur.b + lane);
                if (blk < 0 || blk >= p.num_blocks) {
                    if (p.err) atomicOr(p.err, pa::ERR_BAD_BLOCK);
                    blk = 0;
                }
                tile = blk * p.num_kv_heads + it.cur.g;
            }
            if (u >= kStages &&
                !(ok = wait_w(bar(kEmpty + st), ((u / kStages) - 1) & 1, pa::ERR_WAIT_EMPTY)))
                break;
            const uint32_t full = bar(kFull + st), sb = base + st * kStageBytes;
            if (lane == 0) pa::mbar_arrive_expect_tx(full, nb * (2 * kBS * D));
            __syncwarp();
            if (lane < nb) {
                // later row chunks of the sequence read these blocks again: keep them in L2
                const uint64_t pol = it.cur.C == 1 ? pol_once : pol_again;
                pa::tma_load_2d(sb + lane * (kBS * D), &tmap_k, 0, tile * kBS, full, pol);
                pa::tma_load_2d(sb + kCodes + lane * (kBS * D), &tmap_v, 0, tile * kBS, full, pol);
            }
            it.advance(p, cum, chunks, nb);
        }
        if (lane == 0) {
            // no copy may be in flight when the CTA ends: the last tile of each stage
            for (int k = max(0, u - kStages); k < u; ++k)
                if (!pa::mbar_wait(bar(kFull + k % kStages), (k / kStages) & 1, nullptr, 0)) {
                    if (p.err) atomicOr(p.err, pa::ERR_WAIT_DRAIN);
                    break;
                }
            // a segment cut by this share's end and started in it: this CTA
            // owns its merge, up to the share holding its last block
            if (ok && it.cut && it.seg_b0 == 0)
                pa::sched::write_merge_record(p, wid, 1,
                                              pa::sched::share_of(it.start(it.cur.nbs - 1), B, W),
                                              it.seg_first ? 0 : 1, it.q0, it.rows);
        }
    } else if (warp <= 4) {
        // ---------------- converters: one token per thread ----------------
        const int q4 = warp & 3, t = 32 * q4 + lane;
        const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
        float* const vmax = reinterpret_cast<float*>(smem + kRedOff);   // [2][4]
        const TQ* const qg = static_cast<const TQ*>(p.q);
        Cursor it;
        it.init(p, cum, chunks, f0, f1);
        int ev = -126;            // log2 of the piece's V reference
        float rm_row = 0.f;       // row scale of Q row t of the piece (base-2 softmax units)
        // Scales and zero points of token t of a tile, by plain loads: its
        // block id (through the block table) two tiles ahead, its values one
        // tile ahead, so that neither load is waited for.
        Cursor la = it;          // the tile after the current one
        int nb1 = 0, blk1 = 0;   // blocks of that tile; token t's block in it
        float ks_n = 0.f, vs_n = 0.f;
        int kz_n = 0, vz_n = 0;
        auto block_of = [&](const Cursor& c, int nbc) {
            int blk = 0;
            if (t < nbc * kBS) {
                blk = __ldg(p.block_tables + (int64_t)c.cur.s * p.max_blocks + c.cur.b + (t >> 4));
                if (blk < 0 || blk >= p.num_blocks) blk = 0;   // reported by the producer
            }
            return blk;
        };
        auto values = [&](const Cursor& c, int nbc, int blk) {
            if (t < nbc * kBS) {
                const int64_t e = ((int64_t)blk * p.num_kv_heads + c.cur.g) * kBS + (t & 15);
                ks_n = __ldg(x.k_scale + e);
                vs_n = __ldg(x.v_scale + e);
                kz_n = __ldg(x.k_zp + e);
                vz_n = __ldg(x.v_zp + e);
            }
        };
        values(it, it.blocks(), block_of(it, it.blocks()));
        la.advance(p, cum, chunks, it.blocks());
        if (la.more()) {
            nb1 = la.blocks();
            blk1 = block_of(la, nb1);
        }
        for (int u = 0; it.more(); ++u) {
            const int nb = it.blocks();
            const bool first = it.piece_first();
            const int st = u % kStages, b = u & 1;
            const uint32_t sb = base + st * kStageBytes;
            float ks = ks_n, vs = vs_n;
            const int kz = kz_n, vz = vz_n;
            if (la.more()) {
                values(la, nb1, blk1);                   // tile u + 1
                la.advance(p, cum, chunks, nb1);
                if (la.more()) {
                    nb1 = la.blocks();
                    blk1 = block_of(la, nb1);            // tile u + 2
                }
            }
            wait_w(bar(kFull + st), (u / kStages) & 1, pa::ERR_WAIT_FULL);
            const int tok0 = it.cur.b * kBS;
            const bool valid = t < nb * kBS && tok0 + t < it.L;
            // scales past the context or the tile may hold anything: their weights must be 0
            ks = valid ? ks : 0.f;
            vs = valid && vs > 0.f ? vs : 0.f;
            const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(vs));
            if (lane == 0) vmax[4 * b + q4] = __uint_as_float(wm);
            // info entry b and Kc buffer b are free once the softmax is done with tile u - 2
            if (u >= 2) wait_w(bar(kInfoFree + b), ((u >> 1) - 1) & 1, pa::ERR_WAIT_EMPTY);
            if (first) {
                ev = -126;
                // Q of a new piece: the previous tile's S product must be done reading Q
                if (u >= 1) wait_w(bar(kSFull + ((u - 1) & 1)), ((u - 1) >> 1) & 1, pa::ERR_WAIT_FULL);
                const int rows = it.rows, N = it.cols();
                rm_row = 0.f;
                if (t < N) {
                    uint4 qv[16];
                    float mx = 0.f;
                    if (t < rows) {
                        const int gr = it.cur.c * kRT + t;
                        const uint4* src = reinterpret_cast<const uint4*>(
                            qg + ((int64_t)(it.q0 + gr / G) * p.num_heads + it.cur.g * G + gr % G) * D);
#pragma unroll
                        for (int i = 0; i < 16; ++i) qv[i] = __ldg(src + i);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const TQ* e = reinterpret_cast<const TQ*>(&qv[i]);
#pragma unroll
                            for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fabsf((float)e[k]));
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) qv[i] = make_uint4(0, 0, 0, 0);
                    }
                    int ex = 0;
                    if (mx > 0.f) {
                        ex = (int)((__float_as_uint(mx) >> 23) & 0xff) - 127;   // floor(log2 max|q|)
                        ex = max(-100, min(100, ex));
                    }
                    const float up = exp2i(14 - ex);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const TQ* e = reinterpret_cast<const TQ*>(&qv[i]);
                        uint32_t h[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            __half2 v2 = __floats2half2_rn((float)e[2 * k] * up, (float)e[2 * k + 1] * up);
                            h[k] = *reinterpret_cast<uint32_t*>(&v2);
                        }
                        sts128(base + kQOff + (i >> 3) * kHalfQ + sw128(t, i & 7), h[0], h[1], h[2],
                               h[3]);
                    }
                    rm_row = t < rows ? p.scale_log2 * exp2i(ex - 14) : 0.f;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tc::fence_after_sync();
            {
                // Kc = K codes - zp of token t, as fp16 pairs, into TMEM lane t
                // (16 dims, 8 columns, per chunk)
                const uint32_t zb = zp_bias(kz);
#pragma unroll 2
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = lds128(sb + sw128(t, c));
                    const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
                    uint32_t w[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t u8 = cw[i] ^ 0x80808080u;
                        w[2 * i] = hsub2(prmt(u8, kMagic, 0x4140), zb);
                        w[2 * i + 1] = hsub2(prmt(u8, kMagic, 0x4342), zb);
                    }
                    tc::st_8cols_nowait(trow + kColK + 64 * b + 8 * c, w);
                }
                tc::wait_st();
            }
            pa::named_barrier_sync(1, 128);             // every converter warp's V-scale maximum
            const float tmax = fmaxf(fmaxf(vmax[4 * b], vmax[4 * b + 1]),
                                     fmaxf(vmax[4 * b + 2], vmax[4 * b + 3]));
            const int e_new = max(ev, ceil_log2(tmax));
            const float vfix = exp2i(ev - e_new);      // O's exact rescale to the new reference
            ev = e_new;
            float* const info = reinterpret_cast<float*>(smem + kInfoOff + b * kInfoBytes);
            info[t] = ks;
            if (t < kRT) info[kInfoRm + t] = rm_row;
            if (t == 0) {
                info[kInfoVfix] = vfix;
                info[kInfoVref] = exp2i(ev);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(bar(kKReady + b));
            // V' in place: dims 16c .. 16c + 15 of row t go to 16-byte chunks
            // 2c, 2c + 1 of half c / 4 -- half 0 over this thread's K code row
            // (converted above), half 1 (c >= 4) over code chunks 2c - 8 and
            // 2c - 7 of its V row, which earlier iterations (or this one) read
            {
                const uint32_t zb = zp_bias(vz);
                const __half2 f2 = __float2half2_rn(vs * exp2i(-ev));
                const uint32_t ff = *reinterpret_cast<const uint32_t*>(&f2);
                const uint32_t vrow = sb + t * 128;
#pragma unroll 2
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = lds128(sb + kCodes + sw128(t, c));
                    const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
                    uint32_t o[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t u8 = cw[i] ^ 0x80808080u;
                        o[2 * i] = hmul2(hsub2(prmt(u8, kMagic, 0x4140), zb), ff);
                        o[2 * i + 1] = hmul2(hsub2(prmt(u8, kMagic, 0x4342), zb), ff);
                    }
                    const uint32_t hb = vrow + (c >> 2) * kHalfV;
                    const int ch = (2 * c) & 7;
                    sts128(hb + ((ch ^ (t & 7)) << 4), o[0], o[1], o[2], o[3]);
                    sts128(hb + (((ch + 1) ^ (t & 7)) << 4), o[4], o[5], o[6], o[7]);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(bar(kVReady + st));
            it.advance(p, cum, chunks, nb);
        }
    } else if (warp <= 8) {
        // ---------------- softmax (one thread per token) and epilogue (one per dim) ----------------
        const int q4 = warp & 3, t = 32 * q4 + lane;
        const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
        float* const red = reinterpret_cast<float*>(smem + kRedOff + 64);   // [4][96] column maxima
        float* const mr = red + 4 * kRT;   // running max per column (-inf: none yet)
        float* const mu = mr + kRT;        // the max subtracted (-FLT_MAX while mr is -inf)
        float* const alpha = mu + kRT;     // rescale of a column when its max moved
        int32_t* const bnd = reinterpret_cast<int32_t*>(alpha + kRT);   // last key of each column
        float* const zero = alpha + 2 * kRT;                          // a zero offset per column
        if (t < kRT) zero[t] = 0.f;        // read after the first tile's group barrier
        // epilogue tables over the column-maximum area (free then): 1 / l, output row
        float* const inv_l = red;
        int32_t* const orow = reinterpret_cast<int32_t*>(red + kRT);
        Cursor it;
        it.init(p, cum, chunks, f0, f1);
        for (int u = 0; it.more(); ++u) {
            const int nb = it.blocks();
            const bool first = it.piece_first(), last = it.piece_last(nb);
            const int b = u & 1;
            const int rows = it.rows, nch = it.cols() >> 5;
            const int tok0 = it.cur.b * kBS;
            wait_w(bar(kSFull + b), (u >> 1) & 1, pa::ERR_WAIT_FULL);
            wait_w(bar(kKReady + b), (u >> 1) & 1, pa::ERR_WAIT_FULL);
            tc::fence_after_sync();
            const float* const info = reinterpret_cast<const float*>(smem + kInfoOff + b * kInfoBytes);
            const float ks = info[t], vfix = info[kInfoVfix], vref = info[kInfoVref];
            const bool tvalid = t < nb * kBS && tok0 + t < it.L;
            const int last_q = it.L - it.r, row_off = it.cur.c * kRT;
            // Masks: a token past the context or the tile is past every bound;
            // a key past a verify row's bound (row j of the chunk sees keys up to
            // last_q + (row_off + j) / G, kept per column for the piece).
            const bool mask = !(nb == kTileBlocks && tok0 + kTok <= it.L) ||
                              tok0 + kTok - 1 > last_q + row_off / G;
            const int pos = tvalid ? tok0 + t : 0x7fffffff;
            if (first) {
                if (t < kRT)
                    bnd[t] = t < rows ? min(last_q + (row_off + t) / G, it.L - 1) : it.L - 1;
                pa::named_barrier_sync(2, 128);
            }
            const uint32_t s_tm = trow + kColS + kRT * b;
            // e[j] = S * ks * rm[j] - off[j] over columns 32c .. 32c + 31 (masked: -inf)
            auto scores = [&](int c, float (&e)[32], const float* off) {
                tc::ld_32cols(s_tm + 32 * c, e);
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 rm = *reinterpret_cast<const float4*>(info + kInfoRm + 32 * c + j);
                    const float4 of = *reinterpret_cast<const float4*>(off + 32 * c + j);
                    e[j] = fmaf(e[j] * ks, rm.x, -of.x);
                    e[j + 1] = fmaf(e[j + 1] * ks, rm.y, -of.y);
                    e[j + 2] = fmaf(e[j + 2] * ks, rm.z, -of.z);
                    e[j + 3] = fmaf(e[j + 3] * ks, rm.w, -of.w);
                }
                if (mask) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const int4 bd = *reinterpret_cast<const int4*>(bnd + 32 * c + j);
                        if (pos > bd.x) e[j] = -INFINITY;
                        if (pos > bd.y) e[j + 1] = -INFINITY;
                        if (pos > bd.z) e[j + 2] = -INFINITY;
                        if (pos > bd.w) e[j + 3] = -INFINITY;
                    }
                }
            };
            // P of chunk c as fp16: row j of P holds token t at column t
            const uint32_t pbuf = base + kPOff + b * kPBuf + (t >> 6) * kHalfQ + (t & 7) * 2;
            const int tcol = (t & 63) >> 3;
            auto pack_p = [&](const float (&e)[32], uint32_t (&q)[16]) {
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    __half2 h2 = __floats2half2_rn(pa::ex2(e[j]), pa::ex2(e[j + 1]));
                    q[j >> 1] = *reinterpret_cast<uint32_t*>(&h2);
                }
            };
            int pc = 0;   // the chunk store_packed writes
            auto store_packed = [&](const uint32_t (&q)[16]) {
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const uint32_t r0 = pbuf + (32 * pc + j) * 128;
                    sts16(r0 + ((tcol ^ (j & 7)) << 4), (unsigned short)(q[j >> 1] & 0xffff));
                    sts16(r0 + 128 + ((tcol ^ ((j + 1) & 7)) << 4), (unsigned short)(q[j >> 1] >> 16));
                }
                ++pc;
            };
            // Three passes over the scores, one code path: (0) against the
            // running max -- a score more than 2^8 above its column's max, or
            // any score of a column without one (offset -FLT_MAX), calls for
            // (1) the tile's exact column maxima (always on a piece's first
            // tile), by exchange within a warp and then over the four warps;
            // (2) P = 2^(s - max) into its buffer.
            bool any = first, kept = false;
            uint32_t pk[16];   // P of chunk c as fp16 pairs (columns 2i, 2i + 1)
#pragma unroll 1
            for (int pass = first ? 1 : 0; pass < 3; ++pass) {
                if (pass == 1 && !any) continue;                 // uniform over the group
                if (pass == 2) {
                    if (!first && (any || vfix != 1.f)) {
                        // O and l move to the new maxima and V reference once tile
                        // u - 1's products are done
                        wait_w(bar(kODone + (b ^ 1)), ((u - 1) >> 1) & 1, pa::ERR_WAIT_FULL);
                        tc::fence_after_sync();
                        for (int c = 0; c < nch; ++c) {
                            float ov[32], lv[32];
                            tc::ld_32cols(trow + kColO + 32 * c, ov);
                            tc::ld_32cols(trow + kColL + 32 * c, lv);
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const float al = any ? alpha[32 * c + j] : 1.f;
                                ov[j] *= al * vfix;
                                lv[j] *= al;
                            }
                            tc::st_32cols(trow + kColO + 32 * c, ov);
                            tc::st_32cols(trow + kColL + 32 * c, lv);
                        }
                    }
                    // P buffer b is free once tile u - 2's products are done
                    if (u >= 2) wait_w(bar(kODone + b), ((u >> 1) - 1) & 1, pa::ERR_WAIT_FULL);
                }
                float mx = -INFINITY;
                for (int c = 0; c < nch; ++c) {
                    if (pass == 2 && kept) {   // P of the single chunk, from pass 0
                        store_packed(pk);
                        break;
                    }
                    float e[32];
                    scores(c, e, pass == 1 ? zero : mu);
                    if (pass == 0) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, e[j]);
                        if (nch == 1) pack_p(e, pk);
                    } else if (pass == 1) {
                        red[q4 * kRT + 32 * c + lane] = colmax32(e, lane);
                    } else {
                        pack_p(e, pk);
                        store_packed(pk);
                    }
                }
                if (pass == 0) {
                    any = bar_red_or(2, 128, mx > kLazyMax);
                    kept = nch == 1 && !any;
                } else if (pass == 1) {
                    pa::named_barrier_sync(2, 128);
                    if (t < 32 * nch) {
                        const float cm = fmaxf(fmaxf(red[t], red[kRT + t]),
                                               fmaxf(red[2 * kRT + t], red[3 * kRT + t]));
                        const float mo = first ? -INFINITY : mr[t];
                        const float mn = fmaxf(mo, cm);
                        alpha[t] = mo == -INFINITY ? 0.f : pa::ex2(mo - mn);
                        mr[t] = mn;
                        mu[t] = mn == -INFINITY ? -FLT_MAX : mn;
                    }
                    pa::named_barrier_sync(2, 128);
                }
            }
            tc::fence_before_sync();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                pa::mbar_arrive(bar(kSFree + b));
                pa::mbar_arrive(bar(kInfoFree + b));
                pa::mbar_arrive(bar(kPFull + b));
            }
            if (last) {
                // ---- epilogue of the piece: thread t holds dim t of every row ----
                wait_w(bar(kODone + b), (u >> 1) & 1, pa::ERR_WAIT_FULL);
                tc::fence_after_sync();
                const bool complete = it.seg_b0 == 0 && it.cur.b + nb == it.cur.nbs;   // whole segment
                pa::sched::Slot sl(p.slots + (2 * wid + (it.seg_first ? 0 : 1)) * (int64_t)p.slot_bytes,
                                   kRT);
                if (32 * q4 < rows) {                      // warp-uniform (a TMEM load)
                    // this thread's own column t: l (every lane of l holds it)
                    float lv[32];
                    tc::ld_32cols(trow + kColL + 32 * q4, lv);
                    float l_own = lv[0];
#pragma unroll
                    for (int j = 1; j < 32; ++j) l_own = lane == j ? lv[j] : l_own;
                    if (t < rows && complete) {
                        const int gr = row_off + t, qi = gr / G;
                        inv_l[t] = __fdividef(vref, l_own);
                        orow[t] = (it.q0 + qi) * p.num_heads + it.cur.g * G + (gr - qi * G);
                    } else if (t < rows) {
                        sl.l[t] = l_own;
                        sl.m[t] = mr[t];
                    }
                }
                if (!complete && t == 0) {
                    sl.hdr[0] = it.cur.s;
                    sl.hdr[1] = it.cur.g;
                    sl.hdr[2] = it.cur.c;
                    sl.hdr[3] = it.seg_b0 * kBS;
                    sl.hdr[4] = min((it.cur.b + nb) * kBS, it.L);
                }
                pa::named_barrier_sync(2, 128);
                for (int c = 0; c < nch; ++c) {
                    float ov[32];
                    tc::ld_32cols(trow + kColO + 32 * c, ov);
                    const int n = min(32, rows - 32 * c);        // rows of this chunk
                    if (!complete) {
                        float* dst = sl.o + (int64_t)(32 * c) * D + t;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < n) dst[(int64_t)j * D] = ov[j] * vref;
                    } else if (p.out_f32) {
                        float* dst = static_cast<float*>(p.out) + t;
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            if (j >= n) break;
                            const float4 il = *reinterpret_cast<const float4*>(inv_l + 32 * c + j);
                            const int4 orw = *reinterpret_cast<const int4*>(orow + 32 * c + j);
                            dst[(int64_t)orw.x * D] = ov[j] * il.x;
                            if (j + 1 < n) dst[(int64_t)orw.y * D] = ov[j + 1] * il.y;
                            if (j + 2 < n) dst[(int64_t)orw.z * D] = ov[j + 2] * il.z;
                            if (j + 3 < n) dst[(int64_t)orw.w * D] = ov[j + 3] * il.w;
                        }
                    } else {
                        TQ* dst = static_cast<TQ*>(p.out) + t;
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {
                            if (j >= n) break;
                            const float4 il = *reinterpret_cast<const float4*>(inv_l + 32 * c + j);
                            const int4 orw = *reinterpret_cast<const int4*>(orow + 32 * c + j);
                            dst[(int64_t)orw.x * D] = (TQ)(ov[j] * il.x);
                            if (j + 1 < n) dst[(int64_t)orw.y * D] = (TQ)(ov[j + 1] * il.y);
                            if (j + 2 < n) dst[(int64_t)orw.z * D] = (TQ)(ov[j + 2] * il.z);
                            if (j + 3 < n) dst[(int64_t)orw.w * D] = (TQ)(ov[j + 3] * il.w);
                        }
                    }
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) pa::mbar_arrive(bar(kOFree));
            }
            it.advance(p, cum, chunks, nb);
        }
    } else {
        // ---------------- MMA issue (one elected lane) ----------------
        // Whichever product is ready goes first: S of the next tile needs its
        // Kc (and a free S buffer), the O and l products of the oldest tile
        // its P and V' (and, at a piece's start, the previous piece's
        // epilogue done with O and l).
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        const uint32_t sbase = __shfl_sync(0xffffffffu, base, 0);
        const uint64_t dq = tc::smem_desc_sw128(sbase + kQOff, 16, 1024);
        const uint64_t dp0 = tc::smem_desc_sw128(sbase + kPOff, 16, 1024);
        const uint64_t dv0 = tc::smem_desc_sw128(sbase, kHalfV, 1024);   // V' of stage 0
        const uint64_t d1 = smem_desc_noswizzle(sbase + kOnesOff, 128, 256);
        // a descriptor of address a + o is the one of a plus o >> 4; K steps of 16
        // dims (Q) or tokens (P) within and across the two 64-wide halves
        auto koff = [](int kk) { return (uint64_t)((((kk >> 2) * kHalfQ) + (kk & 3) * 32) >> 4); };
        Cursor cs, cp;   // the tile of the next S product; the tile of the next O, l products
        cs.init(p, cum, chunks, f0, f1);
        cp.init(p, cum, chunks, f0, f1);
        int us = 0, up = 0, piece = -1;
        bool ok = true;
        uint64_t t_idle = 0;
        uint32_t idle = 0;
        while (ok && cp.more()) {
            bool did = false;
            if (cs.more()) {
                const int b = us & 1;
                const bool rdy = __all_sync(
                    0xffffffffu, mbar_test_wait(bar(kKReady + b), (us >> 1) & 1) &&
                                     (us < 2 || mbar_test_wait(bar(kSFree + b), ((us >> 1) - 1) & 1)));
                if (rdy) {
                    // S^T[b] = Kc(us) Q^T
                    tc::fence_after_sync();
                    const uint32_t idesc = tc::idesc_f16(false, false, false, kTok, cs.cols());
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        tc::mma_f16_ts_warp(tm + kColS + kRT * b, tm + kColK + 64 * b + 8 * kk,
                                            dq + koff(kk), idesc, kk > 0 ? 1u : 0u);
                    tc::commit_warp(bar(kSFull + b));
                    cs.advance(p, cum, chunks, cs.blocks());
                    ++us;
                    did = true;
                }
            }
            {
                const int b = up & 1;
                const bool first = cp.piece_first();
                const bool rdy = __all_sync(
                    0xffffffffu, mbar_test_wait(bar(kPFull + b), (up >> 1) & 1) &&
                                     mbar_test_wait(bar(kVReady + up % kStages),
                                                        (up / kStages) & 1) &&
                                     (!first || piece < 0 || mbar_test_wait(bar(kOFree), piece & 1)));
                if (rdy) {
                    // O^T += V'^T P^T and l += 1 P^T over the tile's blocks
                    if (first) ++piece;
                    tc::fence_after_sync();
                    const int nb = cp.blocks(), n = cp.cols();
                    const uint32_t ipv = tc::idesc_f16(false, true, false, kTok, n);
                    const uint32_t il = tc::idesc_f16(false, false, false, kTok, n);
                    const uint64_t dv = dv0 + (uint64_t)(((up % kStages) * kStageBytes) >> 4);
                    const uint64_t dp = dp0 + (uint64_t)((b * kPBuf) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTileBlocks; ++kk) {
                        if (kk < nb) {   // one 16-token block per K step
                            const uint32_t acc = (kk > 0 || !first) ? 1u : 0u;
                            tc::mma_f16_ss_warp(tm + kColO, dv + (uint64_t)((kk * kBS * 128) >> 4),
                                                dp + koff(kk), ipv, acc);
                            tc::mma_f16_ss_warp(tm + kColL, d1, dp + koff(kk), il, acc);
                        }
                    }
                    tc::commit_warp(bar(kODone + b));
                    tc::commit_warp(bar(kEmpty + up % kStages));
                    cp.advance(p, cum, chunks, nb);
                    ++up;
                    did = true;
                }
            }
            if (did) {
                idle = 0;
            } else if ((++idle & 63u) == 1u) {
                // bounded: give up after the wait limit without progress, or at
                // once when another wait has given up
                const uint64_t now = pa::global_timer_ns();
                if (idle == 1u) t_idle = now;
                const bool stop = (p.err && (*reinterpret_cast<volatile unsigned int*>(p.err) &
                                             pa::kAbortMask)) ||
                                  now - t_idle > pa::kWaitNs;
                if (__any_sync(0xffffffffu, stop)) {
                    if (lane == 0 && p.err) atomicOr(p.err, pa::ERR_WAIT_FULL);
                    ok = false;
                }
            } else {
                __nanosleep(32);
            }
        }
        // every product this warp issued has finished before TMEM is freed
        tc::commit_warp(bar(kFin));
        if (!__all_sync(0xffffffffu, pa::mbar_wait(bar(kFin), 0, nullptr, 0)) && lane == 0 && p.err)
            atomicOr(p.err, pa::ERR_WAIT_DRAIN);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 9) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <typename TQ>
pa_status launch_tc(const pa::DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                    pa::sched::Params prm, const Extra& x, int64_t rows) {
    auto kern = paged_decode_int8_tc_kernel<TQ>;
    auto smem_of = [](int n) {
        return kHdrOff + (((n + 1) * 4 + n) + 15) / 16 * 16 + 1024;
    };
    static bool attr_set = false;   // per instantiation; benign race (idempotent)
    if (!attr_set) {
        if (pa_status s = pa::cuda_status(
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem_of(kMaxSeqs)),
                "int8 tensor-core decode: set shared memory size"))
            return s;
        attr_set = true;
    }
    if (pa_status s = pa::cuda_status(
            pa::launch_pdl(kern, dim3((unsigned)prm.workers), dim3(kThreads),
                           (size_t)smem_of(a.num_seqs), a.stream, mk, mv, prm, x),
            "int8 tensor-core decode launch"))
        return s;
    const int max_chunks = (int)((rows + kRT - 1) / kRT);
    const int row_slots = (int)std::min<int64_t>(kRT, rows);
    return pa::cuda_status(
        pa::sched::launch_segment_reduce<TQ, D>(prm, max_chunks, row_slots, a.stream),
        "segment reduce launch");
}

}  // namespace

namespace pa {

// Calls whose query rows per KV head average at least 64 (G x query tokens
// / sequences): there one conversion of each code serves enough rows to
// outweigh the per-piece costs of the tensor-core pipeline; fewer rows (a
// decode step with occasional verify runs) stay with the per-warp kernel.
bool int8_tc_applies(const DecodeArgs& a) {
    const int64_t rows = (int64_t)(a.num_heads / a.num_kv_heads) * a.max_q_len;
    const int64_t avg_rows_x = (int64_t)(a.num_heads / a.num_kv_heads) * a.num_q_tokens;
    // the cost units of a call fit the schedule's 32-bit prefix sums
    const int64_t chunks = (rows + kRT - 1) / kRT;
    const int64_t units = (int64_t)a.num_seqs * a.num_kv_heads * chunks *
                          (kSegCost + (int64_t)(a.max_context_len + kBS - 1) / kBS * block_cost(kRT));
    return a.kv_dtype == PA_INT8 && a.head_dim == D && a.block_size == kBS && rows > 16 &&
           avg_rows_x >= 64 * (int64_t)a.num_seqs && units < 0x7fffffffll &&
           a.num_seqs <= kMaxSeqs && a.partition_size == 0 && !a.lse_out && !a.ctx_start &&
           a.slots != nullptr;
}

// INT8 decode with tokens in M on the tensor cores (see the top of this file).
pa_status launch_decode_int8_tc(const DecodeArgs& a) {
    if (pa_status s = balanced_check(a)) return s;
    if (((uintptr_t)a.k_scale | (uintptr_t)a.v_scale | (uintptr_t)a.k_zp | (uintptr_t)a.v_zp) % 16)
        return fail(PA_ERR_INVALID_ARG, "k_scale, v_scale, k_zp and v_zp must be 16-byte aligned");
    // the caller's workspace holds 2 x workers slots of shape.slot_bytes; this
    // kernel's slots hold 96 rows, so it runs at most as many shares as fit
    const BalancedShape shape = balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads, a.head_dim,
                                               a.max_q_len, a.max_context_len);
    const int64_t slot = sched::slot_bytes(kRT, D);
    int dev = 0, sms = 0;
    if (pa_status s = cuda_status(cudaGetDevice(&dev), "cudaGetDevice")) return s;
    if (pa_status s = cuda_status(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                                  "SM count"))
        return s;
    const int64_t fit = shape.workers * shape.slot_bytes / slot;
    const int64_t workers = std::min<int64_t>({(int64_t)sms, fit, (int64_t)kBalancedMaxWorkers});
    if (workers < 1) return fail(PA_ERR_UNSUPPORTED, "int8 decode: workspace holds no 96-row slot");
    CUtensorMap mk, mv;
    if (pa_status s = cache_tensor_map(&mk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 1))
        return s;
    if (pa_status s = cache_tensor_map(&mv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 1))
        return s;
    sched::Params b{};
    b.out = a.out;
    b.q = a.q;
    b.block_tables = a.block_tables;
    b.context_lens = a.context_lens;
    b.qsl = a.query_start_loc;
    b.cum_out = static_cast<int32_t*>(a.slots);
    b.slots = static_cast<uint8_t*>(a.slots) + shape.cum_bytes;
    b.err = device_error_word();
    b.max_blocks = a.max_blocks_per_seq;
    b.num_heads = a.num_heads;
    b.num_kv_heads = a.num_kv_heads;
    b.group = a.num_heads / a.num_kv_heads;
    b.num_seqs = a.num_seqs;
    b.num_blocks = a.num_blocks;
    b.workers = (int)workers;
    b.rows_per_tile = kRT;
    b.slot_bytes = (int)slot;
    b.scale_log2 = a.scale * 1.4426950408889634f;
    b.out_f32 = a.out_dtype == PA_F32;
    const Extra x{a.k_scale, a.v_scale, a.k_zp, a.v_zp};
    const int64_t rows = (int64_t)b.group * a.max_q_len;
    if (a.q_dtype == PA_BF16) return launch_tc<__nv_bfloat16>(a, mk, mv, b, x, rows);
    return launch_tc<__half>(a, mk, mv, b, x, rows);
}

}  // namespace pa
