// Paged prefill attention on the 5th-generation tensor cores (tcgen05, TMEM).
//
// A long query run (a prefill chunk, "大模型推理优化全攻略" / "LLM推理优化深度实战":
// chunked prefill) turns attention over the paged cache into a dense
// contraction: per KV head, G q heads x r query tokens against the
// sequence's keys, causally masked ("cs336 lecture 10": query i of a run of
// r at position L - r + i sees keys 0 .. L - r + i). A CTA takes 256 rows of
// one (sequence, kv head) as two Q tiles of 128 and streams the key range in
// tiles of 64 tokens (four 16-token blocks, gathered through the block table
// by TMA); per Q tile x:
//
//   S_x = Q_x K^T      tcgen05.mma M128 N64, A = Q_x, B = K (both K-major in
//                      shared memory, 128-byte swizzle), S_x in TMEM;
//   P_x = softmax(S_x) one warpgroup per Q tile, one thread per row: S read
//                      from TMEM into registers (after which the next product
//                      may overwrite it), fp32 online softmax with a running
//                      max moved only when a tile raises it by more than 2^8
//                      (O_x is then rescaled in TMEM), P written back to TMEM
//                      as two 16-bit parts P_hi + P_lo so the weights keep
//                      ~16 mantissa bits;
//   O_x += P_x V       tcgen05.mma M128 N128 with A = P_x read from TMEM and
//                      B = V (MN-major in shared memory: V's rows are tokens,
//                      the contraction index), O_x in TMEM for the whole range;
//   out = O_x / l      read from TMEM at the end.
//
// The MMA warp issues whichever product of either Q tile is ready (products
// of S first), so one group's softmax runs while the other's products do.
// Roles: warp 0 streams K/V tiles into a 4-stage ring (TMA), warps 1 and 10
// issue the MMAs of Q tile 0 and 1 (one elected lane each) and commit them to
// mbarriers, warps 2-5 and 6-9 are the softmax groups. Every wait is bounded; a wait that gives up stops the tile
// loop of every role, and the MMA thread waits for its own operations to
// finish before TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <math.h>
#include <stdlib.h>

#include <algorithm>

#include "pa_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace {

constexpr int kBS = 16;
constexpr int D = 128;
constexpr int kRows = 128;              // query rows per Q tile (MMA M)
constexpr int kQTiles = 2;              // Q tiles per CTA, one softmax warpgroup each
constexpr int kTaskRows = kRows * kQTiles;
constexpr int kTok = 64;                // keys per K/V tile (S columns)
constexpr int kTileBlocks = kTok / kBS; // 4
constexpr int kThreads = 96 + 128 * kQTiles;   // producer, 2 MMA warps, 2 softmax warpgroups
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyMax = 8.f;

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kQBytes = 32 * 1024;              // one Q tile: [2 sub][128 rows][128 B]
constexpr int kQOff = 0;
constexpr int kKVStage = 32 * 1024;             // a K/V stage: K 16 KB, V 16 KB
constexpr int kKBytes = 16 * 1024;              // [2 sub][64 rows][128 B]
constexpr int kSubKV = 8 * 1024;                // one 64-dim half of a K (or V) tile

// The two modes of the kernel. Prefill (kSplit false): two Q tiles of
// different rows over the same keys, each K/V tile read by both, a ring of
// 4 stages. Split keys (kSplit true, the prefix phase of shared-prefix
// decode): one Q tile of at most 128 rows whose two MMA / softmax pipelines
// take two different key chunks, each with its own 3 stages of the ring
// (the second Q tile's shared memory holds the extra stages).
template <bool kSplit>
struct TcLayout {
    static constexpr int kStages = kSplit ? 6 : 4;
    static constexpr int kPerTile = kSplit ? 3 : 4;     // stages a Q tile's stream cycles through
    static constexpr int kKVOff = (kSplit ? 1 : kQTiles) * kQBytes;
    static constexpr int kBarOff = kKVOff + kStages * kKVStage;   // mbarriers and flags
    static constexpr int kSmem = kBarOff + 256 + 1024;            // + alignment slack
    // barrier slots: K/V full and empty per stage; per (Q tile x, S buffer
    // b): S full and P full (index 2x + b); per Q tile: O done (one phase
    // per P V product) and the final commit of its MMA warp (one phase: every
    // product done, which the epilogue waits for); V rows past the context
    // zeroed (single use)
    static constexpr int kBarKVFull = 0, kBarKVEmpty = kStages, kBarSFull = 2 * kStages,
                         kBarPFull = 2 * kStages + 4, kBarODone = 2 * kStages + 8,
                         kBarFin = 2 * kStages + 10, kBarVZero = 2 * kStages + 12;
    static constexpr int kNumBars = 2 * kStages + 13;
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    static_assert(8 * kNumBars + 16 <= 256, "barrier area");
};
// TMEM columns (512): O of Q tile x at 128x; two S buffers per Q tile at
// 256 + 128x + 64b. P of a tile is written over the S buffer it came from
// (P_hi in its first 32 columns, P_lo in the next 32, two 16-bit values per
// column), so the product of S for tile t + 1 runs while the softmax of tile
// t works, and the softmax never waits for a P V product to write P.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 256;

struct PrefillParams {
    void* out;
    const void* q;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* qsl;
    unsigned int* err;
    int max_blocks;
    int num_heads;
    int num_kv_heads;
    int group;
    int num_seqs;
    int num_blocks;
    int max_tasks;      // 256-row tasks per (sequence, kv head)
    float scale_log2;
    int out_f32;
    const int32_t* order;   // task of each CTA, longest first (null: natural order)
    // split-key mode: CTA i takes chunks 2 j and 2 j + 1 of (sequence, kv
    // head) i mod (S x H_kv), j = i / (S x H_kv), each chunk_tiles key tiles,
    // every key visible to every row; each chunk's (m, l, O) goes to partial
    // slot (sequence x H_kv + kv head) x 2 x pairs + chunk
    int chunk_tiles;
    int pairs;
    uint8_t* slots;
    int slot_bytes;
    int slot_rows;
};

// A task: rows task_off .. task_off + task_rows - 1 of (sequence s, kv head g)
// (row = query token x G + q head within the group), over key tiles 0 .. tiles - 1.
struct Task {
    int c, s, g;
    int L, q0, r;
    int task_off, task_rows;
    int end_blocks, tiles;
};

// Natural task index i: 256-row chunk c = i / (S x H_kv), then sequence, then kv head.
__device__ __forceinline__ Task task_of(const PrefillParams& p, int i) {
    Task k;
    const int sh = p.num_seqs * p.num_kv_heads;
    k.c = i / sh;
    k.s = (i % sh) / p.num_kv_heads;
    k.g = (i % sh) % p.num_kv_heads;
    k.L = __ldg(p.context_lens + k.s);
    if (p.qsl) {
        k.q0 = __ldg(p.qsl + k.s);
        k.r = __ldg(p.qsl + k.s + 1) - k.q0;
    } else {
        k.q0 = k.s;
        k.r = 1;
    }
    const int G = p.group;
    k.task_off = k.c * kTaskRows;
    k.task_rows = min(kTaskRows, G * k.r - k.task_off);
    if (k.task_rows <= 0) {
        k.end_blocks = k.tiles = 0;
        return k;
    }
    // the last row of the task sees keys up to L - r + jmax (causal)
    const int jmax = min(k.r - 1, (k.task_off + k.task_rows - 1) / G);
    k.end_blocks = min((k.L + kBS - 1) / kBS, (k.L - k.r + jmax) / kBS + 1);
    k.tiles = (k.end_blocks + kTileBlocks - 1) / kTileBlocks;
    return k;
}

// Longest-first order of the tasks: a counting sort on the key-tile count
// (clamped to kOrderThreads - 1), so that the block scheduler starts the long
// tasks first and the short ones fill the tail. One CTA; thread k owns key
// bucket kOrderThreads - 1 - k, so bucket starts are an exclusive scan in
// thread order.
constexpr int kOrderThreads = 1024;
constexpr int kOrderCached = 16384;   // task keys kept in shared memory

__global__ void __launch_bounds__(kOrderThreads)
    prefill_order_kernel(const PrefillParams p, int num_tasks, int32_t* order) {
    __shared__ int hist[kOrderThreads];
    __shared__ int warp_sum[kOrderThreads / 32];
    __shared__ uint16_t keys[kOrderCached];
    pa::grid_dependency_wait();
    pa::grid_dependents_launch();
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    auto key_of = [&](int i) {
        return (i < kOrderCached) ? (int)keys[i] : min(task_of(p, i).tiles, kOrderThreads - 1);
    };
    hist[tid] = 0;
    __syncthreads();
    for (int i = tid; i < num_tasks; i += kOrderThreads) {
        const int k = min(task_of(p, i).tiles, kOrderThreads - 1);
        if (i < kOrderCached) keys[i] = (uint16_t)k;
        atomicAdd(&hist[k], 1);
    }
    __syncthreads();
    // exclusive scan of the counts in descending key order
    const int cnt = hist[kOrderThreads - 1 - tid];
    int inc = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += v;
    }
    if (lane == 31) warp_sum[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        int w = warp_sum[lane], wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += v;
        }
        warp_sum[lane] = wi - w;                     // exclusive over warps
    }
    __syncthreads();
    hist[kOrderThreads - 1 - tid] = warp_sum[wid] + inc - cnt;
    __syncthreads();
    for (int i = tid; i < num_tasks; i += kOrderThreads) order[atomicAdd(&hist[key_of(i)], 1)] = i;
}

// byte offset of 16-byte chunk c (0..7) of row `row` inside a 128-byte-wide,
// 128-byte-swizzled matrix (8-row atoms of 1024 bytes)
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return row * 128 + ((c ^ (row & 7)) << 4);
}

// packed two-lane fp32 arithmetic (one instruction for two values)
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <typename T>
struct Cvt;
template <>
struct Cvt<__nv_bfloat16> {
    static constexpr bool kBF16 = true;
    // a, b -> hi = bf16(a, b), lo = bf16 of the remainders (a - hi_a, b - hi_b)
    __device__ static void split(float a, float b, uint32_t& hi, uint32_t& lo) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        hi = *reinterpret_cast<uint32_t*>(&h);
        float ra, rb;
        sub2(ra, rb, a, b, __uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u));
        __nv_bfloat162 l = __floats2bfloat162_rn(ra, rb);
        lo = *reinterpret_cast<uint32_t*>(&l);
    }
    __device__ static void store2(void* p, float a, float b) {
        *static_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
    }
};
template <>
struct Cvt<__half> {
    static constexpr bool kBF16 = false;
    __device__ static void split(float a, float b, uint32_t& hi, uint32_t& lo) {
        __half2 h = __floats2half2_rn(a, b);
        hi = *reinterpret_cast<uint32_t*>(&h);
        float ra, rb;
        sub2(ra, rb, a, b, __low2float(h), __high2float(h));
        __half2 l = __floats2half2_rn(ra, rb);
        lo = *reinterpret_cast<uint32_t*>(&l);
    }
    __device__ static void store2(void* p, float a, float b) {
        *static_cast<__half2*>(p) = __floats2half2_rn(a, b);
    }
};

template <typename T, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
    using C = Cvt<T>;
    using LY = TcLayout<kSplit>;
    constexpr int kStages = LY::kStages, kPerTile = LY::kPerTile, kKVOff = LY::kKVOff,
                  kBarOff = LY::kBarOff, kNumBars = LY::kNumBars;
    constexpr int kBarKVFull = LY::kBarKVFull, kBarKVEmpty = LY::kBarKVEmpty,
                  kBarSFull = LY::kBarSFull, kBarPFull = LY::kBarPFull,
                  kBarODone = LY::kBarODone, kBarFin = LY::kBarFin, kBarVZero = LY::kBarVZero;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = pa::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bars = base + kBarOff;
    uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(smem + kBarOff + 8 * kNumBars);
    volatile int* const abort_flag =
        reinterpret_cast<volatile int*>(smem + kBarOff + 8 * kNumBars + 8);

    pa::grid_dependents_launch();
    pa::grid_dependency_wait();

    // The task of this CTA. Prefill: 256 rows of one (sequence, kv head),
    // longest first when ordered, else later chunks (longer key ranges)
    // first; Q tile x holds rows 128 x of the task and both read key tiles
    // 0 .. tiles - 1. Split keys: all rows of one (sequence, kv head) in Q
    // tile 0; the stream of Q tile x is key chunk 2 j + x, tiles first[x] ..
    // first[x] + cnt[x] - 1.
    int s, g, L, q0, r, task_off, task_rows, end_blocks, tiles, pair = 0;
    int first0 = 0, first1 = 0, cnt0 = 0, cnt1 = 0;   // (registers, not an indexed array)
    if constexpr (kSplit) {
        const int sh = p.num_seqs * p.num_kv_heads;
        pair = (int)blockIdx.x / sh;
        s = ((int)blockIdx.x % sh) / p.num_kv_heads;
        g = ((int)blockIdx.x % sh) % p.num_kv_heads;
        L = __ldg(p.context_lens + s);
        if (p.qsl) {
            q0 = __ldg(p.qsl + s);
            r = __ldg(p.qsl + s + 1) - q0;
        } else {
            q0 = s;
            r = 1;
        }
        task_off = 0;
        task_rows = min(p.slot_rows, p.group * r);
        end_blocks = (L + kBS - 1) / kBS;
        tiles = (end_blocks + kTileBlocks - 1) / kTileBlocks;
        first0 = 2 * pair * p.chunk_tiles;
        first1 = first0 + p.chunk_tiles;
        cnt0 = max(0, min(p.chunk_tiles, tiles - first0));
        cnt1 = max(0, min(p.chunk_tiles, tiles - first1));
        if (cnt0 == 0) return;                                   // uniform over the CTA
    } else {
        const int ntask = p.max_tasks * p.num_seqs * p.num_kv_heads;
        const Task tk =
            task_of(p, p.order ? __ldg(p.order + blockIdx.x) : ntask - 1 - (int)blockIdx.x);
        s = tk.s;
        g = tk.g;
        L = tk.L;
        q0 = tk.q0;
        r = tk.r;
        task_off = tk.task_off;
        task_rows = tk.task_rows;
        end_blocks = tk.end_blocks;
        tiles = tk.tiles;
        cnt0 = cnt1 = tiles;
    }
    auto first_of = [&](int x) { return x ? first1 : first0; };
    auto cnt_of = [&](int x) { return x ? cnt1 : cnt0; };
    const int G = p.group;
    if (task_rows <= 0) return;                                  // uniform over the CTA
    // Q tiles with work: prefill, those holding rows; split keys, those with a chunk
    const int nq = kSplit ? (cnt1 > 0 ? 2 : 1) : (task_rows > kRows ? 2 : 1);
    // ring stage and parity of the u-th tile of Q tile x's stream
    auto stage_of = [&](int x, int u) { return kSplit ? x * kPerTile + u % kPerTile : u % kStages; };
    auto phase_of = [&](int u) { return (u / kPerTile) & 1; };

    if (threadIdx.x == 0) {
        // P full and V zeroed take one arrival from each of the four warps of
        // a softmax group; K/V empty one commit from each Q tile's MMA warp
        // that reads the stage (both in prefill, the owner with split keys)
        for (int i = 0; i < kNumBars; ++i)
            pa::mbar_init(bars + 8 * i, ((i >= kBarPFull && i < kBarODone) || i == kBarVZero) ? 4
                                        : (i >= kBarKVEmpty && i < kBarKVEmpty + kStages)
                                            ? (kSplit ? 1 : nq)
                                            : 1);
        *abort_flag = 0;
        pa::fence_barrier_init();
        pa::prefetch_tensormap(&tmap_k);
        pa::prefetch_tensormap(&tmap_v);
    }
    if (warp == 1) {
        pa::tc::tmem_alloc(pa::smem_addr(tmem_holder), kTmemCols);
        pa::tc::tmem_relinquish();
    }
    // Q tiles: 128 rows x 128 dims each, 128-byte swizzled K-major (two 64-dim halves)
    for (int e = threadIdx.x; e < (kSplit ? 1 : nq) * kRows * 16; e += kThreads) {
        const int trow = e >> 4, ch = e & 15;          // task row 0..255
        uint4 v = make_uint4(0, 0, 0, 0);
        if (trow < task_rows) {
            const int gr = task_off + trow;
            const T* src = static_cast<const T*>(p.q) +
                           ((int64_t)(q0 + gr / G) * p.num_heads + g * G + gr % G) * D;
            v = __ldg(reinterpret_cast<const uint4*>(src) + ch);
        }
        const int x = trow / kRows, row = trow % kRows;
        const uint32_t dst =
            base + kQOff + x * kQBytes + (ch >> 3) * (kRows * 128) + sw128(row, ch & 7);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    pa::tc::fence_before_sync();
    __syncthreads();
    pa::tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ---------------- producer: K/V blocks of each tile ----------------
        // lane j handles block j of a tile
        auto block_row = [&](int t) {
            const int nblk = min(kTileBlocks, end_blocks - t * kTileBlocks);
            if (t >= tiles || lane >= nblk) return -1;
            int blk = __ldg(p.block_tables + (int64_t)s * p.max_blocks + t * kTileBlocks + lane);
            if (blk < 0 || blk >= p.num_blocks) {
                if (p.err) atomicOr(p.err, pa::ERR_BAD_BLOCK);
                blk = 0;
            }
            return (blk * p.num_kv_heads + g) * kBS;
        };
        auto load_tile = [&](int t, int st, int row) {
            const int nblk = min(kTileBlocks, end_blocks - t * kTileBlocks);
            const uint32_t bar = bars + 8 * (kBarKVFull + st);
            if (lane == 0) pa::mbar_arrive_expect_tx(bar, nblk * 4 * (kBS * 128));
            __syncwarp();
            if (lane < nblk) {
                const uint32_t kst = base + kKVOff + st * kKVStage + lane * (kBS * 128);
#pragma unroll
                for (int sub = 0; sub < 2; ++sub) {
                    pa::tma_load_2d(kst + sub * kSubKV, &tmap_k, sub * 64, row, bar);
                    pa::tma_load_2d(kst + kKBytes + sub * kSubKV, &tmap_v, sub * 64, row, bar);
                }
            }
        };
        // a stage is free once every product reading its previous tile is done
        auto stage_free = [&](int st, int u) {
            const bool ok = __all_sync(
                0xffffffffu, pa::mbar_wait(bars + 8 * (kBarKVEmpty + st), ((u / kPerTile) - 1) & 1,
                                           p.err, pa::ERR_WAIT_EMPTY));
            if (!ok || *abort_flag) {
                if (lane == 0) *abort_flag = 1;
                return false;
            }
            return true;
        };
        int issued0 = 0, issued1 = 0;
        if constexpr (kSplit) {
            // the two chunks' streams interleaved, each through its own stages
            bool go = true;
            for (int u = 0; go && u < max(cnt0, cnt1); ++u)
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    if (!go || u >= cnt_of(x)) continue;
                    const int st = stage_of(x, u);
                    if (u >= kPerTile && !stage_free(st, u)) {
                        go = false;
                        continue;
                    }
                    load_tile(first_of(x) + u, st, block_row(first_of(x) + u));
                    if (x) issued1 = u + 1;
                    else issued0 = u + 1;
                }
        } else {
            // the block ids of the next tile are fetched before waiting for the stage
            int row = block_row(0);
            for (int t = 0; t < tiles; ++t) {
                const int st = t % kStages;
                const int next_row = block_row(t + 1);
                if (t >= kStages && !stage_free(st, t)) break;
                load_tile(t, st, row);
                row = next_row;
                issued0 = t + 1;
            }
        }
        // drain: no copy may be in flight when the CTA ends; the last kPerTile
        // issued tiles of each stream are waited once more (each completes
        // whether or not it was consumed; earlier ones were consumed before
        // their stage was reused)
        if (lane == 0)
            for (int x = 0; x < (kSplit ? 2 : 1); ++x) {
                const int iss = x ? issued1 : issued0;
                for (int u = iss > kPerTile ? iss - kPerTile : 0; u < iss; ++u)
                    if (!pa::mbar_wait(bars + 8 * (kBarKVFull + stage_of(x, u)), phase_of(u),
                                       nullptr, 0)) {
                        if (p.err) atomicOr(p.err, pa::ERR_WAIT_DRAIN);
                        break;
                    }
            }
    } else if (warp == 1 || warp == 2 + 4 * kQTiles) {
        // ---------------- MMA issue: one warp per Q tile (one elected lane issues) ----------------
        // S is double-buffered: QK_x(u) writes buffer u & 1 once PV_x(u - 2),
        // which read P_x(u - 2) from it, has completed. Order per key tile u
        // of the stream: PV_x(u), then QK_x(u + 2). Each Q tile has its own
        // issuing warp, so the waits and bookkeeping of one overlap the
        // products of the other on the shared tensor pipe. Operands are made
        // warp-uniform (read from lane 0) so the issue stays a converged,
        // uniform instruction stream.
        const int x = warp == 1 ? 0 : 1;
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        const uint32_t sb = __shfl_sync(0xffffffffu, base, 0);
        const uint32_t bb = sb + kBarOff;
        constexpr uint32_t idesc_qk = pa::tc::idesc_f16(C::kBF16, false, false, kRows, kTok);
        constexpr uint32_t idesc_pv = pa::tc::idesc_f16(C::kBF16, false, true, kRows, D);
        auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
            if (__all_sync(0xffffffffu, pa::mbar_try_wait(bar, parity))) return true;
            const bool ok = __all_sync(0xffffffffu, pa::mbar_wait(bar, parity, p.err, pa::ERR_WAIT_FULL));
            return ok && __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
        };
        // descriptors of every operand start: a descriptor of address a + o is
        // the one of a plus o >> 4 (the 14-bit address field does not overflow
        // inside shared memory); with split keys both Q tiles read Q tile 0
        const uint64_t dq = pa::tc::smem_desc_sw128(sb + kQOff + (kSplit ? 0 : x) * kQBytes, 16, 1024);
        const uint64_t dk = pa::tc::smem_desc_sw128(sb + kKVOff, 16, 1024);
        const uint64_t dv = pa::tc::smem_desc_sw128(sb + kKVOff + kKBytes, kSubKV, 1024);
        const uint32_t s_col = tm + kSCol + 128 * x, o_col = tm + 128 * x;
        auto issue_qk = [&](int u) {   // S_x[u & 1] = Q_x K(u)^T
            pa::tc::fence_after_sync();
            const uint64_t b0 = dk + (uint64_t)((stage_of(x, u) * kKVStage) >> 4);
            const uint32_t d = s_col + 64 * (u & 1);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t qa = ((kk >> 2) * (kRows * 128) + (kk & 3) * 32) >> 4;
                const uint32_t kb = ((kk >> 2) * kSubKV + (kk & 3) * 32) >> 4;
                pa::tc::mma_f16_ss_warp(d, dq + qa, b0 + kb, idesc_qk, kk > 0 ? 1u : 0u);
            }
            pa::tc::commit_warp(bb + 8 * (kBarSFull + 2 * x + (u & 1)));
        };
        auto issue_pv = [&](int u) {   // O_x += P_x(u) V(u)
            pa::tc::fence_after_sync();
            const uint64_t v0 = dv + (uint64_t)((stage_of(x, u) * kKVStage) >> 4);
            const int nblk = min(kTileBlocks, end_blocks - (first_of(x) + u) * kTileBlocks);
            const uint32_t pc = s_col + 64 * (u & 1);
            const uint32_t acc0 = u > 0 ? 1u : 0u;
#pragma unroll
            for (int kb = 0; kb < kTileBlocks; ++kb) {
                if (kb < nblk) {
                    const uint64_t bv = v0 + (uint64_t)((kb * (kBS * 128)) >> 4);
                    pa::tc::mma_f16_ts_warp(o_col, pc + 8 * kb, bv, idesc_pv, kb > 0 ? 1u : acc0);
                    pa::tc::mma_f16_ts_warp(o_col, pc + 32 + 8 * kb, bv, idesc_pv, 1u);
                }
            }
            pa::tc::commit_warp(bb + 8 * (kBarODone + x));
        };
        auto kv_ready = [&](int u) {
            return wait(bb + 8 * (kBarKVFull + stage_of(x, u)), phase_of(u));
        };
        // prefill: the last tile may hold V rows past the context, which Q
        // tile 0's softmax zeroes before its P of that tile is ready (with
        // split keys the tile's own softmax group does it before its P)
        const int zero_tile = !kSplit && end_blocks * kBS > L ? tiles - 1 : -1;
        const int n = cnt_of(x);
        bool ok = x < nq;
        if (ok) {
            // both S buffers start free: the products of S for tiles 0 and 1
            for (int u = 0; ok && u < min(n, 2); ++u) {
                ok = kv_ready(u);
                if (ok) issue_qk(u);
            }
            for (int u = 0; ok && u < n; ++u) {
                ok = wait(bb + 8 * (kBarPFull + 2 * x + (u & 1)), (u >> 1) & 1);
                if (ok && x == 1 && u == zero_tile) ok = wait(bb + 8 * kBarVZero, 0);
                if (!ok) break;
                issue_pv(u);
                // every product of this Q tile reading K/V tile u has been issued
                pa::tc::commit_warp(bb + 8 * (kBarKVEmpty + stage_of(x, u)));
                if (u + 2 < n) {
                    // PV_x(u) read S_x[u & 1]
                    ok = kv_ready(u + 2) && wait(bb + 8 * (kBarODone + x), u & 1);
                    if (ok) issue_qk(u + 2);
                }
            }
            if (!ok && lane == 0) *abort_flag = 1;
            // every MMA this warp issued has finished before TMEM is freed
            pa::tc::commit_warp(bb + 8 * (kBarFin + x));
            if (!__all_sync(0xffffffffu, pa::mbar_wait(bb + 8 * (kBarFin + x), 0, nullptr, 0)) &&
                lane == 0 && p.err)
                atomicOr(p.err, pa::ERR_WAIT_DRAIN);
        }
    } else if ((warp - 2) / 4 < nq) {
        // ---------------- softmax and epilogue: one thread per row of Q tile x ----------------
        const int x = (warp - 2) / 4;
        const int lane_base = 32 * (warp & 3);
        const int row = lane_base + lane;                    // tile row = TMEM lane
        const int row_off = kSplit ? 0 : task_off + x * kRows;
        const int rows = kSplit ? task_rows : min(kRows, task_rows - x * kRows);
        const int gr = row_off + row;
        const bool valid = row < rows;
        const int jq = valid ? gr / G : 0;
        // keys past a row's bound are masked; padding rows (Q = 0) need no
        // mask; with split keys every key before L is visible to every row
        const int bound = kSplit ? L - 1 : valid ? min(L - r + jq, L - 1) : 0x7fffffff;
        // the smallest bound of the tile's rows: tiles ending at or before it need no mask
        const int bound_min = kSplit ? L - 1 : min(L - r + row_off / G, L - 1);
        const uint32_t trow = tmem + ((uint32_t)lane_base << 16);
        const uint32_t s_tm = trow + kSCol + 128 * x, o_tm = trow + 128 * x;
        const uint32_t bar_odone = bars + 8 * (kBarODone + x);
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        const int grp_tid = (warp - 2 - 4 * x) * 32 + lane;  // 0..127 within the group
        const int n = cnt_of(x);
        const bool live = lane_base < rows;                  // warp-uniform
        int done = 0;
        for (int u = 0; u < n; ++u) {
            const int b = u & 1;                               // S / P buffer of this tile
            bool ok = __all_sync(0xffffffffu, pa::mbar_wait(bars + 8 * (kBarSFull + 2 * x + b),
                                                            (u >> 1) & 1, p.err, pa::ERR_WAIT_FULL));
            if (!ok || *abort_flag) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            pa::tc::fence_after_sync();
            const int t = first_of(x) + u;                     // key tile
            const int tok0 = t * kTok;
            // A warp whose 32 rows are all padding (Q = 0: S, and so P, are
            // zero in TMEM already) skips the softmax; it still waits for S
            // and arrives on P full in order, which keeps the barrier phases.
            if (live) {
            float sv[kTok];
            pa::tc::ld_64cols(s_tm + 64 * b, *reinterpret_cast<uint32_t(*)[64]>(sv));
            if (tok0 + kTok - 1 > bound_min) {               // a tile some row must not see all of
#pragma unroll
                for (int j = 0; j < kTok; ++j)
                    if (tok0 + j > bound) sv[j] = -INFINITY;
            }
            float m4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
            for (int j = 4; j < kTok; j += 8)
#pragma unroll
                for (int q = 0; q < 4; ++q) m4[q] = max3(m4[q], sv[j + 2 * q], sv[j + 2 * q + 1]);
            float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            mx = mx == -INFINITY ? mx : mx * sl2;            // the scale is positive
            float alpha = 1.f;
            bool moved = false;
            if (mx > m_run + kLazyMax) {
                alpha = pa::ex2(m_run - mx);                   // 0 while m_run is -inf
                m_run = mx;
                moved = true;
            }
            const float nm = m_run == -INFINITY ? 0.f : -m_run;
#pragma unroll
            for (int j = 0; j < kTok; j += 2) {
                fma2(sv[j], sv[j + 1], sv[j], sv[j + 1], sl2, sl2, nm, nm);
                sv[j] = pa::ex2(sv[j]);
                sv[j + 1] = pa::ex2(sv[j + 1]);
            }
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < kTok; j += 4) {
                add2(s4[0], s4[1], s4[0], s4[1], sv[j], sv[j + 1]);
                add2(s4[2], s4[3], s4[2], s4[3], sv[j + 2], sv[j + 3]);
            }
            l_run = l_run * alpha + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
            uint32_t pk[64];
#pragma unroll
            for (int j = 0; j < kTok / 2; ++j) C::split(sv[2 * j], sv[2 * j + 1], pk[j], pk[32 + j]);
            // O_x may be rescaled once the P V product of tile u - 1 is done
            // (rare: the running max moves by more than 2^8 after the first tile)
            if (u >= 1 && __any_sync(0xffffffffu, moved)) {
                ok = __all_sync(0xffffffffu,
                                pa::mbar_wait(bar_odone, (u - 1) & 1, p.err, pa::ERR_WAIT_FULL));
                if (!ok || *abort_flag) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
                pa::tc::fence_after_sync();
                // rescale this warp's rows of O in TMEM (alpha = 1 for the others)
#pragma unroll 1
                for (int q = 0; q < D / 16; ++q) {
                    uint32_t ov[16];
                    pa::tc::ld_16cols(o_tm + 16 * q, ov);
#pragma unroll
                    for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    pa::tc::st_16cols(o_tm + 16 * q, ov);
                }
            }
            // P over the S buffer it came from (this thread's row only)
            pa::tc::st_64cols(s_tm + 64 * b, pk);
            }
            // V rows past the context (in the sequence's last block) may hold
            // anything: zero them so that P = 0 never meets a NaN (prefill: Q
            // tile 0's group does it and signals Q tile 1's MMA warp; split
            // keys: the one stream holding that tile)
            const int nblk = min(kTileBlocks, end_blocks - t * kTileBlocks);
            const int tok_end = tok0 + nblk * kBS;
            if ((kSplit || x == 0) && L < tok_end) {
                const int z0 = L - tok0, zrows = tok_end - L;      // local token rows to zero
                for (int e = grp_tid; e < zrows * 16; e += 128) {
                    const int lr = z0 + e / 16, ch = e % 16;
                    const uint32_t dst = base + kKVOff + stage_of(x, u) * kKVStage + kKBytes +
                                         (ch >> 3) * kSubKV + lr * 128 + ((ch & 7) << 4);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0u)
                                 : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            // each warp releases its part (no group-wide barrier a stalled warp could hold)
            pa::tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                pa::mbar_arrive(bars + 8 * (kBarPFull + 2 * x + b));
                // Q tile 1's product of this tile reads the zeroed rows
                if (!kSplit && x == 0 && L < tok_end) pa::mbar_arrive(bars + 8 * kBarVZero);
            }
            done = u + 1;
        }
        // epilogue: O / l for this row (prefill), or the chunk's partial (m, l, O)
        if (live && done == n && n > 0) {
            // every product of this Q tile is done: the MMA warp's final
            // commit, a barrier with one phase in the CTA's life. (Waiting for
            // the last P V products on the O-done barrier by parity is not
            // safe: if the last one completes before the wait for the one
            // before it is observed, the barrier is two phases on and that
            // parity names a phase that never completes.)
            bool ok = __all_sync(0xffffffffu, pa::mbar_wait(bars + 8 * (kBarFin + x), 0, p.err,
                                                            pa::ERR_WAIT_FULL));
            if (ok) {
                pa::tc::fence_after_sync();
                if constexpr (kSplit) {
                    const int64_t slot =
                        ((int64_t)s * p.num_kv_heads + g) * 2 * p.pairs + 2 * pair + x;
                    uint8_t* const sp = p.slots + slot * (int64_t)p.slot_bytes;
                    float* const sm_ = reinterpret_cast<float*>(sp + 32);
                    float* const sl_ = sm_ + p.slot_rows;
                    float* const so = sl_ + p.slot_rows;
                    if (valid) {
                        sm_[row] = m_run;
                        sl_[row] = l_run;
                    }
#pragma unroll
                    for (int qd = 0; qd < D / 32; ++qd) {
                        float ov[32];
                        pa::tc::ld_32cols(o_tm + 32 * qd, ov);
                        if (valid) {
                            float* dst = so + (int64_t)row * D + 32 * qd;
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4*>(dst + i) =
                                    make_float4(ov[i], ov[i + 1], ov[i + 2], ov[i + 3]);
                        }
                    }
                } else {
                    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                    const int64_t orow =
                        valid ? ((int64_t)(q0 + gr / G) * p.num_heads + g * G + gr % G) : 0;
#pragma unroll
                    for (int qd = 0; qd < D / 32; ++qd) {
                        float ov[32];
                        pa::tc::ld_32cols(o_tm + 32 * qd, ov);
                        if (valid) {
                            if (p.out_f32) {
                                float* dst = static_cast<float*>(p.out) + orow * D + 32 * qd;
#pragma unroll
                                for (int i = 0; i < 32; i += 4)
                                    *reinterpret_cast<float4*>(dst + i) =
                                        make_float4(ov[i] * inv, ov[i + 1] * inv, ov[i + 2] * inv,
                                                    ov[i + 3] * inv);
                            } else {
                                T* dst = static_cast<T*>(p.out) + orow * D + 32 * qd;
#pragma unroll
                                for (int i = 0; i < 32; i += 2)
                                    C::store2(dst + i, ov[i] * inv, ov[i + 1] * inv);
                            }
                        }
                    }
                }
            } else if (lane == 0) {
                *abort_flag = 1;
            }
        }
    }
    pa::tc::fence_before_sync();
    __syncthreads();
    pa::tc::fence_after_sync();
    if (warp == 1) pa::tc::tmem_dealloc(tmem, kTmemCols);
}

// Split keys: merges the key chunks of every (sequence, kv head) row, one
// warp per (sequence, kv head, row) item, into the normalised fp32 output
// row and its base-2 log-sum-exp, by the log-sum-exp rule: out = sum 2^(m_c
// - M) O_c / sum 2^(m_c - M) l_c. A sequence with no key writes nothing.
__global__ void __launch_bounds__(128) prefix_chunk_reduce_kernel(const PrefillParams p,
                                                                  float* lse_out) {
    constexpr int EPL = D / 32;
    pa::grid_dependency_wait();     // every chunk's partial is written
    pa::grid_dependents_launch();
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int row = (int)(item % p.slot_rows);
    const int64_t seg = item / p.slot_rows;
    if (seg >= (int64_t)p.num_seqs * p.num_kv_heads) return;
    const int s = (int)(seg / p.num_kv_heads), g = (int)(seg % p.num_kv_heads);
    int q0 = s, r = 1;
    if (p.qsl) {
        q0 = __ldg(p.qsl + s);
        r = __ldg(p.qsl + s + 1) - q0;
    }
    const int G = p.group;
    if (row >= min(p.slot_rows, G * r)) return;
    const int L = __ldg(p.context_lens + s);
    const int tiles = ((L + kBS - 1) / kBS + kTileBlocks - 1) / kTileBlocks;
    const int nch = min(2 * p.pairs, (tiles + p.chunk_tiles - 1) / p.chunk_tiles);
    if (nch <= 0) return;
    float M = -INFINITY, den = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    for (int c = 0; c < nch; ++c) {
        const uint8_t* sp = p.slots + (seg * 2 * p.pairs + c) * (int64_t)p.slot_bytes;
        const float* m = reinterpret_cast<const float*>(sp + 32);
        const float l = __ldg(m + p.slot_rows + row);
        if (!(l > 0.f)) continue;
        const float mc = __ldg(m + row);
        const float4 o = __ldg(reinterpret_cast<const float4*>(m + 2 * p.slot_rows +
                                                               (int64_t)row * D + lane * EPL));
        const float Mn = fmaxf(M, mc);
        const float a = exp2f(M - Mn), w = exp2f(mc - Mn);
        den = den * a + w * l;
        acc[0] = acc[0] * a + w * o.x;
        acc[1] = acc[1] * a + w * o.y;
        acc[2] = acc[2] * a + w * o.z;
        acc[3] = acc[3] * a + w * o.w;
        M = Mn;
    }
    if (!(den > 0.f)) return;
    const int64_t orow = (int64_t)(q0 + row / G) * p.num_heads + g * G + row % G;
    const float inv = 1.f / den;
    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * D + lane * EPL) =
        make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    if (lane == 0) lse_out[orow] = M + log2f(den);
}

template <typename T, bool kSplit>
pa_status launch(const pa::DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                 const PrefillParams& prm, int64_t grid) {
    auto kern = paged_prefill_tc_kernel<T, kSplit>;
    constexpr int smem = TcLayout<kSplit>::kSmem;
    static bool attr_set = false;   // per instantiation; benign race (idempotent)
    if (!attr_set) {
        if (pa_status s = pa::cuda_status(
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                "prefill: set shared memory size"))
            return s;
        attr_set = true;
    }
    return pa::cuda_status(
        pa::launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, a.stream, mk, mv, prm),
        "prefill launch");
}

PrefillParams base_params(const pa::DecodeArgs& a) {
    PrefillParams prm{};
    prm.out = a.out;
    prm.q = a.q;
    prm.block_tables = a.block_tables;
    prm.context_lens = a.context_lens;
    prm.qsl = a.query_start_loc;
    prm.err = pa::device_error_word();
    prm.max_blocks = a.max_blocks_per_seq;
    prm.num_heads = a.num_heads;
    prm.num_kv_heads = a.num_kv_heads;
    prm.group = a.num_heads / a.num_kv_heads;
    prm.num_seqs = a.num_seqs;
    prm.num_blocks = a.num_blocks;
    prm.scale_log2 = a.scale * kLog2e;
    prm.out_f32 = a.out_dtype == PA_F32;
    return prm;
}

// Split keys: key tiles per chunk at least this many (shorter chunks would
// spend more on the per-chunk prologue and the partials than they save)
constexpr int kMinChunkTiles = 8;
// rows of a split-key task (the partial slots of the balanced schedule's
// 64-row tiles hold them)
constexpr int kSplitRows = 64;

}  // namespace

namespace pa {

// Long query runs over a 16-bit cache with head_dim 128 (and no token offset
// or log-sum-exp output): at least 256 query rows per KV head.
bool prefill_tc_applies(const DecodeArgs& a) {
    const int64_t rows = (int64_t)(a.num_heads / a.num_kv_heads) * a.max_q_len;
    return (a.kv_dtype == PA_BF16 || a.kv_dtype == PA_F16) && a.head_dim == 128 &&
           a.partition_size == 0 && !a.ctx_start && !a.lse_out && !a.unmasked && rows >= 256;
}

pa_status launch_prefill_tc(const DecodeArgs& a) {
    const int G = a.num_heads / a.num_kv_heads;
    const int64_t max_tasks = ((int64_t)G * a.max_q_len + kTaskRows - 1) / kTaskRows;
    const int64_t grid = max_tasks * a.num_seqs * a.num_kv_heads;
    if (grid > 0x7fffffff) return fail(PA_ERR_UNSUPPORTED, "prefill grid too large");
    CUtensorMap mk, mv;
    if (pa_status s = cache_tensor_map(&mk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 2))
        return s;
    if (pa_status s = cache_tensor_map(&mv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 2))
        return s;
    PrefillParams prm = base_params(a);
    prm.max_tasks = (int)max_tasks;
    // the task order goes to the start of the balanced schedule's workspace
    // (the caller sized it with pa_decode_workspace_size, 256-byte aligned)
    const BalancedShape ws = balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads, a.head_dim,
                                            a.max_q_len, a.max_context_len);
    if (a.slots && grid * 4 <= ws.workspace_bytes) {
        prm.order = static_cast<int32_t*>(a.slots);
        if (pa_status s = pa::cuda_status(
                pa::launch_pdl(prefill_order_kernel, dim3(1), dim3(kOrderThreads), 0, a.stream,
                               prm, (int)grid, static_cast<int32_t*>(a.slots)),
                "prefill order launch"))
            return s;
    }
    if (a.kv_dtype == PA_BF16) return launch<__nv_bfloat16, false>(a, mk, mv, prm, grid);
    return launch<__half, false>(a, mk, mv, prm, grid);
}

// The prefix phase of shared-prefix decode over a 16-bit cache with
// head_dim 128: every key visible to every row (no causal offset), a
// log-sum-exp per row, 17 to 64 rows per (group, kv head), long prefixes.
bool prefix_tc_applies(const DecodeArgs& a) {
    const int64_t rows = (int64_t)(a.num_heads / a.num_kv_heads) * a.max_q_len;
    return (a.kv_dtype == PA_BF16 || a.kv_dtype == PA_F16) && a.head_dim == 128 &&
           a.partition_size == 0 && !a.ctx_start && a.lse_out && a.unmasked &&
           a.out_dtype == PA_F32 && rows > 16 && rows <= kSplitRows &&
           a.max_context_len >= 2 * kMinChunkTiles * kTok;
}

// Split keys: (group, kv head) tasks cut into key chunks so that the CTAs
// (one per SM) about fill the GPU: chunk pairs per task and key tiles per chunk.
static void split_shape(const DecodeArgs& a, int sms, int64_t* pairs, int64_t* chunk_tiles) {
    const int64_t segs = (int64_t)a.num_seqs * a.num_kv_heads;
    const int64_t tiles_max = ((a.max_context_len + kBS - 1) / kBS + kTileBlocks - 1) / kTileBlocks;
    const int64_t pairs_by_len = std::max<int64_t>(1, tiles_max / (2 * kMinChunkTiles));
    *pairs = std::max<int64_t>(1, std::min<int64_t>(sms / segs, pairs_by_len));
    *chunk_tiles = (tiles_max + 2 * *pairs - 1) / (2 * *pairs);
}

// CTAs of the split-key launch for these arguments (0 where it does not apply).
int64_t prefix_tc_ctas(const DecodeArgs& a, int sms) {
    if (!prefix_tc_applies(a)) return 0;
    int64_t pairs = 0, chunk_tiles = 0;
    split_shape(a, sms, &pairs, &chunk_tiles);
    return (int64_t)a.num_seqs * a.num_kv_heads * pairs;
}

// Split keys, then the chunks merged per row.
pa_status launch_prefix_tc(const DecodeArgs& a) {
    int dev = 0, sms = 0;
    if (pa_status s = pa::cuda_status(cudaGetDevice(&dev), "cudaGetDevice")) return s;
    if (pa_status s = pa::cuda_status(
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count"))
        return s;
    const int64_t segs = (int64_t)a.num_seqs * a.num_kv_heads;
    int64_t pairs = 0, chunk_tiles = 0;
    split_shape(a, sms, &pairs, &chunk_tiles);
    const int64_t grid = segs * pairs;
    // the partials go to the balanced schedule's slots (64-row tiles) of this workspace
    const BalancedShape ws = balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads, a.head_dim,
                                            a.max_q_len, a.max_context_len);
    if (!a.slots || ws.rows_per_tile != kSplitRows || segs * 2 * pairs > 2 * ws.workers ||
        grid > 0x7fffffff)
        return fail(PA_ERR_UNSUPPORTED, "prefix phase: workspace too small for the key chunks");
    CUtensorMap mk, mv;
    if (pa_status s = cache_tensor_map(&mk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 2))
        return s;
    if (pa_status s = cache_tensor_map(&mv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 2))
        return s;
    PrefillParams prm = base_params(a);
    prm.chunk_tiles = (int)chunk_tiles;
    prm.pairs = (int)pairs;
    prm.slots = static_cast<uint8_t*>(a.slots) + ws.cum_bytes;
    prm.slot_bytes = (int)ws.slot_bytes;
    prm.slot_rows = kSplitRows;
    pa_status st = a.kv_dtype == PA_BF16 ? launch<__nv_bfloat16, true>(a, mk, mv, prm, grid)
                                         : launch<__half, true>(a, mk, mv, prm, grid);
    if (st != PA_OK) return st;
    const int64_t items = segs * kSplitRows;
    return pa::cuda_status(
        pa::launch_pdl(prefix_chunk_reduce_kernel, dim3((unsigned)((items + 3) / 4)), dim3(128),
                       0, a.stream, prm, a.lse_out),
        "prefix chunk reduce launch");
}

}  // namespace pa
