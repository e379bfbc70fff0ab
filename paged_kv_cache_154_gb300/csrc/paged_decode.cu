// Paged decode attention for F16/BF16 caches, and its partial-result merges.
//
// What it computes: "KV Cache ... PagedAttention" (devpress.csdn.net) §二,
// softmax(Q K^T / sqrt(d)) V, over the keys a sequence holds in its blocks
// (§七: the block table maps logical block b to a physical block); "cs336
// lecture 10", decode workflow: the new token's q against every cached K,
// weighted sum of the cached V; GQA/MQA from the same lecture: the q heads
// of one group share one KV head, so one KV read serves the whole group.
//
// Per 16-token block a warp computes S = Q K^T with m16n8k16 tensor-core
// MMAs (the query rows of one KV head -- G q heads x r query tokens -- in M,
// padded to 16; fp32 accumulate), applies the causal/length mask, updates an
// fp32 online softmax (running max and sum, base-2 exponentials) and
// accumulates O += P V with P split as P_hi + P_lo in the 16-bit type, so the
// weights keep ~16 mantissa bits. K and V tiles reach shared memory by 2-D
// bulk tensor copies (TMA, 128-byte swizzle) completing on mbarriers.
//
// Two schedules share that block step:
//   * balanced (default, partition_size == 0): a persistent grid of warps,
//     each an independent worker with its own TMA ring. The (sequence, kv
//     head, block) space is cut into equal contiguous shares, one per warp,
//     so every warp streams the same number of blocks. A (sequence, kv head)
//     segment that a warp covers whole is written as final output; where a
//     share boundary cuts a segment, each side writes a partial (m, l, O)
//     and segment_reduce_kernel merges them with the log-sum-exp rule.
//   * partitioned (partition_size > 0): grid (partition, kv head, sequence),
//     one producer warp + four consumer warps per CTA, partitions merged by
//     split_kv_reduce_kernel.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <math.h>

#include <algorithm>
#include <mutex>

#include "balanced.cuh"
#include "pa_internal.h"
#include "ptx.cuh"

#ifdef PA_TEST_HOOKS
// Test builds only (-DPA_TEST_HOOKS): the balanced kernel's first worker
// skips issuing the copy of its k-th block when k == g_test_skip_copy, so
// that the wait for that block runs out and the kernel reports it.
__device__ int g_test_skip_copy = -1;
extern "C" pa_status pa_test_skip_copy(int k) {
    return pa::cuda_status(cudaMemcpyToSymbol(g_test_skip_copy, &k, sizeof k), "test hook");
}
#endif

namespace {

constexpr int kBS = 16;                  // tokens per block
constexpr int kConsumerWarps = 4;        // partitioned schedule
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxPartBlocks = 256;      // partition_size <= 4096 tokens
constexpr int kWorkerWarps = 4;          // balanced schedule: warps per CTA
constexpr float kLog2e = 1.4426950408889634f;

template <typename T>
struct Pack;
template <>
struct Pack<__nv_bfloat16> {
    static constexpr bool kBF16 = true;
    __device__ static uint32_t pack(float lo, float hi, float& rlo, float& rhi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        rlo = lo - __low2float(v);
        rhi = hi - __high2float(v);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ static void store(void* p, float x) {
        *static_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(x);
    }
    __device__ static void store2(void* p, float a, float b) {
        *static_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
    }
};
template <>
struct Pack<__half> {
    static constexpr bool kBF16 = false;
    __device__ static uint32_t pack(float lo, float hi, float& rlo, float& rhi) {
        __half2 v = __floats2half2_rn(lo, hi);
        rlo = lo - __low2float(v);
        rhi = hi - __high2float(v);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ static uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ static void store(void* p, float x) { *static_cast<__half*>(p) = __float2half_rn(x); }
    __device__ static void store2(void* p, float a, float b) {
        *static_cast<__half2*>(p) = __floats2half2_rn(a, b);
    }
};

// Byte offset of the 16-byte chunk `chunk` of row `row` in a K/V tile laid
// out by the 128B-swizzled TMA box [16 rows][64 columns] per sub-tile.
__device__ __forceinline__ uint32_t tile_offset(int row, int chunk) {
    const int sub = chunk >> 3, c = chunk & 7;
    return sub * (kBS * 128) + row * 128 + ((c ^ (row & 7)) << 4);
}

// Issue the K and V copies of one (block, kv head) tile into a stage: one
// copy each (head_dim 128 through the whole-tile view, 64 through one box).
template <int D>
__device__ __forceinline__ void issue_tile(uint32_t stage, uint32_t bar, const CUtensorMap* mk,
                                           const CUtensorMap* mv, int row, uint64_t pol) {
    constexpr int kTile = kBS * D * 2;
    pa::mbar_arrive_expect_tx(bar, 2 * kTile);
    if constexpr (D == 128) {
        pa::tma_load_3d(stage, mk, 0, row, 0, bar, pol);
        pa::tma_load_3d(stage + kTile, mv, 0, row, 0, bar, pol);
    } else {
        pa::tma_load_2d(stage, mk, 0, row, bar, pol);
        pa::tma_load_2d(stage + kTile, mv, 0, row, bar, pol);
    }
}

// One warp's attention state over some blocks of one (sequence, kv head):
// MT m-tiles of 16 query rows, fp32 O accumulators, running max and sum
// (per thread: its two rows of each m-tile; l is a per-thread partial sum
// until quad_sum()).
template <typename T, int D, int MT>
struct WarpAttn {
    static constexpr int kKSteps = D / 16;
    static constexpr int kNTiles = D / 8;
    float o[MT][kNTiles][4];
    float m_run[MT][2];
    float l_run[MT][2];

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int nt = 0; nt < kNTiles; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
            m_run[mt][0] = m_run[mt][1] = -INFINITY;
            l_run[mt][0] = l_run[mt][1] = 0.f;
        }
    }

    // One 16-token block staged at kb (K tile) and kb + tile (V tile).
    //   qreg   A fragments of Q (MT == 1), or qsm: smem Q tile base (MT > 1 or
    //          QSMEM; rows at a pitch of QPITCH bytes)
    //   tok0   absolute position of the block's first token
    //   last_q L - r: query row i sees keys <= L - r + i (row i = row / G)
    //   row_off index of this tile's first query row among the KV head's rows
    template <int QPITCH, bool QSMEM = false>
    __device__ __forceinline__ void block(uint32_t kb, const uint32_t (*qreg)[4], uint32_t qsm,
                                          int tok0, int last_q, int row_off, int L, int G,
                                          float scale_log2, int lane) {
        using PK = Pack<T>;
        constexpr int kTile = kBS * D * 2;
        const uint32_t vb = kb + kTile;
        const int quad = lane >> 2, qc = lane & 3;
        const int mat = lane >> 3, mrow = lane & 7;
        const int k_tok = (mat >> 1) * 8 + mrow, k_chk = mat & 1;
        const int v_tok = (mat & 1) * 8 + mrow, v_chk = mat >> 1;

        float sacc[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < kKSteps; ++ks) {
            uint32_t b0, b1, b2, b3;
            pa::ldmatrix_x4(kb + tile_offset(k_tok, 2 * ks + k_chk), b0, b1, b2, b3);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                if constexpr (MT == 1 && !QSMEM) {
                    a[0] = qreg[ks][0];
                    a[1] = qreg[ks][1];
                    a[2] = qreg[ks][2];
                    a[3] = qreg[ks][3];
                } else {
                    const int arow = mt * 16 + (mat & 1) * 8 + mrow;
                    const int achk = 2 * ks + (mat >> 1);
                    pa::ldmatrix_x4(qsm + arow * QPITCH + achk * 16, a[0], a[1], a[2], a[3]);
                }
                pa::mma_16816<PK::kBF16>(sacc[mt][0], a, b0, b1);
                pa::mma_16816<PK::kBF16>(sacc[mt][1], a, b2, b3);
            }
        }

        const bool need_mask = tok0 + kBS - 1 > last_q;   // block reaches past some row's bound
        uint32_t phi[MT][4], plo[MT][4];
        float alpha[MT][2];
        bool rescale = false;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = mt * 16 + quad + 8 * h;
                const int bound = min(last_q + (row_off + row) / G, L - 1);
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float v = sacc[mt][nt][2 * h + e] * scale_log2;
                        if (need_mask && tok0 + nt * 8 + 2 * qc + e > bound) v = -INFINITY;
                        sacc[mt][nt][2 * h + e] = v;
                        mx = fmaxf(mx, v);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[mt][h], mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                alpha[mt][h] = pa::ex2(m_run[mt][h] - m_use);
                m_run[mt][h] = m_new;
                float sum = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv = pa::ex2(sacc[mt][nt][2 * h + e] - m_use);
                        sacc[mt][nt][2 * h + e] = pv;
                        sum += pv;
                    }
                l_run[mt][h] = l_run[mt][h] * alpha[mt][h] + sum;
                rescale |= alpha[mt][h] != 1.f;
            }
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < kNTiles; ++nt) {
                    o[mt][nt][0] *= alpha[mt][0];
                    o[mt][nt][1] *= alpha[mt][0];
                    o[mt][nt][2] *= alpha[mt][1];
                    o[mt][nt][3] *= alpha[mt][1];
                }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            // A fragment of P (16 rows x 16 tokens) straight from the S accumulators
            float r0, r1, r2, r3, r4, r5, r6, r7;
            phi[mt][0] = PK::pack(sacc[mt][0][0], sacc[mt][0][1], r0, r1);
            phi[mt][1] = PK::pack(sacc[mt][0][2], sacc[mt][0][3], r2, r3);
            phi[mt][2] = PK::pack(sacc[mt][1][0], sacc[mt][1][1], r4, r5);
            phi[mt][3] = PK::pack(sacc[mt][1][2], sacc[mt][1][3], r6, r7);
            plo[mt][0] = PK::pack(r0, r1);
            plo[mt][1] = PK::pack(r2, r3);
            plo[mt][2] = PK::pack(r4, r5);
            plo[mt][3] = PK::pack(r6, r7);
        }

        const int valid = L - tok0;   // tokens of this block inside the context (>= 1)
#pragma unroll
        for (int nd = 0; nd < D / 16; ++nd) {
            uint32_t v0, v1, v2, v3;
            pa::ldmatrix_x4_trans(vb + tile_offset(v_tok, 2 * nd + v_chk), v0, v1, v2, v3);
            if (valid < kBS) {
                // slots past the context may hold anything (even NaN patterns): zero them
                const int t_lo = 2 * qc, t_hi = 2 * qc + 8;
                auto keep = [&](uint32_t x, int t) -> uint32_t {
                    const uint32_t lo = (t < valid) ? (x & 0xffffu) : 0u;
                    const uint32_t hi = (t + 1 < valid) ? (x & 0xffff0000u) : 0u;
                    return lo | hi;
                };
                v0 = keep(v0, t_lo);
                v2 = keep(v2, t_lo);
                v1 = keep(v1, t_hi);
                v3 = keep(v3, t_hi);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                pa::mma_16816<PK::kBF16>(o[mt][2 * nd], phi[mt], v0, v1);
                pa::mma_16816<PK::kBF16>(o[mt][2 * nd], plo[mt], v0, v1);
                pa::mma_16816<PK::kBF16>(o[mt][2 * nd + 1], phi[mt], v2, v3);
                pa::mma_16816<PK::kBF16>(o[mt][2 * nd + 1], plo[mt], v2, v3);
            }
        }
    }

    __device__ __forceinline__ void quad_sum() {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                l_run[mt][h] += __shfl_xor_sync(0xffffffffu, l_run[mt][h], 1);
                l_run[mt][h] += __shfl_xor_sync(0xffffffffu, l_run[mt][h], 2);
            }
    }
};

// Q fragments of one m-tile in registers (MT == 1): tile rows quad and quad + 8,
// i.e. query rows row_lo + quad (+ 8) of kv head g, zero at or past row_hi.
template <typename T, int D>
__device__ __forceinline__ void load_q_regs(uint32_t (*qreg)[4], const void* q, int q0, int G,
                                            int row_lo, int row_hi, int g, int num_heads,
                                            int lane) {
    const int quad = lane >> 2, qc = lane & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int row = row_lo + quad + 8 * h;
        const T* src = row < row_hi ? static_cast<const T*>(q) +
                                          ((int64_t)(q0 + row / G) * num_heads + g * G + row % G) * D
                                    : nullptr;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t lo = 0, hi = 0;
            if (src) {
                lo = __ldg(reinterpret_cast<const uint32_t*>(src + ks * 16 + 2 * qc));
                hi = __ldg(reinterpret_cast<const uint32_t*>(src + ks * 16 + 8 + 2 * qc));
            }
            qreg[ks][h] = lo;
            qreg[ks][2 + h] = hi;
        }
    }
}

// ===========================================================================
// balanced schedule (see balanced.cuh)
// ===========================================================================

template <int D, int MT, int S>
struct BalancedLayout {
    static constexpr int kStage = 2 * kBS * D * 2;
    static constexpr int kRing = S * kStage;
    static constexpr int kQPitch = D * 2 + 16;
    static constexpr int kQTile = MT > 1 ? 16 * MT * kQPitch : 0;
    __host__ __device__ static int smem_bytes(int num_seqs) {
        return pa::sched::header_bytes(num_seqs, S) + kWorkerWarps * (kRing + kQTile) + 1024;
    }
};

template <typename T, int D, int MT, int S>
__global__ void __launch_bounds__(kWorkerWarps * 32, 3)
    paged_decode_balanced_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                 const __grid_constant__ CUtensorMap tmap_v,
                                 const pa::sched::Params p) {
    using namespace pa::sched;
    using Lay = BalancedLayout<D, MT, S>;
    using PK = Pack<T>;
    constexpr int kKSteps = D / 16;
    constexpr int kNTiles = D / 8;
    constexpr int RT = 16 * MT;
    static_assert(Lay::kRing >= fold_stage_bytes(D), "the merges stage partials in the ring");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = pa::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hkv = p.num_kv_heads, G = p.group, n_seqs = p.num_seqs;
    int32_t* const cum = reinterpret_cast<int32_t*>(smem + kWorkerWarps * S * 8);
    uint8_t* const chunks = reinterpret_cast<uint8_t*>(cum + n_seqs + 1);
    const uint32_t bars = base + warp * S * 8;
    const int hdr = header_bytes(n_seqs, S);
    const uint32_t ring = base + hdr + warp * Lay::kRing;
    const uint32_t qtile = base + hdr + kWorkerWarps * Lay::kRing + warp * Lay::kQTile;

    build_prefix(cum, chunks, p);
    const int64_t B = cum[n_seqs];
    const int64_t wid = (int64_t)blockIdx.x * kWorkerWarps + warp;
    const int64_t W = share_count(p, B);
    const int64_t f0 = share_start(wid, B, W);
    const int64_t f1 = share_start(wid + 1, B, W);
    const int n = (int)(f1 - f0);
    if (lane == 0) write_merge_record(p, wid, 0, 0, 0);   // none unless set at the end
    if (wid >= W || n <= 0) return;   // the grid's last CTA may have spare warps

    if (lane == 0) {
        for (int i = 0; i < S; ++i) pa::mbar_init(bars + 8 * i, 1);
        pa::fence_barrier_init();
    }
    __syncwarp();

    // Producer side (all lanes run it; lane 0 issues): each lane keeps the TMA
    // row of virtual block (win + lane) of this share.
    uint64_t pol = 0;
    if (lane == 0) {
        pa::prefetch_tensormap(&tmap_k);
        pa::prefetch_tensormap(&tmap_v);
        pol = pa::policy_evict_first();
    }
    int win = -32, my_row = 0;
    auto refresh = [&](int wbase) {
        win = wbase;
        const int64_t f = f0 + wbase + lane;
        my_row = 0;
        if (f < f1) {
            const Pos q = locate(p, cum, chunks, f);
            int blk = __ldg(p.block_tables + (int64_t)q.s * p.max_blocks + first_block(p, q.s) +
                            q.b);
            if (blk < 0 || blk >= p.num_blocks) {
                if (p.err) atomicOr(p.err, pa::ERR_BAD_BLOCK);
                blk = 0;
            }
            my_row = (blk * hkv + q.g) * kBS;
        }
    };
    auto issue = [&](int k) {   // warp-uniform
        if (k >= win + 32) refresh(k & ~31);
        const int row = __shfl_sync(0xffffffffu, my_row, k - win);
#ifdef PA_TEST_HOOKS
        if (wid == 0 && k == g_test_skip_copy) return;   // this block's wait will run out
#endif
        if (lane == 0)
            issue_tile<D>(ring + (k % S) * Lay::kStage, bars + 8 * (k % S), &tmap_k, &tmap_v,
                          row, pol);
    };
    int issued = 0;
    for (; issued < S && issued < n; ++issued) issue(issued);

    // Consumer side: walk the share block by block, segment by segment.
    Pos cur = locate(p, cum, chunks, f0);
    int64_t seg_f = f0 - cur.b;   // virtual index of the current segment's first block
    WarpAttn<T, D, MT> st;
    uint32_t qreg[MT == 1 ? kKSteps : 1][4];
    int L = 0, r = 1, q0 = 0, rows = 0, row_off = 0, seg_b0 = cur.b, sb = 0, last_q = 0;
    bool seg_first = true;
    auto start_segment = [&]() {
        L = __ldg(p.context_lens + cur.s);
        r = query_run(p.qsl, cur.s, &q0);
        sb = first_block(p, cur.s);
        last_q = p.unmasked ? L - 1 : L - r;
        row_off = cur.c * RT;
        rows = min(RT, G * r - row_off);
        if constexpr (MT == 1) {
            load_q_regs<T, D>(qreg, p.q, q0, G, row_off, row_off + rows, cur.g, p.num_heads, lane);
        } else {
            __syncwarp();
            for (int e = lane; e < RT * (D / 8); e += 32) {
                const int row = e / (D / 8), ch = e - row * (D / 8);
                uint4 v = make_uint4(0, 0, 0, 0);
                if (row < rows) {
                    const int gr = row_off + row;
                    const T* src = static_cast<const T*>(p.q) +
                                   ((int64_t)(q0 + gr / G) * p.num_heads + cur.g * G + gr % G) * D;
                    v = __ldg(reinterpret_cast<const uint4*>(src) + ch);
                }
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                                 qtile + row * Lay::kQPitch + ch * 16),
                             "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
            __syncwarp();
        }
        st.reset();
    };
    auto finish_segment = [&](bool complete, int slot_idx, int tok_end) {
        st.quad_sum();
        const int quad = lane >> 2, qc = lane & 3;
        if (complete) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = mt * 16 + quad + 8 * h;
                    if (row >= rows) continue;
                    const int gr = row_off + row;
                    const float inv = 1.f / st.l_run[mt][h];
                    const int64_t orow = (int64_t)(q0 + gr / G) * p.num_heads + cur.g * G + gr % G;
                    const int64_t obase = orow * D;
                    if (p.lse_out && qc == 0)
                        p.lse_out[orow] = st.m_run[mt][h] + log2f(st.l_run[mt][h]);
#pragma unroll
                    for (int nt = 0; nt < kNTiles; ++nt) {
                        const float a = st.o[mt][nt][2 * h] * inv;
                        const float b = st.o[mt][nt][2 * h + 1] * inv;
                        const int64_t idx = obase + nt * 8 + 2 * qc;
                        if (p.out_f32)
                            *reinterpret_cast<float2*>(static_cast<float*>(p.out) + idx) =
                                make_float2(a, b);
                        else
                            PK::store2(static_cast<T*>(p.out) + idx, a, b);
                    }
                }
        } else {
            Slot sl(p.slots + (2 * wid + slot_idx) * (int64_t)p.slot_bytes, RT);
            if (lane == 0) {
                sl.hdr[0] = cur.s;
                sl.hdr[1] = cur.g;
                sl.hdr[2] = cur.c;
                sl.hdr[3] = (sb + seg_b0) * kBS;
                sl.hdr[4] = tok_end;
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = mt * 16 + quad + 8 * h;
                    if (row >= rows) continue;
                    if (qc == 0) {
                        sl.m[row] = st.m_run[mt][h];
                        sl.l[row] = st.l_run[mt][h];
                    }
#pragma unroll
                    for (int nt = 0; nt < kNTiles; ++nt)
                        *reinterpret_cast<float2*>(sl.o + (int64_t)row * D + nt * 8 + 2 * qc) =
                            make_float2(st.o[mt][nt][2 * h], st.o[mt][nt][2 * h + 1]);
                }
        }
    };
    start_segment();

    int consumed = 0;
    for (int k = 0; k < n; ++k) {
        if (!pa::mbar_wait(bars + 8 * (k % S), (k / S) & 1, p.err, pa::ERR_WAIT_FULL)) break;
        consumed = k + 1;
        st.template block<Lay::kQPitch>(ring + (k % S) * Lay::kStage, qreg, qtile,
                                        (sb + cur.b) * kBS, last_q, row_off, L, G, p.scale_log2,
                                        lane);
        __syncwarp();
        if (issued < n) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(issued);
            ++issued;
        }
        ++cur.b;
        const bool seg_done = cur.b == cur.nbs;
        if (seg_done || k == n - 1) {
            const bool whole = seg_b0 == 0 && seg_done;
            finish_segment(whole, seg_first ? 0 : 1, min((sb + cur.b) * kBS, L));
            if (k == n - 1) {
                if (lane == 0 && !p.arrivals)
                    record_last_segment(p, wid, f1, B, seg_done, seg_b0,
                                        cur.nbs - cur.b, seg_first, q0, rows);
                break;
            }
            next_segment(p, cur, cum, chunks);
            seg_f = f0 + k + 1;
            seg_b0 = 0;
            seg_first = false;
            start_segment();
        }
    }
    // drain: no copy of this warp may still be in flight when it exits
    bool drained = true;
    for (int k = consumed; k < issued; ++k)
        if (!pa::mbar_wait(bars + 8 * (k % S), (k / S) & 1, p.err, pa::ERR_WAIT_DRAIN)) {
            drained = false;
            break;
        }
    // the cut segments' pieces of this share, merged by whichever piece is
    // last (after the stream, where the accumulators are no longer live and
    // the ring is free to stage partials in): the first segment if it began
    // before the share and ended inside it (its position found again), and
    // the last if the share did not hold it whole
    if (p.arrivals && consumed == n && drained) {
        const Pos h = locate(p, cum, chunks, f0);
        const bool has_h = h.b > 0 && h.nbs - h.b < n;        // ends in this share: wb = wid
        const bool has_t = !(seg_b0 == 0 && cur.b == cur.nbs);
        CutPiece hp{}, tp{};
        if (has_h) {
            int hq0;
            const int hr = query_run(p.qsl, h.s, &hq0);
            hp = cut_piece(p, B, wid, f0 - h.b, h.nbs - h.b, h.nbs, h.s, h.g, h.c, hq0,
                           min(RT, G * hr - h.c * RT), -1, 0, wid);
        }
        if (has_t)   // starts in this share (wa = wid) unless it began before it
            tp = cut_piece(p, B, wid, seg_f, cur.b - seg_b0, cur.nbs, cur.s, cur.g, cur.c, q0,
                           rows, seg_f >= f0 ? wid : -1, f0, -1);
        const int done = arrive_pair(p, hp, has_h, tp, has_t, lane);
        if (done & 1) merge_cut<T, D>(p, B, hp, ring, lane);
        if (done & 2) merge_cut<T, D>(p, B, tp, ring, lane);
    }
}

// ---------------------------------------------------------------------------
// Balanced schedule with 64-row tiles (more than 16 query rows per KV head:
// large GQA groups with verify runs, MQA, the prefix phase of shared-prefix
// decode). One CTA per share: warp 0 streams the K/V tiles of the share's
// blocks through a ring the CTA shares, and warp w computes tile rows
// 16w .. 16w + 15 against every block, so each block is read once for up to
// 64 rows. A stage is refilled when all four warps have released it (an
// mbarrier with four arrivals); warps with no rows in a segment still wait
// for every block and release it, which keeps them in step with the ring.
// ---------------------------------------------------------------------------

constexpr int kRowsTile = 64;
constexpr int kRowsStages = 4;   // 4 CTAs of ~52 KB shared memory per SM

template <int D, int S>
struct RowsLayout {
    static constexpr int kStage = 2 * kBS * D * 2;
    static constexpr int kRing = S * kStage;
    static constexpr int kQPitch = D * 2 + 16;          // padded: conflict-free ldmatrix
    static constexpr int kQTile = 16 * kQPitch;         // one warp's 16 query rows
    __host__ __device__ static int smem_bytes(int num_seqs) {
        return pa::sched::header_bytes(num_seqs, S) + kRing + kWorkerWarps * kQTile + 1024;
    }
};

template <typename T, int D, int S>
__global__ void __launch_bounds__(kWorkerWarps * 32, 4)
    paged_decode_rows_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v,
                             const pa::sched::Params p) {
    using namespace pa::sched;
    using Lay = RowsLayout<D, S>;
    using PK = Pack<T>;
    constexpr int kNTiles = D / 8;
    constexpr int RT = kRowsTile;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = pa::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hkv = p.num_kv_heads, G = p.group, n_seqs = p.num_seqs;
    int32_t* const cum = reinterpret_cast<int32_t*>(smem + kWorkerWarps * S * 8);
    uint8_t* const chunks = reinterpret_cast<uint8_t*>(cum + n_seqs + 1);
    const uint32_t full = base, empty = base + 8 * S;
    const uint32_t ring = base + header_bytes(n_seqs, S);   // 1024-aligned
    const uint32_t qtile = ring + Lay::kRing + warp * Lay::kQTile;

    build_prefix(cum, chunks, p);
    const int64_t B = cum[n_seqs];
    const int64_t wid = blockIdx.x;                          // one share per CTA
    const int64_t W = share_count(p, B);
    const int64_t f0 = share_start(wid, B, W);
    const int64_t f1 = share_start(wid + 1, B, W);
    const int n = (int)(f1 - f0);
    if (threadIdx.x == 0) write_merge_record(p, wid, 0, 0, 0);   // none unless set at the end
    if (wid >= W || n <= 0) return;                  // uniform over the CTA

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            pa::mbar_init(full + 8 * i, 1);
            pa::mbar_init(empty + 8 * i, kWorkerWarps);
        }
        pa::fence_barrier_init();
        pa::prefetch_tensormap(&tmap_k);
        pa::prefetch_tensormap(&tmap_v);
    }
    __syncthreads();

    // Producer (warp 0): each lane keeps the TMA row of virtual block win +
    // lane and whether that block is read by one row chunk only (then it is
    // loaded with an evict-first hint; blocks that further chunks read again
    // stay at normal priority).
    uint64_t pol_once = 0, pol_again = 0;
    if (warp == 0 && lane == 0) {
        pol_once = pa::policy_evict_first();
        pol_again = pa::policy_evict_normal();
    }
    int win = -32, my_row = 0, my_once = 1;
    auto refresh = [&](int wbase) {
        win = wbase;
        const int64_t f = f0 + wbase + lane;
        my_row = 0;
        my_once = 1;
        if (f < f1) {
            const Pos q = locate(p, cum, chunks, f);
            int blk = __ldg(p.block_tables + (int64_t)q.s * p.max_blocks + first_block(p, q.s) +
                            q.b);
            if (blk < 0 || blk >= p.num_blocks) {
                if (p.err) atomicOr(p.err, pa::ERR_BAD_BLOCK);
                blk = 0;
            }
            my_row = (blk * hkv + q.g) * kBS;
            my_once = q.C == 1;
        }
    };
    auto issue = [&](int k) {   // warp 0, warp-uniform
        if (k >= win + 32) refresh(k & ~31);
        const int row = __shfl_sync(0xffffffffu, my_row, k - win);
        const int once = __shfl_sync(0xffffffffu, my_once, k - win);
        if (lane == 0)
            issue_tile<D>(ring + (k % S) * Lay::kStage, full + 8 * (k % S), &tmap_k, &tmap_v, row,
                          once ? pol_once : pol_again);
    };
    int issued = 0, consumed = 0;
    if (warp == 0)
        for (; issued < S && issued < n; ++issued) issue(issued);

    Pos cur = locate(p, cum, chunks, f0);
    // Q stays in shared memory (this warp's 16 rows) and is read with ldmatrix
    // per block: keeping the fragments in registers would cost 32 registers a
    // thread and one CTA per SM.
    WarpAttn<T, D, 1> st;
    int L = 0, r = 1, q0 = 0, rows = 0, row_off = 0, seg_b0 = cur.b, sb = 0, last_q = 0;
    bool seg_first = true, busy = false;
    auto start_segment = [&]() {
        L = __ldg(p.context_lens + cur.s);
        r = query_run(p.qsl, cur.s, &q0);
        sb = first_block(p, cur.s);
        last_q = p.unmasked ? L - 1 : L - r;
        row_off = cur.c * RT;
        rows = min(RT, G * r - row_off);
        busy = 16 * warp < rows;
        if (busy) {
            __syncwarp();
            for (int e = lane; e < 16 * (D / 8); e += 32) {
                const int row = e / (D / 8), ch = e - row * (D / 8);
                const int tr = 16 * warp + row;               // tile row
                uint4 v = make_uint4(0, 0, 0, 0);
                if (tr < rows) {
                    const int gr = row_off + tr;
                    const T* src = static_cast<const T*>(p.q) +
                                   ((int64_t)(q0 + gr / G) * p.num_heads + cur.g * G + gr % G) * D;
                    v = __ldg(reinterpret_cast<const uint4*>(src) + ch);
                }
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                                 qtile + row * Lay::kQPitch + ch * 16),
                             "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
            __syncwarp();
        }
        st.reset();
    };
    auto finish_segment = [&](bool complete, int slot_idx, int tok_end) {
        Slot sl(p.slots + (2 * wid + slot_idx) * (int64_t)p.slot_bytes, RT);
        if (!complete && warp == 0 && lane == 0) {
            sl.hdr[0] = cur.s;
            sl.hdr[1] = cur.g;
            sl.hdr[2] = cur.c;
            sl.hdr[3] = (sb + seg_b0) * kBS;
            sl.hdr[4] = tok_end;
        }
        if (!busy) return;
        st.quad_sum();
        const int quad = lane >> 2, qc = lane & 3;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = 16 * warp + quad + 8 * h;          // tile row
            if (row >= rows) continue;
            if (complete) {
                const int gr = row_off + row;
                const float inv = 1.f / st.l_run[0][h];
                const int64_t orow = (int64_t)(q0 + gr / G) * p.num_heads + cur.g * G + gr % G;
                if (p.lse_out && qc == 0) p.lse_out[orow] = st.m_run[0][h] + log2f(st.l_run[0][h]);
#pragma unroll
                for (int nt = 0; nt < kNTiles; ++nt) {
                    const float a = st.o[0][nt][2 * h] * inv;
                    const float b = st.o[0][nt][2 * h + 1] * inv;
                    const int64_t idx = orow * D + nt * 8 + 2 * qc;
                    if (p.out_f32)
                        *reinterpret_cast<float2*>(static_cast<float*>(p.out) + idx) =
                            make_float2(a, b);
                    else
                        PK::store2(static_cast<T*>(p.out) + idx, a, b);
                }
            } else {
                if (qc == 0) {
                    sl.m[row] = st.m_run[0][h];
                    sl.l[row] = st.l_run[0][h];
                }
#pragma unroll
                for (int nt = 0; nt < kNTiles; ++nt)
                    *reinterpret_cast<float2*>(sl.o + (int64_t)row * D + nt * 8 + 2 * qc) =
                        make_float2(st.o[0][nt][2 * h], st.o[0][nt][2 * h + 1]);
            }
        }
    };
    start_segment();

    for (int k = 0; k < n; ++k) {
        const int stg = k % S;
        if (!__all_sync(0xffffffffu,
                        pa::mbar_wait(full + 8 * stg, (k / S) & 1, p.err, pa::ERR_WAIT_FULL)))
            break;
        if (warp == 0) consumed = k + 1;
        if (busy)
            st.template block<Lay::kQPitch, true>(ring + stg * Lay::kStage, nullptr, qtile,
                                                  (sb + cur.b) * kBS, last_q, row_off + 16 * warp,
                                                  L, G, p.scale_log2, lane);
        __syncwarp();
        if (lane == 0) pa::mbar_arrive(empty + 8 * stg);     // this warp is done with the stage
        // warp 0 refills the stage block k - 1 used once every warp has released it
        if (warp == 0 && k >= 1 && k - 1 + S < n) {
            const int kp = k - 1;
            if (!__all_sync(0xffffffffu, pa::mbar_wait(empty + 8 * (kp % S), (kp / S) & 1, p.err,
                                                       pa::ERR_WAIT_EMPTY)))
                break;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(kp + S);
            ++issued;
        }
        ++cur.b;
        const bool seg_done = cur.b == cur.nbs;
        if (seg_done || k == n - 1) {
            finish_segment(seg_b0 == 0 && seg_done, seg_first ? 0 : 1,
                           min((sb + cur.b) * kBS, L));
            if (k == n - 1) {
                if (threadIdx.x == 0)
                    record_last_segment(p, wid, f1, B, seg_done, seg_b0,
                                        cur.nbs - cur.b, seg_first, q0, rows);
                break;
            }
            next_segment(p, cur, cum, chunks);
            seg_b0 = 0;
            seg_first = false;
            start_segment();
        }
    }
    // no copy may still be in flight when the CTA exits (this wait ignores the
    // abort bits: it ends when the copy lands or after its own time limit)
    if (warp == 0 && lane == 0)
        for (int k = consumed; k < issued; ++k)
            if (!pa::mbar_wait(full + 8 * (k % S), (k / S) & 1, nullptr, 0)) {
                if (p.err) atomicOr(p.err, pa::ERR_WAIT_DRAIN);
                break;
            }
}

// ===========================================================================
// partitioned schedule
// ===========================================================================

struct DecodeParams {
    void* out;
    const void* q;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* qsl;
    float* o_part;
    float* m_part;
    float* l_part;
    unsigned int* err;
    int max_blocks;
    int num_heads;
    int num_kv_heads;
    int group;             // q heads per kv head
    int partition_size;    // tokens
    int num_partitions;    // P (workspace stride)
    int num_blocks;
    float scale_log2;      // softmax scale * log2(e)
    int out_f32;
};

template <int D, int MT, int STAGES>
struct Layout {
    static constexpr int kTileBytes = kBS * D * 2;      // one K (or V) tile
    static constexpr int kStageBytes = 2 * kTileBytes;  // K then V
    static constexpr int kRingBytes = STAGES * kStageBytes;
    static constexpr int kRows = 16 * MT;
    // merge scratch (reuses the ring): per warp m[kRows], l[kRows], O[kRows][D]
    static constexpr int kMergeBytes = kConsumerWarps * kRows * (D + 2) * 4;
    static constexpr int kQPitch = D * 2 + 16;          // padded row pitch of the Q tile (MT > 1)
    static constexpr int kQBytes = MT > 1 ? kRows * kQPitch : 0;
    static constexpr int kBodyBytes = (kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes);
    static constexpr int kQOffset = kBodyBytes;
    static constexpr int kBarOffset = kQOffset + ((kQBytes + 15) / 16) * 16;
    static constexpr int kBlkOffset = kBarOffset + 2 * STAGES * 8;
    static constexpr int kSmemBytes = kBlkOffset + kMaxPartBlocks * 4 + 1024;  // + alignment slack
};

template <typename T, int D, int MT, int STAGES>
__global__ void __launch_bounds__(kThreads)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
    using Lay = Layout<D, MT, STAGES>;
    using PK = Pack<T>;
    constexpr int kKSteps = D / 16;
    constexpr int kNTiles = D / 8;

    const int part = blockIdx.x;
    const int g = blockIdx.y;
    const int s = blockIdx.z;
    pa::grid_dependents_launch();
    pa::grid_dependency_wait();
    const int L = __ldg(p.context_lens + s);
    const int t_begin = part * p.partition_size;
    if (t_begin >= L) return;
    const int t_end = min(L, t_begin + p.partition_size);
    const int nblk = (t_end - t_begin + kBS - 1) / kBS;
    const int blk0 = t_begin / kBS;
    int q0, r;
    if (p.qsl) {
        q0 = __ldg(p.qsl + s);
        r = __ldg(p.qsl + s + 1) - q0;
    } else {
        q0 = s;
        r = 1;
    }
    const int G = p.group;
    const int R = G * r;          // query rows served by this CTA
    const bool single = L <= p.partition_size;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = pa::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;          // 1024-aligned for the swizzle atom
    uint8_t* const smem = smem_raw + (base - raw);
    const uint32_t bar_full = base + Lay::kBarOffset;      // STAGES x 8 bytes
    const uint32_t bar_empty = bar_full + STAGES * 8;
    int32_t* const s_blk = reinterpret_cast<int32_t*>(smem + Lay::kBlkOffset);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // physical block ids of this partition, range-checked once
    for (int i = threadIdx.x; i < nblk; i += kThreads) {
        int b = __ldg(p.block_tables + (int64_t)s * p.max_blocks + blk0 + i);
        if (b < 0 || b >= p.num_blocks) {
            if (p.err) atomicOr(p.err, pa::ERR_BAD_BLOCK);
            b = 0;
        }
        s_blk[i] = b;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            pa::mbar_init(bar_full + 8 * i, 1);
            pa::mbar_init(bar_empty + 8 * i, 1);
        }
        pa::fence_barrier_init();
    }
    if (MT > 1) {
        // Q tile [kRows][D] (padded pitch) for ldmatrix; rows >= R are zero
        for (int e = threadIdx.x; e < Lay::kRows * (D / 8); e += kThreads) {
            const int row = e / (D / 8), ch = e % (D / 8);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (row < R) {
                const T* src = static_cast<const T*>(p.q) +
                               ((int64_t)(q0 + row / G) * p.num_heads + g * G + row % G) * D;
                v = __ldg(reinterpret_cast<const uint4*>(src) + ch);
            }
            *reinterpret_cast<uint4*>(smem + Lay::kQOffset + row * Lay::kQPitch + ch * 16) = v;
        }
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            pa::prefetch_tensormap(&tmap_k);
            pa::prefetch_tensormap(&tmap_v);
            const uint64_t pol = pa::policy_evict_first();
            int issued = 0;
            for (int i = 0; i < nblk; ++i) {
                const int st = i % STAGES;
                const int n = i / STAGES;
                if (n > 0 && !pa::mbar_wait(bar_empty + 8 * st, (n - 1) & 1, p.err,
                                            pa::ERR_WAIT_EMPTY))
                    break;
                const int row = (s_blk[i] * p.num_kv_heads + g) * kBS;
                issue_tile<D>(base + st * Lay::kStageBytes, bar_full + 8 * st, &tmap_k, &tmap_v,
                              row, pol);
                issued = i + 1;
            }
            // drain: no copy may be in flight when the CTA exits
            for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
                if (!pa::mbar_wait(bar_full + 8 * (i % STAGES), (i / STAGES) & 1, p.err,
                                   pa::ERR_WAIT_DRAIN))
                    break;
        }
        return;
    }

    // ------------------------------- consumers -------------------------------
    const int quad = lane >> 2;
    const int qc = lane & 3;
    uint32_t qreg[MT == 1 ? kKSteps : 1][4];
    if constexpr (MT == 1) load_q_regs<T, D>(qreg, p.q, q0, G, 0, R, g, p.num_heads, lane);
    WarpAttn<T, D, MT> st;
    st.reset();

    bool ok = true;
    for (int i = warp; i < nblk; i += kConsumerWarps) {
        const int stg = i % STAGES;
        if (!pa::mbar_wait(bar_full + 8 * stg, (i / STAGES) & 1, p.err, pa::ERR_WAIT_FULL)) {
            ok = false;
            break;
        }
        st.template block<Lay::kQPitch>(base + stg * Lay::kStageBytes, qreg, base + Lay::kQOffset,
                                        t_begin + i * kBS, L - r, 0, L, G, p.scale_log2, lane);
        __syncwarp();
        if (lane == 0) pa::mbar_arrive(bar_empty + 8 * stg);
    }

    // ---- merge the consumer warps through shared memory (the ring is free now) ----
    pa::named_barrier_sync(1, kConsumerWarps * 32);
    constexpr int kRows = Lay::kRows;
    float* const m_sh = reinterpret_cast<float*>(smem);                        // [W][kRows]
    float* const l_sh = m_sh + kConsumerWarps * kRows;                         // [W][kRows]
    float* const o_sh = l_sh + kConsumerWarps * kRows;                         // [W][kRows][D]
    st.quad_sum();
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = mt * 16 + quad + 8 * h;
            if (qc == 0) {
                m_sh[warp * kRows + row] = ok ? st.m_run[mt][h] : -INFINITY;
                l_sh[warp * kRows + row] = ok ? st.l_run[mt][h] : 0.f;
            }
#pragma unroll
            for (int nt = 0; nt < kNTiles; ++nt) {
                float2 v = make_float2(st.o[mt][nt][2 * h], st.o[mt][nt][2 * h + 1]);
                *reinterpret_cast<float2*>(o_sh + ((size_t)warp * kRows + row) * D + nt * 8 +
                                           2 * qc) = v;
            }
        }
    }
    pa::named_barrier_sync(1, kConsumerWarps * 32);
    const int tid = threadIdx.x;
    for (int e = tid; e < R * D; e += kConsumerWarps * 32) {
        const int row = e / D, col = e - (e / D) * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, m_sh[w * kRows + row]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float tot = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float wt = exp2f(m_sh[w * kRows + row] - Mu);
            tot += wt * l_sh[w * kRows + row];
            acc += wt * o_sh[((size_t)w * kRows + row) * D + col];
        }
        const int qi = q0 + row / G;
        const int h = g * G + row % G;
        if (single) {
            const int64_t idx = ((int64_t)qi * p.num_heads + h) * D + col;
            const float val = acc / tot;
            if (p.out_f32) static_cast<float*>(p.out)[idx] = val;
            else PK::store(static_cast<T*>(p.out) + idx, val);
        } else {
            const int64_t prow = ((int64_t)qi * p.num_heads + h) * p.num_partitions + part;
            p.o_part[prow * D + col] = tot > 0.f ? acc / tot : 0.f;
            if (col == 0) {
                p.m_part[prow] = M;
                p.l_part[prow] = tot;
            }
        }
    }
}

// Log-sum-exp merge of the partitions: out = sum_p w_p o_p / sum_p w_p with
// w_p = l_p 2^(m_p - M), M = max_p m_p (m in base-2 units). grid =
// (ceil(H / 4), num_seqs); one warp per (sequence, q head), all its query rows.
template <typename T, int D>
__global__ void __launch_bounds__(128)
    split_kv_reduce_kernel(void* out, int out_f32, const float* __restrict__ o_part,
                           const float* __restrict__ m_part, const float* __restrict__ l_part,
                           const int32_t* __restrict__ context_lens,
                           const int32_t* __restrict__ qsl, int num_heads, int num_partitions,
                           int partition_size) {
    constexpr int EPL = D / 32;
    pa::grid_dependency_wait();
    const int s = blockIdx.y;
    const int h = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (h >= num_heads) return;
    const int L = __ldg(context_lens + s);
    const int np = (L + partition_size - 1) / partition_size;
    if (np <= 1) return;   // written directly by the decode kernel
    int q0, r;
    if (qsl) {
        q0 = __ldg(qsl + s);
        r = __ldg(qsl + s + 1) - q0;
    } else {
        q0 = s;
        r = 1;
    }
    for (int qi = q0; qi < q0 + r; ++qi) {
        const int64_t prow = ((int64_t)qi * num_heads + h) * num_partitions;
        float M = -INFINITY;
        for (int pp = lane; pp < np; pp += 32) M = fmaxf(M, __ldg(m_part + prow + pp));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float Mu = M == -INFINITY ? 0.f : M;
        float acc[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
        float tot = 0.f;
        for (int pp = 0; pp < np; ++pp) {
            const float l = __ldg(l_part + prow + pp);
            if (l <= 0.f) continue;
            const float w = l * exp2f(__ldg(m_part + prow + pp) - Mu);
            tot += w;
            const float* src = o_part + (prow + pp) * D + lane * EPL;
            if constexpr (EPL == 4) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(src));
                acc[0] += w * v.x;
                acc[1] += w * v.y;
                acc[2] += w * v.z;
                acc[3] += w * v.w;
            } else {
                const float2 v = __ldg(reinterpret_cast<const float2*>(src));
                acc[0] += w * v.x;
                acc[1] += w * v.y;
            }
        }
        const float inv = 1.f / tot;
        const int64_t obase = ((int64_t)qi * num_heads + h) * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const float val = acc[e] * inv;
            if (out_f32) static_cast<float*>(out)[obase + e] = val;
            else Pack<T>::store(static_cast<T*>(out) + obase + e, val);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------



constexpr int kBalancedStages = 2;

template <typename T, int D, int MT>
pa_status launch_partitioned(const pa::DecodeArgs& a, const CUtensorMap& mk,
                             const CUtensorMap& mv, const DecodeParams& prm) {
    constexpr int STAGES = 8;
    using Lay = Layout<D, MT, STAGES>;
    auto kern = paged_decode_kernel<T, D, MT, STAGES>;
    static bool attr_set = false;   // per instantiation; benign race (idempotent)
    if (!attr_set) {
        if (pa_status s = pa::cuda_status(
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Lay::kSmemBytes),
                "decode: set shared memory size"))
            return s;
        attr_set = true;
    }
    dim3 grid(a.num_partitions, a.num_kv_heads, a.num_seqs);
    if (pa_status s = pa::cuda_status(
            pa::launch_pdl(kern, grid, dim3(kThreads), Lay::kSmemBytes, a.stream, mk, mv, prm),
            "decode launch"))
        return s;
    if (a.num_partitions > 1) {
        dim3 rgrid((a.num_heads + 3) / 4, a.num_seqs);
        if (pa_status s = pa::cuda_status(
                pa::launch_pdl(split_kv_reduce_kernel<T, D>, rgrid, dim3(128), 0, a.stream,
                               a.out, (int)(a.out_dtype == PA_F32), a.o_part, a.m_part, a.l_part,
                               a.context_lens, a.query_start_loc, a.num_heads, a.num_partitions,
                               a.partition_size),
                "split-KV reduce launch"))
            return s;
    }
    return PA_OK;
}

// Resident CTAs per SM for a kernel and shared-memory size, and the SM count, per device.
struct Residency {
    std::mutex mu;
    struct E {
        const void* fn;
        int smem, device, ctas, sms;
    } e[64];
    int n = 0;
    pa_status get(const void* fn, int smem, int* ctas, int* sms) {
        int dev = 0;
        if (pa_status s = pa::cuda_status(cudaGetDevice(&dev), "cudaGetDevice")) return s;
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n; ++i)
            if (e[i].fn == fn && e[i].smem == smem && e[i].device == dev) {
                *ctas = e[i].ctas;
                *sms = e[i].sms;
                return PA_OK;
            }
        int c = 0, m = 0;
        if (pa_status s = pa::cuda_status(
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, fn, kWorkerWarps * 32, smem),
                "occupancy query"))
            return s;
        if (pa_status s = pa::cuda_status(
                cudaDeviceGetAttribute(&m, cudaDevAttrMultiProcessorCount, dev), "SM count"))
            return s;
        if (n < 64) e[n++] = E{fn, smem, dev, c, m};
        *ctas = c;
        *sms = m;
        return PA_OK;
    }
};
Residency g_residency;

template <typename T, int D, int MT>
pa_status launch_balanced(const pa::DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                          pa::sched::Params prm) {
    constexpr int S = kBalancedStages;
    using Lay = BalancedLayout<D, MT, S>;
    auto kern = paged_decode_balanced_kernel<T, D, MT, S>;
    const int smem = Lay::smem_bytes(a.num_seqs);
    static bool attr_set = false;   // per instantiation and process; benign race (idempotent)
    if (!attr_set) {
        // the largest size any call of this instantiation can ask for
        if (pa_status s = pa::cuda_status(
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Lay::smem_bytes(pa::kBalancedMaxSeqs)),
                "decode: set shared memory size"))
            return s;
        attr_set = true;
    }
    int ctas = 0, sms = 0;
    if (pa_status s = g_residency.get(reinterpret_cast<const void*>(kern), smem, &ctas, &sms))
        return s;
    if (ctas < 1) return pa::fail(PA_ERR_UNSUPPORTED, "decode kernel does not fit on an SM");
    const pa::BalancedShape shape = pa::balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads,
                                                       a.head_dim, a.max_q_len, a.max_context_len);
    int64_t workers = std::min<int64_t>((int64_t)ctas * sms * kWorkerWarps, shape.workers);
    if (a.max_workers > 0) workers = std::min<int64_t>(workers, a.max_workers);
    prm.workers = (int)workers;
    // The in-kernel merge pays off when shares are long. When a call can
    // hold fewer than 8 blocks per worker (a small call), the merges'
    // round trips at the end of each short stream cost more than the
    // reduce kernel.
    if (shape.virtual_blocks < 8 * workers) prm.arrivals = nullptr;
    const int grid = (int)((workers + kWorkerWarps - 1) / kWorkerWarps);
    if (pa_status s = pa::cuda_status(
            pa::launch_pdl(kern, dim3(grid), dim3(kWorkerWarps * 32), smem, a.stream, mk, mv, prm),
            "decode launch"))
        return s;
    if (prm.arrivals) return PA_OK;   // cut segments merged by the decode kernel
    const int row_slots = (int)std::min<int64_t>(shape.rows_per_tile, (int64_t)(a.num_heads / a.num_kv_heads) *
                                                          a.max_q_len);
    return pa::cuda_status(pa::sched::launch_segment_reduce<T, D>(prm, (int)shape.max_chunks,
                                                                    row_slots, a.stream),
                           "segment reduce launch");
}

template <typename T, int D>
pa_status launch_rows(const pa::DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                      pa::sched::Params prm) {
    constexpr int S = kRowsStages;
    using Lay = RowsLayout<D, S>;
    auto kern = paged_decode_rows_kernel<T, D, S>;
    const int smem = Lay::smem_bytes(a.num_seqs);
    static bool attr_set = false;   // per instantiation and process; benign race (idempotent)
    if (!attr_set) {
        if (pa_status s = pa::cuda_status(
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Lay::smem_bytes(pa::kBalancedMaxSeqs)),
                "decode: set shared memory size"))
            return s;
        attr_set = true;
    }
    int ctas = 0, sms = 0;
    if (pa_status s = g_residency.get(reinterpret_cast<const void*>(kern), smem, &ctas, &sms))
        return s;
    if (ctas < 1) return pa::fail(PA_ERR_UNSUPPORTED, "decode kernel does not fit on an SM");
    const pa::BalancedShape shape = pa::balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads,
                                                       a.head_dim, a.max_q_len, a.max_context_len);
    const int64_t workers = std::min<int64_t>((int64_t)ctas * sms, shape.workers);
    prm.workers = (int)workers;
    prm.arrivals = nullptr;   // this kernel leaves the merges to the reduce kernel
    if (pa_status s = pa::cuda_status(
            pa::launch_pdl(kern, dim3((unsigned)workers), dim3(kWorkerWarps * 32), smem, a.stream,
                           mk, mv, prm),
            "decode launch"))
        return s;
    const int row_slots = (int)std::min<int64_t>(kRowsTile, (int64_t)(a.num_heads / a.num_kv_heads) *
                                                          a.max_q_len);
    return pa::cuda_status(pa::sched::launch_segment_reduce<T, D>(prm, (int)shape.max_chunks,
                                                                    row_slots, a.stream),
                           "segment reduce launch");
}

template <typename T>
pa_status launch_dtype(const pa::DecodeArgs& a, int mt, const CUtensorMap& mk,
                       const CUtensorMap& mv, const DecodeParams& prm,
                       const pa::sched::Params& bprm) {
    if (a.partition_size == 0) {
        // 16-row tiles: one warp per share; larger tiles: one CTA per share
        if (a.head_dim == 128)
            return bprm.rows_per_tile == 16 ? launch_balanced<T, 128, 1>(a, mk, mv, bprm)
                                            : launch_rows<T, 128>(a, mk, mv, bprm);
        return bprm.rows_per_tile == 16 ? launch_balanced<T, 64, 1>(a, mk, mv, bprm)
                                        : launch_rows<T, 64>(a, mk, mv, bprm);
    }
    if (a.head_dim == 128)
        return mt == 1 ? launch_partitioned<T, 128, 1>(a, mk, mv, prm)
                       : launch_partitioned<T, 128, 2>(a, mk, mv, prm);
    return mt == 1 ? launch_partitioned<T, 64, 1>(a, mk, mv, prm)
                   : launch_partitioned<T, 64, 2>(a, mk, mv, prm);
}

}  // namespace

namespace pa {

pa_status launch_decode_int8(const DecodeArgs& a);
pa_status launch_decode_fp8(const DecodeArgs& a);
bool prefill_tc_applies(const DecodeArgs& a);
pa_status launch_prefill_tc(const DecodeArgs& a);
bool prefix_tc_applies(const DecodeArgs& a);
pa_status launch_prefix_tc(const DecodeArgs& a);

pa_status launch_decode(const DecodeArgs& a) {
    if ((a.ctx_start || a.lse_out || a.unmasked) &&
        (a.kv_dtype == PA_INT8 || a.kv_dtype == PA_FP8_E4M3 || a.partition_size))
        return fail(PA_ERR_UNSUPPORTED,
                    "token offsets, log-sum-exp output and unmasked rows need a 16-bit cache and "
                    "the balanced schedule");
    if (a.kv_dtype == PA_INT8) return launch_decode_int8(a);
    if (a.kv_dtype == PA_FP8_E4M3) return launch_decode_fp8(a);
    if (prefill_tc_applies(a)) return launch_prefill_tc(a);
    if (prefix_tc_applies(a)) return launch_prefix_tc(a);
    if (a.partition_size > kMaxPartBlocks * kBS)
        return fail(PA_ERR_UNSUPPORTED, "partition_size %d > %d", a.partition_size,
                    kMaxPartBlocks * kBS);
    const int G = a.num_heads / a.num_kv_heads;
    const int64_t rows = (int64_t)G * a.max_q_len;
    int mt = rows > 16 ? 2 : 1;
    if (a.partition_size > 0 && rows > 32)
        return fail(PA_ERR_UNSUPPORTED,
                    "%lld query rows per KV head (q heads per KV head x max_q_len) > 32 with "
                    "fixed partitions; use partition_size 0", (long long)rows);
    if (a.partition_size == 0)
        if (pa_status s = balanced_check(a)) return s;
    CUtensorMap mk, mv;
    if (a.head_dim == 128) {
        if (pa_status s = cache_tensor_map_tile(&mk, a.k_cache, a.num_blocks, a.num_kv_heads))
            return s;
        if (pa_status s = cache_tensor_map_tile(&mv, a.v_cache, a.num_blocks, a.num_kv_heads))
            return s;
    } else {
        if (pa_status s = cache_tensor_map(&mk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 2))
            return s;
        if (pa_status s = cache_tensor_map(&mv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 2))
            return s;
    }
    DecodeParams prm{};
    prm.out = a.out;
    prm.q = a.q;
    prm.block_tables = a.block_tables;
    prm.context_lens = a.context_lens;
    prm.qsl = a.query_start_loc;
    prm.o_part = a.o_part;
    prm.m_part = a.m_part;
    prm.l_part = a.l_part;
    prm.err = device_error_word();
    prm.max_blocks = a.max_blocks_per_seq;
    prm.num_heads = a.num_heads;
    prm.num_kv_heads = a.num_kv_heads;
    prm.group = G;
    prm.partition_size = a.partition_size;
    prm.num_partitions = a.num_partitions;
    prm.num_blocks = a.num_blocks;
    prm.scale_log2 = a.scale * kLog2e;
    prm.out_f32 = a.out_dtype == PA_F32;
    const BalancedShape shape = balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads,
                                               a.head_dim, a.max_q_len, a.max_context_len);
    pa::sched::Params b{};
    b.out = a.out;
    b.q = a.q;
    b.block_tables = a.block_tables;
    b.context_lens = a.context_lens;
    b.qsl = a.query_start_loc;
    b.cum_out = static_cast<int32_t*>(a.slots);
    b.slots = static_cast<uint8_t*>(a.slots) + shape.cum_bytes;
    b.err = prm.err;
    b.max_blocks = a.max_blocks_per_seq;
    b.num_heads = a.num_heads;
    b.num_kv_heads = a.num_kv_heads;
    b.group = G;
    b.num_seqs = a.num_seqs;
    b.num_blocks = a.num_blocks;
    b.rows_per_tile = shape.rows_per_tile;
    b.slot_bytes = (int)shape.slot_bytes;
    b.scale_log2 = prm.scale_log2;
    b.out_f32 = prm.out_f32;
    b.ctx_start = a.ctx_start;
    b.lse_out = a.lse_out;
    b.unmasked = a.unmasked;
    b.arrivals = a.arrivals;
    if (a.kv_dtype == PA_BF16) return launch_dtype<__nv_bfloat16>(a, mt, mk, mv, prm, b);
    return launch_dtype<__half>(a, mt, mk, mv, prm, b);
}

}  // namespace pa
