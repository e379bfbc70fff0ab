// Paged decode attention for F16/BF16 caches, and the split-KV reduce.
//
// What it computes: "KV Cache ... PagedAttention" (devpress.csdn.net) §二,
// softmax(Q K^T / sqrt(d)) V, over the keys a sequence holds in its blocks
// (§七: the block table maps logical block b to a physical block); "cs336
// lecture 10", decode workflow: the new token's q against every cached K,
// weighted sum of the cached V; GQA/MQA from the same lecture: the q heads
// of one group share one KV head, so one KV read serves the whole group.
//
// How (this library's design for sm_103a):
//   * grid = (partition, kv head, sequence). A CTA owns one partition of one
//     sequence's keys for one KV head and every query row that reads that KV
//     head: G q heads x r query tokens (r > 1 for speculative verify runs).
//   * One producer warp streams the partition's 16-token K and V tiles into
//     a ring of shared-memory stages with 2-D bulk tensor copies (TMA,
//     128-byte swizzle), one mbarrier per stage and direction.
//   * Four consumer warps take the stages round-robin. Per 16-token block a
//     warp computes S = Q K^T with m16n8k16 tensor-core MMAs (query rows in
//     M, padded to 16; fp32 accumulate), applies the causal/length mask,
//     updates an fp32 online softmax (running max and sum, base-2
//     exponentials) and accumulates O += P V, P split as P_hi + P_lo in the
//     16-bit type so the product keeps ~16 mantissa bits.
//   * The four warps' (m, l, O) are merged through shared memory; a CTA
//     whose sequence fits one partition writes the normalised output, the
//     others write (o, m, l) partials that split_kv_reduce merges with the
//     log-sum-exp rule.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <math.h>

#include <mutex>

#include "pa_internal.h"
#include "ptx.cuh"

namespace {

constexpr int kBS = 16;                  // tokens per block
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxPartBlocks = 256;      // partition_size <= 4096 tokens
constexpr float kLog2e = 1.4426950408889634f;

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
};

template <int D, int MT, int STAGES>
struct Layout {
    static constexpr int kSub = D / 64;                 // 128-byte-wide sub-tiles per tile row
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

// Byte offset of the 16-byte chunk `chunk` of row `row` in a K/V tile laid
// out by the 128B-swizzled TMA box [16 rows][64 columns] per sub-tile.
template <int D>
__device__ __forceinline__ uint32_t tile_offset(int row, int chunk) {
    const int sub = chunk >> 3, c = chunk & 7;
    return sub * (kBS * 128) + row * 128 + ((c ^ (row & 7)) << 4);
}

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
                const uint32_t kdst = base + st * Lay::kStageBytes;
                const uint32_t vdst = kdst + Lay::kTileBytes;
                pa::mbar_arrive_expect_tx(bar_full + 8 * st, Lay::kStageBytes);
#pragma unroll
                for (int sub = 0; sub < Lay::kSub; ++sub) {
                    pa::tma_load_2d(kdst + sub * kBS * 128, &tmap_k, sub * 64, row,
                                    bar_full + 8 * st, pol);
                    pa::tma_load_2d(vdst + sub * kBS * 128, &tmap_v, sub * 64, row,
                                    bar_full + 8 * st, pol);
                }
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
    const int quad = lane >> 2;      // row within an 8-row half of an m-tile
    const int qc = lane & 3;         // column pair within an n-tile

    uint32_t qreg[MT == 1 ? kKSteps : 1][4];
    if constexpr (MT == 1) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = quad + 8 * h;
            const T* src = row < R ? static_cast<const T*>(p.q) +
                                         ((int64_t)(q0 + row / G) * p.num_heads + g * G + row % G) * D
                                   : nullptr;
#pragma unroll
            for (int ks = 0; ks < kKSteps; ++ks) {
                uint32_t lo = 0, hi = 0;
                if (src) {
                    lo = __ldg(reinterpret_cast<const uint32_t*>(src + ks * 16 + 2 * qc));
                    hi = __ldg(reinterpret_cast<const uint32_t*>(src + ks * 16 + 8 + 2 * qc));
                }
                qreg[ks][h] = lo;          // a0 / a1: k = 2qc, 2qc+1
                qreg[ks][2 + h] = hi;      // a2 / a3: k = 8 + 2qc, ...
            }
        }
    }

    float o[MT][kNTiles][4];
    float m_run[MT][2], l_run[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int nt = 0; nt < kNTiles; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
        m_run[mt][0] = m_run[mt][1] = -INFINITY;
        l_run[mt][0] = l_run[mt][1] = 0.f;
    }

    // per-lane ldmatrix row addresses (before adding the stage base)
    const int mat = lane >> 3, mrow = lane & 7;
    const int k_tok = (mat >> 1) * 8 + mrow;   // K: m0,m1 tokens 0-7; m2,m3 tokens 8-15
    const int k_chk = mat & 1;                 //    m0,m2 low 8 dims; m1,m3 high 8 dims
    const int v_tok = (mat & 1) * 8 + mrow;    // V: m0,m2 tokens 0-7; m1,m3 tokens 8-15
    const int v_chk = mat >> 1;                //    m0,m1 low 8 dims; m2,m3 high 8 dims
    const int last_q_pos = L - r;              // query row i sees keys <= L - r + i

    bool ok = true;
    for (int i = warp; i < nblk; i += kConsumerWarps) {
        const int st = i % STAGES;
        if (!pa::mbar_wait(bar_full + 8 * st, (i / STAGES) & 1, p.err, pa::ERR_WAIT_FULL)) {
            ok = false;
            break;
        }
        const uint32_t kb = base + st * Lay::kStageBytes;
        const uint32_t vb = kb + Lay::kTileBytes;

        // ---- S = Q K^T ----
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
            pa::ldmatrix_x4(kb + tile_offset<D>(k_tok, 2 * ks + k_chk), b0, b1, b2, b3);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                if constexpr (MT == 1) {
                    a[0] = qreg[ks][0]; a[1] = qreg[ks][1]; a[2] = qreg[ks][2]; a[3] = qreg[ks][3];
                } else {
                    const int arow = mt * 16 + (mat & 1) * 8 + mrow;
                    const int achk = 2 * ks + (mat >> 1);
                    pa::ldmatrix_x4(base + Lay::kQOffset + arow * Lay::kQPitch + achk * 16, a[0],
                                    a[1], a[2], a[3]);
                }
                pa::mma_16816<PK::kBF16>(sacc[mt][0], a, b0, b1);
                pa::mma_16816<PK::kBF16>(sacc[mt][1], a, b2, b3);
            }
        }

        // ---- mask, online softmax, P ----
        const int tok0 = t_begin + i * kBS;                 // absolute position of token 0
        const bool need_mask = tok0 + kBS - 1 > last_q_pos;  // block reaches past some row's bound
        uint32_t phi[MT][4], plo[MT][4];
        float alpha[MT][2];
        bool rescale = false;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = mt * 16 + quad + 8 * h;
                const int bound = min(last_q_pos + row / G, L - 1);
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float v = sacc[mt][nt][2 * h + e] * p.scale_log2;
                        if (need_mask && tok0 + nt * 8 + 2 * qc + e > bound) v = -INFINITY;
                        sacc[mt][nt][2 * h + e] = v;
                        mx = fmaxf(mx, v);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[mt][h], mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                alpha[mt][h] = exp2f(m_run[mt][h] - m_use);
                m_run[mt][h] = m_new;
                float sum = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv = exp2f(sacc[mt][nt][2 * h + e] - m_use);
                        sacc[mt][nt][2 * h + e] = pv;
                        sum += pv;
                    }
                l_run[mt][h] = l_run[mt][h] * alpha[mt][h] + sum;
                if (alpha[mt][h] != 1.f) rescale = true;
            }
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const float a0 = alpha[mt][0], a1 = alpha[mt][1];
#pragma unroll
                for (int nt = 0; nt < kNTiles; ++nt) {
                    o[mt][nt][0] *= a0;
                    o[mt][nt][1] *= a0;
                    o[mt][nt][2] *= a1;
                    o[mt][nt][3] *= a1;
                }
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

        // ---- O += P V ----
        const int valid = L - tok0;   // tokens of this block inside the context (>= 1)
#pragma unroll
        for (int nd = 0; nd < D / 16; ++nd) {
            uint32_t v0, v1, v2, v3;
            pa::ldmatrix_x4_trans(vb + tile_offset<D>(v_tok, 2 * nd + v_chk), v0, v1, v2, v3);
            if (valid < kBS) {
                // slots past the context may hold anything (even NaN patterns): zero them
                const int t_lo = 2 * qc, t_hi = 2 * qc + 8;
                auto keep = [&](uint32_t x, int t) -> uint32_t {
                    uint32_t lo = (t < valid) ? (x & 0xffffu) : 0u;
                    uint32_t hi = (t + 1 < valid) ? (x & 0xffff0000u) : 0u;
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
        __syncwarp();
        if (lane == 0) pa::mbar_arrive(bar_empty + 8 * st);
    }

    // ---- merge the consumer warps through shared memory (the ring is free now) ----
    pa::named_barrier_sync(1, kConsumerWarps * 32);
    constexpr int kRows = Lay::kRows;
    float* const m_sh = reinterpret_cast<float*>(smem);                        // [W][kRows]
    float* const l_sh = m_sh + kConsumerWarps * kRows;                         // [W][kRows]
    float* const o_sh = l_sh + kConsumerWarps * kRows;                         // [W][kRows][D]
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float l = l_run[mt][h];
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            const int row = mt * 16 + quad + 8 * h;
            if (qc == 0) {
                m_sh[warp * kRows + row] = ok ? m_run[mt][h] : -INFINITY;
                l_sh[warp * kRows + row] = ok ? l : 0.f;
            }
#pragma unroll
            for (int nt = 0; nt < kNTiles; ++nt) {
                float2 v = make_float2(o[mt][nt][2 * h], o[mt][nt][2 * h + 1]);
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor map of one cache viewed as rows of head_dim 16-bit elements:
// [num_blocks * num_kv_heads * 16 rows][head_dim], box 16 rows x 64 columns,
// 128-byte swizzle.
pa_status make_cache_map(CUtensorMap* m, const void* cache, int num_blocks, int num_kv_heads,
                         int head_dim) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return pa::fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const uint64_t rows = (uint64_t)num_blocks * num_kv_heads * kBS;
    if (rows > 0x7fffffffull) return pa::fail(PA_ERR_UNSUPPORTED, "cache has too many rows for TMA");
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kBS};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(cache), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return pa::fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PA_OK;
}

// A few recently used maps, so a decode step does not re-encode them.
struct MapCache {
    struct Entry {
        const void* ptr;
        int num_blocks, num_kv_heads, head_dim, device;
        CUtensorMap map;
    };
    std::mutex mu;
    Entry e[16];
    int n = 0, next = 0;

    pa_status get(CUtensorMap* out, const void* ptr, int nb, int hkv, int d) {
        int dev = 0;
        cudaGetDevice(&dev);
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n; ++i)
            if (e[i].ptr == ptr && e[i].num_blocks == nb && e[i].num_kv_heads == hkv &&
                e[i].head_dim == d && e[i].device == dev) {
                *out = e[i].map;
                return PA_OK;
            }
        CUtensorMap m;
        if (pa_status st = make_cache_map(&m, ptr, nb, hkv, d)) return st;
        Entry& x = e[next];
        x = Entry{ptr, nb, hkv, d, dev, m};
        next = (next + 1) % 16;
        if (n < 16) ++n;
        *out = m;
        return PA_OK;
    }
};
MapCache g_maps;

template <typename T, int D, int MT>
pa_status launch_typed(const pa::DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                       const DecodeParams& prm) {
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
    kern<<<grid, kThreads, Lay::kSmemBytes, a.stream>>>(mk, mv, prm);
    if (pa_status s = pa::cuda_status(cudaGetLastError(), "decode launch")) return s;
    if (a.num_partitions > 1) {
        dim3 rgrid((a.num_heads + 3) / 4, a.num_seqs);
        split_kv_reduce_kernel<T, D><<<rgrid, 128, 0, a.stream>>>(
            a.out, a.out_dtype == PA_F32, a.o_part, a.m_part, a.l_part, a.context_lens,
            a.query_start_loc, a.num_heads, a.num_partitions, a.partition_size);
        if (pa_status s = pa::cuda_status(cudaGetLastError(), "split-KV reduce launch")) return s;
    }
    return PA_OK;
}

template <typename T>
pa_status launch_dtype(const pa::DecodeArgs& a, int mt, const CUtensorMap& mk,
                       const CUtensorMap& mv, const DecodeParams& prm) {
    if (a.head_dim == 128) {
        if (mt == 1) return launch_typed<T, 128, 1>(a, mk, mv, prm);
        return launch_typed<T, 128, 2>(a, mk, mv, prm);
    }
    if (mt == 1) return launch_typed<T, 64, 1>(a, mk, mv, prm);
    return launch_typed<T, 64, 2>(a, mk, mv, prm);
}

}  // namespace

namespace pa {

pa_status launch_decode_int8(const DecodeArgs& a);

pa_status launch_decode(const DecodeArgs& a) {
    if (a.kv_dtype == PA_INT8) return launch_decode_int8(a);
    if (a.partition_size > kMaxPartBlocks * kBS)
        return fail(PA_ERR_UNSUPPORTED, "partition_size %d > %d", a.partition_size,
                    kMaxPartBlocks * kBS);
    const int G = a.num_heads / a.num_kv_heads;
    const int64_t rows = (int64_t)G * a.max_q_len;
    const int mt = (int)((rows + 15) / 16);
    if (mt > 2)
        return fail(PA_ERR_UNSUPPORTED,
                    "%lld query rows per KV head (q heads per KV head x max_q_len) > 32 for a "
                    "16-bit cache", (long long)rows);
    CUtensorMap mk, mv;
    if (pa_status s = g_maps.get(&mk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim)) return s;
    if (pa_status s = g_maps.get(&mv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim)) return s;
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
    if (a.kv_dtype == PA_BF16) return launch_dtype<__nv_bfloat16>(a, mt, mk, mv, prm);
    return launch_dtype<__half>(a, mt, mk, mv, prm);
}

}  // namespace pa
