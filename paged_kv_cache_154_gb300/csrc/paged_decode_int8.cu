// Paged decode attention over an INT8 cache, one warp per share.
//
// The cache holds codes x_q with one fp32 scale and int8 zero point per
// (token, kv head); a value is (x_q - zero_point) * scale ("cs336 lecture 10",
// Quantization). The attention, softmax(Q K^T / sqrt(d)) V ("KV Cache ...
// PagedAttention" §二), is computed on fp16 tensor cores without forming the
// dequantised values:
//
//   S[i][t] = scale_t * sum_j q_ij (x_q[t][j] - zp_t)
//   O[i][j] = sum_t P[i][t] * scale_t * (x_q[t][j] - zp_t)
//
// (x_q - zp) is an integer in [-255, 255], exact in fp16, made from the code
// bytes with the 1024-bias trick; q goes to fp16 after an exact power-of-two
// scaling per row; the per-token V scale is folded into P against a running
// power-of-two reference (the largest scale seen, rounded up), so the fp16 P
// never exceeds the softmax weight and a new reference rescales O exactly.
//
// Work split: the balanced schedule (balanced.cuh) with the per-warp layout
// of the FP8 kernel: every warp streams its own share through its own TMA
// ring (code tiles by TMA, scales and zero points by bulk copies on the same
// barrier) and computes 16 query rows against all 16 tokens of each block,
// so every code is converted once per tile of rows; more rows per kv head
// (MQA, verify runs) become more row chunks, whose repeated reads of a block
// mostly hit L2 (their segments sit next to each other in the schedule).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <math.h>

#include <algorithm>

#include "balanced.cuh"
#include "pa_internal.h"
#include "ptx.cuh"

namespace {

using pa::sched::kBS;
using pa::sched::kWorkerWarps;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kStages = 4;
constexpr int kScaleBytes = 160;   // per stage: k scale[16], v scale[16] (fp32), k zp[16], v zp[16]
constexpr float kLazyMax = 8.f;    // base-2 headroom before the running max is moved
constexpr uint32_t kMagic = 0x64646464u;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

// fp16 pair (1152 + z_i, 1152 + z_j) for the zero points in bytes i and j of
// the word zw: (z ^ 0x80) = z + 128 placed in the mantissa of 1024.0, as the
// codes are. Subtracting it from (1024 + (code ^ 0x80)) leaves code - zp exactly.
__device__ __forceinline__ uint32_t zp_pair(uint32_t zw, int i, int j) {
    return prmt(zw ^ 0x80808080u, kMagic, 0x4040u | (uint32_t)i | ((uint32_t)j << 8));
}

// (code - zp) of the two code bytes in the low (sel 0x4140) or high (0x4342)
// half of a word whose bytes were XOR-ed with 0x80, as an fp16 pair
__device__ __forceinline__ uint32_t code_pair(uint32_t u, uint32_t sel, uint32_t zb) {
    return hsub2(prmt(u, kMagic, sel), zb);
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

// byte offset of 16-byte chunk `chunk` of token row `row` in a code tile as
// the tensor map writes it: 128-byte swizzle for d = 128, 64-byte for d = 64
template <int D>
__device__ __forceinline__ uint32_t tile8_offset(int row, int chunk) {
    if constexpr (D == 128) return row * 128 + ((chunk ^ (row & 7)) << 4);
    else return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
}

// Per warp: kStages stages of (K codes, V codes), then the stages' scale
// areas, padded so the next warp's ring starts on a 1024-byte boundary.
template <int D>
struct Q8Layout {
    static constexpr int kTile = kBS * D;                 // one K (or V) code tile
    static constexpr int kStage = 2 * kTile;
    static constexpr int kRing = kStages * kStage;
    static constexpr int kScalesAt = kRing;
    static constexpr int kWarp = (kRing + kStages * kScaleBytes + 1023) / 1024 * 1024;
    static_assert(kTile % 1024 == 0, "TMA swizzle alignment");
    __host__ __device__ static int smem_bytes(int num_seqs) {
        return pa::sched::header_bytes(num_seqs, kStages) + kWorkerWarps * kWarp + 1024;
    }
};

struct Q8Extra {
    const float* k_scale;   // [num_blocks][num_kv_heads][16]
    const float* v_scale;
    const int8_t* k_zp;
    const int8_t* v_zp;
};

template <typename TQ, int D>
__global__ void __launch_bounds__(kWorkerWarps * 32)
    paged_decode_int8_kernel(const __grid_constant__ CUtensorMap tmap_k,
                              const __grid_constant__ CUtensorMap tmap_v,
                              const pa::sched::Params p, const Q8Extra x) {
    using namespace pa::sched;
    using Lay = Q8Layout<D>;
    constexpr int S = kStages;
    constexpr int KCH = D / 16;          // 16-dim chunks = k-steps of Q K^T
    constexpr int NT = D / 8;            // n-tiles of O

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = pa::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = lane >> 2, qc = lane & 3;
    const int mat = lane >> 3, mrow = lane & 7;
    const int ld_tok = (mat & 1) * 8 + mrow;   // m0, m2: tokens 0-7; m1, m3: tokens 8-15
    const int ld_chk = mat >> 1;               // m0, m1: chunk 2pp; m2, m3: chunk 2pp + 1
    const int hkv = p.num_kv_heads, G = p.group, n_seqs = p.num_seqs;
    int32_t* const cum = reinterpret_cast<int32_t*>(smem + kWorkerWarps * S * 8);
    uint8_t* const chunks = reinterpret_cast<uint8_t*>(cum + n_seqs + 1);
    const uint32_t bars = base + warp * S * 8;
    const int hdr = header_bytes(n_seqs, S);
    const uint32_t ring = base + hdr + warp * Lay::kWarp;
    const uint8_t* const scales = smem + hdr + warp * Lay::kWarp + Lay::kScalesAt;

    build_prefix(cum, chunks, p);
    const int64_t B = cum[n_seqs];
    const int64_t wid = (int64_t)blockIdx.x * kWorkerWarps + warp;
    const int64_t W = share_count(p, B);
    const int64_t f0 = share_start(wid, B, W);
    const int64_t f1 = share_start(wid + 1, B, W);
    const int n = (int)(f1 - f0);
    if (lane == 0) write_merge_record(p, wid, 0, 0, 0);   // none unless set at the end
    if (wid >= W || n <= 0) return;   // the grid's last CTA may have spare warps

    uint64_t pol_once = 0, pol_again = 0;
    if (lane == 0) {
        for (int i = 0; i < S; ++i) pa::mbar_init(bars + 8 * i, 1);
        pa::fence_barrier_init();
        pa::prefetch_tensormap(&tmap_k);
        pa::prefetch_tensormap(&tmap_v);
        pol_once = pa::policy_evict_first();
        pol_again = pa::policy_evict_normal();
    }
    __syncwarp();

    // each lane keeps the (block x H_kv + kv head) tile of virtual block
    // win + lane and whether later row chunks read that block again
    int win = -32, my_tile = 0, my_once = 1;
    auto refresh = [&](int wbase) {
        win = wbase;
        const int64_t f = f0 + wbase + lane;
        my_tile = 0;
        my_once = 1;
        if (f < f1) {
            const Pos q = locate(p, cum, chunks, f);
            int blk = __ldg(p.block_tables + (int64_t)q.s * p.max_blocks + q.b);
            if (blk < 0 || blk >= p.num_blocks) {
                if (p.err) atomicOr(p.err, pa::ERR_BAD_BLOCK);
                blk = 0;
            }
            my_tile = blk * hkv + q.g;
            my_once = q.C == 1;
        }
    };
    auto issue = [&](int k) {   // warp-uniform
        if (k >= win + 32) refresh(k & ~31);
        const int tile = __shfl_sync(0xffffffffu, my_tile, k - win);
        const int once = __shfl_sync(0xffffffffu, my_once, k - win);
        if (lane == 0) {
            const uint32_t bar = bars + 8 * (k % S);
            const uint32_t dst = ring + (k % S) * Lay::kStage;
            const uint32_t sd = ring + Lay::kScalesAt + (k % S) * kScaleBytes;
            const uint64_t pol = once ? pol_once : pol_again;
            pa::mbar_arrive_expect_tx(bar, 2 * Lay::kTile + kScaleBytes);
            pa::tma_load_2d(dst, &tmap_k, 0, tile * kBS, bar, pol);
            pa::tma_load_2d(dst + Lay::kTile, &tmap_v, 0, tile * kBS, bar, pol);
            bulk_load(sd, x.k_scale + (int64_t)tile * kBS, 64, bar);
            bulk_load(sd + 64, x.v_scale + (int64_t)tile * kBS, 64, bar);
            bulk_load(sd + 128, x.k_zp + (int64_t)tile * kBS, 16, bar);
            bulk_load(sd + 144, x.v_zp + (int64_t)tile * kBS, 16, bar);
        }
    };
    int issued = 0;
    for (; issued < S && issued < n; ++issued) issue(issued);

    Pos cur = locate(p, cum, chunks, f0);
    float o[NT][4];
    float m_run[2], l_run[2], rowmul[2];
    uint32_t qa[KCH][4];
    int ev = -126;                       // log2 of the running V-scale reference
    int L = 0, r = 1, q0 = 0, rows = 0, row_off = 0, seg_b0 = cur.b, last_q = 0;
    bool seg_first = true;

    // Segment start: this warp's 16 q rows as fp16 A fragments, each row
    // scaled by 2^(14 - e_row); the lane's dims of k-step ks are 16 ks + 4 qc
    // .. + 3, placed at MMA k positions (2 qc, 2 qc + 1) and (2 qc + 8, 2 qc +
    // 9) -- the order in which a K fragment holds the code bytes.
    auto start_segment = [&]() {
        L = __ldg(p.context_lens + cur.s);
        r = query_run(p.qsl, cur.s, &q0);
        last_q = L - r;
        row_off = cur.c * kBS;
        rows = min(kBS, G * r - row_off);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = quad + 8 * h;
            float v[KCH][4];
            if (row < rows) {
                const int gr = row_off + row;
                const TQ* src = static_cast<const TQ*>(p.q) +
                                ((int64_t)(q0 + gr / G) * p.num_heads + cur.g * G + gr % G) * D +
                                4 * qc;
#pragma unroll
                for (int ks = 0; ks < KCH; ++ks) {
                    const uint2 u = __ldg(reinterpret_cast<const uint2*>(src + 16 * ks));
                    const TQ* t = reinterpret_cast<const TQ*>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[ks][e] = (float)t[e];
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < KCH; ++ks)
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[ks][e] = 0.f;
            }
            float mx = 0.f;
#pragma unroll
            for (int ks = 0; ks < KCH; ++ks)
#pragma unroll
                for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fabsf(v[ks][e]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            int ex = 0;
            if (mx > 0.f) {
                ex = (int)((__float_as_uint(mx) >> 23) & 0xff) - 127;   // floor(log2 max|q|)
                ex = max(-100, min(100, ex));
            }
            const float up = exp2i(14 - ex);
#pragma unroll
            for (int ks = 0; ks < KCH; ++ks) {
                __half2 lo = __floats2half2_rn(v[ks][0] * up, v[ks][1] * up);
                __half2 hi = __floats2half2_rn(v[ks][2] * up, v[ks][3] * up);
                qa[ks][h] = *reinterpret_cast<uint32_t*>(&lo);
                qa[ks][2 + h] = *reinterpret_cast<uint32_t*>(&hi);
            }
            rowmul[h] = row < rows ? p.scale_log2 * exp2i(ex - 14) : 0.f;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
        ev = -126;
    };

    // Segment end: the output rows (segment held whole) or the partial slot;
    // O is in units of the V-scale reference 2^ev.
    auto finish_segment = [&](bool complete, int slot_idx, int tok_end) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
        }
        Slot sl(p.slots + (2 * wid + slot_idx) * (int64_t)p.slot_bytes, kBS);
        if (!complete && lane == 0) {
            sl.hdr[0] = cur.s;
            sl.hdr[1] = cur.g;
            sl.hdr[2] = cur.c;
            sl.hdr[3] = seg_b0 * kBS;
            sl.hdr[4] = tok_end;
        }
        const float vref = exp2i(ev);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = quad + 8 * h;
            if (row >= rows) continue;
            const float mul = complete ? vref / l_run[h] : vref;
            int64_t obase = 0;
            if (complete) {
                const int gr = row_off + row;
                obase = ((int64_t)(q0 + gr / G) * p.num_heads + cur.g * G + gr % G) * D;
            } else if (qc == 0) {
                sl.m[row] = m_run[h];
                sl.l[row] = l_run[h];
            }
#pragma unroll
            for (int c = 0; c < KCH; ++c) {
                // n-tile 2c holds dims 16c + 4qc and + 2, n-tile 2c + 1 dims + 1 and + 3
                const float4 v = make_float4(o[2 * c][2 * h] * mul, o[2 * c + 1][2 * h] * mul,
                                             o[2 * c][2 * h + 1] * mul,
                                             o[2 * c + 1][2 * h + 1] * mul);
                const int col = 16 * c + 4 * qc;
                if (!complete) {
                    *reinterpret_cast<float4*>(sl.o + (int64_t)row * D + col) = v;
                } else if (p.out_f32) {
                    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + obase + col) = v;
                } else {
                    TQ* o16 = static_cast<TQ*>(p.out) + obase + col;
                    if constexpr (std::is_same<TQ, __half>::value) {
                        *reinterpret_cast<__half2*>(o16) = __floats2half2_rn(v.x, v.y);
                        *reinterpret_cast<__half2*>(o16 + 2) = __floats2half2_rn(v.z, v.w);
                    } else {
                        *reinterpret_cast<__nv_bfloat162*>(o16) = __floats2bfloat162_rn(v.x, v.y);
                        *reinterpret_cast<__nv_bfloat162*>(o16 + 2) =
                            __floats2bfloat162_rn(v.z, v.w);
                    }
                }
            }
        }
    };

    start_segment();
    int consumed = 0;
    for (int k = 0; k < n; ++k) {
        const int st = k % S;
        if (!pa::mbar_wait(bars + 8 * st, (k / S) & 1, p.err, pa::ERR_WAIT_FULL)) break;
        consumed = k + 1;
        const uint32_t kb = ring + st * Lay::kStage, vb = kb + Lay::kTile;
        const uint8_t* sp = scales + st * kScaleBytes;
        const float* ksc = reinterpret_cast<const float*>(sp);
        const float* vsc = ksc + 16;
        const uint32_t* kzw = reinterpret_cast<const uint32_t*>(sp + 128);   // 4 zero points a word
        const uint32_t* vzw = kzw + 4;
        const int tok0 = cur.b * kBS;
        const int valid = L - tok0;   // tokens of this block inside the context (>= 1)

        // ---- S = Q (K codes - zp)^T over the block's 16 tokens (two n-tiles of 8) ----
        // the lane's K fragments hold tokens quad (n-tile 0) and 8 + quad (n-tile 1)
        const int qb = quad & 3;
        const uint32_t zk0 = zp_pair(kzw[quad >> 2], qb, qb);
        const uint32_t zk1 = zp_pair(kzw[2 + (quad >> 2)], qb, qb);
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int pp = 0; pp < KCH / 2; ++pp) {
            uint32_t rr[4];
            pa::ldmatrix_x4(kb + tile8_offset<D>(ld_tok, 2 * pp + ld_chk), rr[0], rr[1], rr[2],
                            rr[3]);
            // rr[j]: k-step 2pp + j/2, tokens (j & 1) * 8 + quad, dims 4qc .. 4qc + 3
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t u = rr[j] ^ 0x80808080u;
                const uint32_t zb = (j & 1) ? zk1 : zk0;
                mma_f16(s[j & 1], qa[2 * pp + (j >> 1)], code_pair(u, 0x4140, zb),
                        code_pair(u, 0x4342, zb));
            }
        }

        // ---- scales, mask, online softmax (lazy max) ----
        // the lane's S columns: tokens 2qc, 2qc + 1 (n-tile 0), 8 + 2qc, 9 + 2qc (n-tile 1)
        const int t0 = 2 * qc;
        const float2 ks_a = *reinterpret_cast<const float2*>(ksc + t0);
        const float2 ks_b = *reinterpret_cast<const float2*>(ksc + 8 + t0);
        const float2 vs_a = *reinterpret_cast<const float2*>(vsc + t0);
        const float2 vs_b = *reinterpret_cast<const float2*>(vsc + 8 + t0);
        // scales past the context may hold anything: their weights must be 0
        const float kss[4] = {ks_a.x, ks_a.y, ks_b.x, ks_b.y};
        float vss[4] = {t0 < valid ? vs_a.x : 0.f, t0 + 1 < valid ? vs_a.y : 0.f,
                        t0 + 8 < valid ? vs_b.x : 0.f, t0 + 9 < valid ? vs_b.y : 0.f};
        float vmax = fmaxf(fmaxf(vss[0], vss[1]), fmaxf(vss[2], vss[3]));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
        const int ev_new = max(ev, ceil_log2(vmax));
        const float vfix = exp2i(ev - ev_new);          // exact rescale of O to the new reference
        ev = ev_new;
        const float inv_vref = exp2i(-ev);
        const bool need_mask = tok0 + kBS - 1 > last_q;
        float alpha[2];
        bool rescale = vfix != 1.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = quad + 8 * h;
            const float rm = rowmul[h];
            float a[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) a[2 * nt + e] = s[nt][2 * h + e] * kss[2 * nt + e] * rm;
            if (need_mask) {
                const int bound = min(last_q + (row_off + row) / G, L - 1);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        if (tok0 + nt * 8 + t0 + e > bound) a[2 * nt + e] = -INFINITY;
            }
            float mx = fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            float al = 1.f;
            if (mx > m_run[h] + kLazyMax) {
                al = pa::ex2(m_run[h] - mx);         // 0 while m_run is -inf
                m_run[h] = mx;
                rescale = true;
            }
            const float m_use = m_run[h] == -INFINITY ? 0.f : m_run[h];
            float sum = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pv = pa::ex2(a[2 * nt + e] - m_use);
                    sum += pv;
                    s[nt][2 * h + e] = pv * (vss[2 * nt + e] * inv_vref);
                }
            l_run[h] = l_run[h] * al + sum;
            alpha[h] = al * vfix;
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                o[nt][0] *= alpha[0];
                o[nt][1] *= alpha[0];
                o[nt][2] *= alpha[1];
                o[nt][3] *= alpha[1];
            }
        }
        uint32_t pa_[4];
        {
            __half2 h0 = __floats2half2_rn(s[0][0], s[0][1]);
            __half2 h1 = __floats2half2_rn(s[0][2], s[0][3]);
            __half2 h2 = __floats2half2_rn(s[1][0], s[1][1]);
            __half2 h3 = __floats2half2_rn(s[1][2], s[1][3]);
            pa_[0] = *reinterpret_cast<uint32_t*>(&h0);
            pa_[1] = *reinterpret_cast<uint32_t*>(&h1);
            pa_[2] = *reinterpret_cast<uint32_t*>(&h2);
            pa_[3] = *reinterpret_cast<uint32_t*>(&h3);
        }

        // ---- O += P' (V codes - zp) ----
        // the lane's V pairs: tokens 2qc, 2qc + 1 (b0) and 2qc + 8, 2qc + 9 (b1)
        const int tb = t0 & 3;   // tokens t0, t0 + 1 are bytes tb, tb + 1 of word t0 / 4
        const uint32_t zv0 = zp_pair(vzw[t0 >> 2], tb, tb + 1);
        const uint32_t zv1 = zp_pair(vzw[2 + (t0 >> 2)], tb, tb + 1);
#pragma unroll
        for (int pp = 0; pp < KCH / 2; ++pp) {
            uint32_t rr[4];
            pa::ldmatrix_x4_trans(vb + tile8_offset<D>(ld_tok, 2 * pp + ld_chk), rr[0], rr[1],
                                  rr[2], rr[3]);
            // rr[2 half + 0]: tokens 2qc, 2qc + 1; rr[2 half + 1]: tokens 2qc + 8, + 9;
            // bytes (t, dim 2 quad), (t, dim 2 quad + 1), (t + 1, 2 quad), (t + 1, 2 quad + 1)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int c = 2 * pp + half;
                // one prmt per pair of words: (t, dim a) and (t + 1, dim a) into the low
                // half, (t, dim b) and (t + 1, dim b) into the high half
                const uint32_t w0 = prmt(rr[2 * half], rr[2 * half + 1], 0x3120) ^ 0x80808080u;
                const uint32_t w1 = prmt(rr[2 * half], rr[2 * half + 1], 0x7564) ^ 0x80808080u;
                mma_f16(o[2 * c], pa_, code_pair(w0, 0x4140, zv0), code_pair(w1, 0x4140, zv1));
                mma_f16(o[2 * c + 1], pa_, code_pair(w0, 0x4342, zv0),
                        code_pair(w1, 0x4342, zv1));
            }
        }
        __syncwarp();
        if (issued < n) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(issued);
            ++issued;
        }
        ++cur.b;
        const bool seg_done = cur.b == cur.nbs;
        if (seg_done || k == n - 1) {
            finish_segment(seg_b0 == 0 && seg_done, seg_first ? 0 : 1, min(cur.b * kBS, L));
            if (k == n - 1) {
                if (lane == 0)
                    record_last_segment(p, wid, f1, B, seg_done, seg_b0, cur.nbs - cur.b,
                                        seg_first, q0, rows);
                break;
            }
            next_segment(p, cur, cum, chunks);
            seg_b0 = 0;
            seg_first = false;
            start_segment();
        }
    }
    // drain: no copy of this warp may still be in flight when it exits
    for (int k = consumed; k < issued; ++k)
        if (!pa::mbar_wait(bars + 8 * (k % S), (k / S) & 1, p.err, pa::ERR_WAIT_DRAIN)) break;
}

template <typename TQ, int D>
pa_status launch_int8(const pa::DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                       pa::sched::Params prm, const Q8Extra& x) {
    using Lay = Q8Layout<D>;
    auto kern = paged_decode_int8_kernel<TQ, D>;
    static bool attr_set = false;   // per instantiation; benign race (idempotent)
    if (!attr_set) {
        if (pa_status s = pa::cuda_status(
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Lay::smem_bytes(pa::kBalancedMaxSeqs)),
                "int8 decode: set shared memory size"))
            return s;
        attr_set = true;
    }
    const int smem = Lay::smem_bytes(a.num_seqs);
    int dev = 0, sms = 0, ctas = 0;
    if (pa_status s = pa::cuda_status(cudaGetDevice(&dev), "cudaGetDevice")) return s;
    if (pa_status s = pa::cuda_status(
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count"))
        return s;
    if (pa_status s = pa::cuda_status(
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas, kern, kWorkerWarps * 32, smem),
            "occupancy query"))
        return s;
    if (ctas < 1) return pa::fail(PA_ERR_UNSUPPORTED, "int8 decode kernel does not fit on an SM");
    const pa::BalancedShape shape = pa::balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads,
                                                       a.head_dim, a.max_q_len, a.max_context_len,
                                                       pa::kTileInt8);
    const int64_t workers =
        std::min<int64_t>((int64_t)ctas * sms * kWorkerWarps, shape.workers);
    prm.workers = (int)workers;
    const int grid = (int)((workers + kWorkerWarps - 1) / kWorkerWarps);
    if (pa_status s = pa::cuda_status(
            pa::launch_pdl(kern, dim3(grid), dim3(kWorkerWarps * 32), smem, a.stream, mk, mv, prm,
                           x),
            "int8 decode launch"))
        return s;
    const int row_slots = (int)std::min<int64_t>(kBS, (int64_t)(a.num_heads / a.num_kv_heads) *
                                                          a.max_q_len);
    return pa::cuda_status(pa::sched::launch_segment_reduce<TQ, D>(prm, (int)shape.max_chunks,
                                                                    row_slots, a.stream),
                           "segment reduce launch");
}

}  // namespace

namespace pa {

// INT8 decode: one warp per share, 16-row tiles (see the top of this file).
pa_status launch_decode_int8(const DecodeArgs& a) {
    if (a.partition_size != 0)
        return fail(PA_ERR_UNSUPPORTED, "INT8 caches use the balanced schedule (partition_size 0)");
    if (int8_tc_applies(a)) return launch_decode_int8_tc(a);
    if (pa_status s = balanced_check(a)) return s;
    if (((uintptr_t)a.k_scale | (uintptr_t)a.v_scale | (uintptr_t)a.k_zp | (uintptr_t)a.v_zp) % 16)
        return fail(PA_ERR_INVALID_ARG, "k_scale, v_scale, k_zp and v_zp must be 16-byte aligned");
    const BalancedShape shape = balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads,
                                               a.head_dim, a.max_q_len, a.max_context_len,
                                               kTileInt8);
    CUtensorMap mk, mv;
    if (pa_status s = cache_tensor_map(&mk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 1))
        return s;
    if (pa_status s = cache_tensor_map(&mv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 1))
        return s;
    pa::sched::Params b{};
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
    b.rows_per_tile = shape.rows_per_tile;
    b.slot_bytes = (int)shape.slot_bytes;
    b.scale_log2 = a.scale * kLog2e;
    b.out_f32 = a.out_dtype == PA_F32;
    const Q8Extra x{a.k_scale, a.v_scale, a.k_zp, a.v_zp};
    if (a.q_dtype == PA_BF16)
        return a.head_dim == 128 ? launch_int8<__nv_bfloat16, 128>(a, mk, mv, b, x)
                                 : launch_int8<__nv_bfloat16, 64>(a, mk, mv, b, x);
    return a.head_dim == 128 ? launch_int8<__half, 128>(a, mk, mv, b, x)
                             : launch_int8<__half, 64>(a, mk, mv, b, x);
}

}  // namespace pa
