// Paged decode attention over an INT8 cache.
//
// The cache holds codes x_q with one fp32 scale and int8 zero point per
// (token, kv head); a value is (x_q - zero_point) * scale ("cs336 lecture 10",
// Quantization). Attention is the same softmax(Q K^T / sqrt(d)) V as the
// 16-bit path ("KV Cache ... PagedAttention" §二), computed on fp16 tensor
// cores without ever forming the dequantised values:
//
//   S[i][t] = scale_t * sum_j q_ij (x_q[t][j] - zp_t)
//   O[i][j] = sum_t P[i][t] * scale_t * (x_q[t][j] - zp_t)
//
// (x_q - zp) is an integer in [-255, 255], exact in fp16; it is made from
// the code bytes with the 1024-bias trick (byte ^ 0x80 placed in the
// mantissa of 1024.0, minus 1152 + zp). q is converted to fp16 after an
// exact power-of-two scaling per row that puts its largest |q| in [2^14,
// 2^15) (a bf16 value has 8 significant bits, so the conversion is exact
// for every element within 2^-28 of the row maximum); the scale is undone
// on S. The per-token scale_t multiplies S column-wise; on the PV side it is
// folded into P together with a running power-of-two reference (the largest
// scale seen so far, rounded up), so the fp16 P stays in [0, 1]; a larger
// reference rescales O exactly, like the running max of the softmax.
//
// Schedule, tiles and reduce: balanced.cuh (equal shares of (sequence, kv
// head, row chunk, block) work per warp, each warp with its own TMA ring).
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

namespace {

using pa::sched::kBS;
using pa::sched::kWorkerWarps;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kStages = 3;
constexpr int kScaleBytes = 160;   // per stage: k scale[16], v scale[16] (fp32), k zp[16], v zp[16]

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

// fp16 pair (1152 + z0, 1152 + z1): subtracting it from (1024 + (code ^ 0x80))
// leaves code - zp exactly.
__device__ __forceinline__ uint32_t zp_bias(int z0, int z1) {
    __half2 h = __halves2half2(__int2half_rn(1152 + z0), __int2half_rn(1152 + z1));
    return *reinterpret_cast<uint32_t*>(&h);
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

template <int D>
__device__ __forceinline__ uint32_t tile8_offset(int row, int chunk) {
    if constexpr (D == 128) return row * 128 + ((chunk ^ (row & 7)) << 4);          // 128B swizzle
    else return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);                        // 64B swizzle
}

// Shared memory after the schedule header: the four warps' rings (each a
// multiple of 1024 bytes, so every stage starts on a 1024-byte boundary as
// TMA and the swizzle need), then per warp its stage scale areas, its Q tile
// and its row factors.
template <int D, int MT>
struct Q8Layout {
    static constexpr int RT = 16 * MT;
    static constexpr int kTile = kBS * D;                         // codes of one K (or V) tile
    static constexpr int kStage = ((2 * kTile) + 1023) / 1024 * 1024;
    static constexpr int kRing = kStages * kStage;
    static constexpr int kScales = kStages * kScaleBytes;
    static constexpr int kQPitch = D * 2 + 16;
    static constexpr int kQTile = RT * kQPitch;
    static constexpr int kRowMul = RT * 4;
    static_assert(kRing % 1024 == 0, "rings must keep 1024-byte alignment");
    static_assert(kScales % 16 == 0 && kQTile % 16 == 0, "16-byte alignment");
    static constexpr int kRings = kWorkerWarps * kRing;
    static constexpr int kScalesAt = kRings;
    static constexpr int kQAt = kScalesAt + kWorkerWarps * kScales;
    static constexpr int kRowMulAt = kQAt + kWorkerWarps * kQTile;
    static constexpr int kBody = kRowMulAt + kWorkerWarps * kRowMul;
    __host__ __device__ static int smem_bytes(int num_seqs) {
        return pa::sched::header_bytes(num_seqs, kStages) + kBody + 1024;
    }
};

struct Q8Extra {
    const float* k_scale;
    const float* v_scale;
    const int8_t* k_zp;
    const int8_t* v_zp;
};

template <typename TQ, int D, int MT>
__global__ void __launch_bounds__(kWorkerWarps * 32)
    paged_decode_int8_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v,
                             const pa::sched::Params p, const Q8Extra x) {
    using namespace pa::sched;
    using Lay = Q8Layout<D, MT>;
    constexpr int S = kStages;
    constexpr int RT = Lay::RT;
    constexpr int kNTiles = D / 8;
    constexpr int kChunks = D / 16;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = pa::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = lane >> 2, qc = lane & 3;
    const int hkv = p.num_kv_heads, G = p.group, n_seqs = p.num_seqs;
    int32_t* const cum = reinterpret_cast<int32_t*>(smem + kWorkerWarps * S * 8);
    uint8_t* const chunks = reinterpret_cast<uint8_t*>(cum + n_seqs + 1);
    const uint32_t bars = base + warp * S * 8;
    const int hdr = header_bytes(n_seqs, S);            // a multiple of 1024
    const uint32_t ring = base + hdr + warp * Lay::kRing;
    const uint32_t scl = base + hdr + Lay::kScalesAt + warp * Lay::kScales;   // S x 160 bytes
    const uint32_t qtile = base + hdr + Lay::kQAt + warp * Lay::kQTile;
    uint8_t* const scl_p = smem + hdr + Lay::kScalesAt + warp * Lay::kScales;
    float* const rowmul_p =
        reinterpret_cast<float*>(smem + hdr + Lay::kRowMulAt + warp * Lay::kRowMul);

    build_prefix(cum, chunks, p);
    const int64_t B = cum[n_seqs];
    const int64_t wid = (int64_t)blockIdx.x * kWorkerWarps + warp;
    const int64_t f0 = share_start(wid, B, p.workers);
    const int64_t f1 = share_start(wid + 1, B, p.workers);
    const int n = (int)(f1 - f0);
    if (n <= 0) return;

    if (lane == 0) {
        for (int i = 0; i < S; ++i) pa::mbar_init(bars + 8 * i, 1);
        pa::fence_barrier_init();
    }
    __syncwarp();

    if (lane == 0) {
        pa::prefetch_tensormap(&tmap_k);
        pa::prefetch_tensormap(&tmap_v);
    }
    // each lane keeps the (block * H_kv + kv head) tile index of virtual block win + lane
    int win = -32, my_tile = 0;
    auto refresh = [&](int wb) {
        win = wb;
        const int64_t f = f0 + wb + lane;
        my_tile = 0;
        if (f < f1) {
            const Pos q = locate(cum, chunks, n_seqs, hkv, f);
            int blk = __ldg(p.block_tables + (int64_t)q.s * p.max_blocks + q.b);
            if (blk < 0 || blk >= p.num_blocks) {
                if (p.err) atomicOr(p.err, pa::ERR_BAD_BLOCK);
                blk = 0;
            }
            my_tile = blk * hkv + q.g;
        }
    };
    auto issue = [&](int k) {   // warp-uniform
        if (k >= win + 32) refresh(k & ~31);
        const int tile = __shfl_sync(0xffffffffu, my_tile, k - win);
        if (lane == 0) {
            const int st = k % S;
            const uint32_t bar = bars + 8 * st;
            const uint32_t dst = ring + st * Lay::kStage;
            const uint32_t sd = scl + st * kScaleBytes;
            pa::mbar_arrive_expect_tx(bar, 2 * Lay::kTile + kScaleBytes);
            pa::tma_load_2d(dst, &tmap_k, 0, tile * kBS, bar);
            pa::tma_load_2d(dst + Lay::kTile, &tmap_v, 0, tile * kBS, bar);
            bulk_load(sd, x.k_scale + (int64_t)tile * kBS, 64, bar);
            bulk_load(sd + 64, x.v_scale + (int64_t)tile * kBS, 64, bar);
            bulk_load(sd + 128, x.k_zp + (int64_t)tile * kBS, 16, bar);
            bulk_load(sd + 144, x.v_zp + (int64_t)tile * kBS, 16, bar);
        }
    };
    int issued = 0;
    for (; issued < S && issued < n; ++issued) issue(issued);

    Pos cur = locate(cum, chunks, n_seqs, hkv, f0);
    float o[MT][kNTiles][4];
    float m_run[MT][2], l_run[MT][2], rowmul[MT][2];
    int ev = -126;                       // log2 of the running V-scale reference
    int L = 0, r = 1, q0 = 0, rows = 0, row_off = 0, seg_b0 = cur.b;
    bool seg_first = true;

    auto start_segment = [&]() {
        L = __ldg(p.context_lens + cur.s);
        r = query_run(p.qsl, cur.s, &q0);
        row_off = cur.c * RT;
        rows = min(RT, G * r - row_off);
        __syncwarp();
        // Q tile: fp16, scaled by 2^(14 - e_row), dims in the MMA's k order.
        // Eight rows' loads are issued together, then reduced and stored.
        constexpr int EPL = D / 32;
        for (int r0 = 0; r0 < RT; r0 += 8) {
            float v[8][EPL];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int row = r0 + j;
#pragma unroll
                for (int e = 0; e < EPL; ++e) v[j][e] = 0.f;
                if (row < rows) {
                    const int gr = row_off + row;
                    const TQ* src = static_cast<const TQ*>(p.q) +
                                    ((int64_t)(q0 + gr / G) * p.num_heads + cur.g * G + gr % G) *
                                        D +
                                    lane * EPL;
                    if constexpr (EPL == 4) {
                        const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
                        const TQ* t = reinterpret_cast<const TQ*>(&u);
#pragma unroll
                        for (int e = 0; e < 4; ++e) v[j][e] = (float)t[e];
                    } else {
                        const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(src));
                        const TQ* t = reinterpret_cast<const TQ*>(&u);
                        v[j][0] = (float)t[0];
                        v[j][1] = (float)t[1];
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int row = r0 + j;
                float mx = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) mx = fmaxf(mx, fabsf(v[j][e]));
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                int ex = 0;
                if (mx > 0.f) {
                    ex = (int)((__float_as_uint(mx) >> 23) & 0xff) - 127;   // floor(log2 max|q|)
                    ex = max(-100, min(100, ex));
                }
                const float up = exp2i(14 - ex);
                const uint32_t rowb = qtile + row * Lay::kQPitch;
                if constexpr (D == 128) {
                    // lane holds dims 4*lane .. +3: chunk lane/4, a = lane%4 -> k 2a, 2a+1, 8+2a, 9+2a
                    const int ch = lane >> 2, a = lane & 3;
                    const __half2 lo = __floats2half2_rn(v[j][0] * up, v[j][1] * up);
                    const __half2 hi = __floats2half2_rn(v[j][2] * up, v[j][3] * up);
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(rowb + (ch * 16 + 2 * a) * 2),
                                 "r"(*reinterpret_cast<const uint32_t*>(&lo)) : "memory");
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(rowb + (ch * 16 + 8 + 2 * a) * 2),
                                 "r"(*reinterpret_cast<const uint32_t*>(&hi)) : "memory");
                } else {
                    // lane holds dims 2*lane, +1: chunk lane/8, a = (lane%8)/2, b = lane%2
                    const int ch = lane >> 3, a = (lane & 7) >> 1, b = lane & 1;
                    const __half2 h = __floats2half2_rn(v[j][0] * up, v[j][1] * up);
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(
                                     rowb + (ch * 16 + 8 * b + 2 * a) * 2),
                                 "r"(*reinterpret_cast<const uint32_t*>(&h)) : "memory");
                }
                if (lane == 0) rowmul_p[row] = row < rows ? p.scale_log2 * exp2i(ex - 14) : 0.f;
            }
        }
        __syncwarp();
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) rowmul[mt][h] = rowmul_p[mt * 16 + quad + 8 * h];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int nt = 0; nt < kNTiles; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
            m_run[mt][0] = m_run[mt][1] = -INFINITY;
            l_run[mt][0] = l_run[mt][1] = 0.f;
        }
        ev = -126;
    };

    auto finish_segment = [&](bool complete, int slot_idx, int tok_end) {
        const float vref = exp2i(ev);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                l_run[mt][h] += __shfl_xor_sync(0xffffffffu, l_run[mt][h], 1);
                l_run[mt][h] += __shfl_xor_sync(0xffffffffu, l_run[mt][h], 2);
            }
        Slot sl(p.slots + (2 * wid + slot_idx) * (int64_t)p.slot_bytes, RT);
        if (!complete && lane == 0) {
            sl.hdr[0] = cur.s;
            sl.hdr[1] = cur.g;
            sl.hdr[2] = cur.c;
            sl.hdr[3] = seg_b0 * kBS;
            sl.hdr[4] = tok_end;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = mt * 16 + quad + 8 * h;
                if (row >= rows) continue;
                const int gr = row_off + row;
                const float mul = complete ? vref / l_run[mt][h] : vref;
                float* dst = sl.o + (int64_t)row * D;
                int64_t obase = 0;
                if (complete) {
                    obase = ((int64_t)(q0 + gr / G) * p.num_heads + cur.g * G + gr % G) * D;
                } else {
                    if (qc == 0) {
                        sl.m[row] = m_run[mt][h];
                        sl.l[row] = l_run[mt][h];
                    }
                }
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    // n-tile 2c holds dims 16c + 4qc and + 2, n-tile 2c+1 dims + 1 and + 3
                    const float4 v = make_float4(o[mt][2 * c][2 * h] * mul,
                                                 o[mt][2 * c + 1][2 * h] * mul,
                                                 o[mt][2 * c][2 * h + 1] * mul,
                                                 o[mt][2 * c + 1][2 * h + 1] * mul);
                    const int col = 16 * c + 4 * qc;
                    if (!complete) {
                        *reinterpret_cast<float4*>(dst + col) = v;
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
    const uint32_t kMagic = 0x64646464u;
    const int mat = lane >> 3, mrow = lane & 7;
    const int ld_tok = (mat & 1) * 8 + mrow;   // m0, m2: tokens 0-7; m1, m3: tokens 8-15
    const int ld_chk = mat >> 1;               // m0, m1: chunk 2p; m2, m3: chunk 2p + 1

    int consumed = 0;
    for (int k = 0; k < n; ++k) {
        const int st = k % S;
        if (!pa::mbar_wait(bars + 8 * st, (k / S) & 1, p.err, pa::ERR_WAIT_FULL)) break;
        consumed = k + 1;
        const uint32_t kb = ring + st * Lay::kStage, vb = kb + Lay::kTile;
        const float* ksc = reinterpret_cast<const float*>(scl_p + st * kScaleBytes);
        const float* vsc = ksc + 16;
        const int8_t* kzp = reinterpret_cast<const int8_t*>(ksc + 32);
        const int8_t* vzp = kzp + 16;
        const int tok0 = cur.b * kBS;
        const int valid = L - tok0;
        const int last_q = L - r;

        // ---- S = Q (K codes - zp)^T ----
        const uint32_t zk0 = zp_bias(kzp[quad], kzp[quad]);
        const uint32_t zk1 = zp_bias(kzp[8 + quad], kzp[8 + quad]);
        float sacc[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.f;
#pragma unroll
        for (int pch = 0; pch < kChunks / 2; ++pch) {
            uint32_t r0, r1, r2, r3;
            pa::ldmatrix_x4(kb + tile8_offset<D>(ld_tok, 2 * pch + ld_chk), r0, r1, r2, r3);
            // r0: k-step 2pch, tokens 0-7; r1: tokens 8-15; r2, r3: k-step 2pch + 1
            const uint32_t rr[4] = {r0, r1, r2, r3};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int ks = 2 * pch + (j >> 1), nt = j & 1;
                const uint32_t u = rr[j] ^ 0x80808080u;
                const uint32_t zb = nt ? zk1 : zk0;
                const uint32_t b0 = hsub2(prmt(u, kMagic, 0x4140), zb);
                const uint32_t b1 = hsub2(prmt(u, kMagic, 0x4342), zb);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t a[4];
                    const int arow = mt * 16 + (mat & 1) * 8 + mrow;
                    const int achk = 2 * ks + (mat >> 1);
                    pa::ldmatrix_x4(qtile + arow * Lay::kQPitch + achk * 16, a[0], a[1], a[2],
                                    a[3]);
                    mma_f16(sacc[mt][nt], a, b0, b1);
                }
            }
        }

        // ---- scales, mask, online softmax ----
        float ks4[2][2], vs4[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = nt * 8 + 2 * qc + e;
                ks4[nt][e] = ksc[t];
                vs4[nt][e] = t < valid ? vsc[t] : 0.f;
            }
        float vmax = fmaxf(fmaxf(vs4[0][0], vs4[0][1]), fmaxf(vs4[1][0], vs4[1][1]));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
        const int ev_new = max(ev, ceil_log2(vmax));
        const float vfix = exp2i(ev - ev_new);   // exact rescale of O to the new reference
        ev = ev_new;
        const float inv_vref = exp2i(-ev);
        const bool need_mask = tok0 + kBS - 1 > last_q;
        float alpha[MT][2];
        bool rescale = vfix != 1.f;
        uint32_t pa_[MT][4];
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
                        float v = sacc[mt][nt][2 * h + e] * (rowmul[mt][h] * ks4[nt][e]);
                        if (need_mask && tok0 + nt * 8 + 2 * qc + e > bound) v = -INFINITY;
                        sacc[mt][nt][2 * h + e] = v;
                        mx = fmaxf(mx, v);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[mt][h], mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float al = pa::ex2(m_run[mt][h] - m_use);
                m_run[mt][h] = m_new;
                float sum = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float pv = pa::ex2(sacc[mt][nt][2 * h + e] - m_use);
                        sum += pv;
                        sacc[mt][nt][2 * h + e] = pv * vs4[nt][e] * inv_vref;
                    }
                l_run[mt][h] = l_run[mt][h] * al + sum;
                alpha[mt][h] = al * vfix;
                rescale |= al != 1.f;
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
            __half2 h0 = __floats2half2_rn(sacc[mt][0][0], sacc[mt][0][1]);
            __half2 h1 = __floats2half2_rn(sacc[mt][0][2], sacc[mt][0][3]);
            __half2 h2 = __floats2half2_rn(sacc[mt][1][0], sacc[mt][1][1]);
            __half2 h3 = __floats2half2_rn(sacc[mt][1][2], sacc[mt][1][3]);
            pa_[mt][0] = *reinterpret_cast<uint32_t*>(&h0);
            pa_[mt][1] = *reinterpret_cast<uint32_t*>(&h1);
            pa_[mt][2] = *reinterpret_cast<uint32_t*>(&h2);
            pa_[mt][3] = *reinterpret_cast<uint32_t*>(&h3);
        }

        // ---- O += P' (V codes - zp) ----
        const uint32_t zv0 = zp_bias(vzp[2 * qc], vzp[2 * qc + 1]);
        const uint32_t zv1 = zp_bias(vzp[8 + 2 * qc], vzp[9 + 2 * qc]);
#pragma unroll
        for (int pch = 0; pch < kChunks / 2; ++pch) {
            uint32_t r0, r1, r2, r3;
            pa::ldmatrix_x4_trans(vb + tile8_offset<D>(ld_tok, 2 * pch + ld_chk), r0, r1, r2,
                                  r3);
            // r0: chunk 2pch tokens 0-7 (bytes t0d0 t0d1 t1d0 t1d1), r1: tokens 8-15,
            // r2, r3: chunk 2pch + 1
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int c = 2 * pch + half;
                const uint32_t u0 = (half ? r2 : r0) ^ 0x80808080u;
                const uint32_t u1 = (half ? r3 : r1) ^ 0x80808080u;
                const uint32_t xb0 = hsub2(prmt(u0, kMagic, 0x4240), zv0);   // even dims
                const uint32_t yb0 = hsub2(prmt(u0, kMagic, 0x4341), zv0);   // odd dims
                const uint32_t xb1 = hsub2(prmt(u1, kMagic, 0x4240), zv1);
                const uint32_t yb1 = hsub2(prmt(u1, kMagic, 0x4341), zv1);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    mma_f16(o[mt][2 * c], pa_[mt], xb0, xb1);
                    mma_f16(o[mt][2 * c + 1], pa_[mt], yb0, yb1);
                }
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
            if (k == n - 1) break;
            next_segment(cur, cum, chunks, n_seqs, hkv);
            seg_b0 = 0;
            seg_first = false;
            start_segment();
        }
    }
    for (int k = consumed; k < issued; ++k)
        if (!pa::mbar_wait(bars + 8 * (k % S), (k / S) & 1, p.err, pa::ERR_WAIT_DRAIN)) break;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// INT8 cache as rows of head_dim bytes: [num_blocks * H_kv * 16][head_dim],
// box = one (block, kv head) tile of 16 rows, 128-byte (d = 128) or 64-byte
// (d = 64) swizzle.
pa_status make_map8(CUtensorMap* m, const void* cache, int num_blocks, int hkv, int d) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return pa::fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const uint64_t rows = (uint64_t)num_blocks * hkv * kBS;
    if (rows > 0x7fffffffull) return pa::fail(PA_ERR_UNSUPPORTED, "cache has too many rows for TMA");
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d};
    cuuint32_t box[2] = {(cuuint32_t)d, (cuuint32_t)kBS};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return pa::fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PA_OK;
}

struct Map8Cache {
    struct Entry {
        const void* ptr;
        int nb, hkv, d, dev;
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
            if (e[i].ptr == ptr && e[i].nb == nb && e[i].hkv == hkv && e[i].d == d &&
                e[i].dev == dev) {
                *out = e[i].map;
                return PA_OK;
            }
        CUtensorMap m;
        if (pa_status s = make_map8(&m, ptr, nb, hkv, d)) return s;
        e[next] = Entry{ptr, nb, hkv, d, dev, m};
        next = (next + 1) % 16;
        if (n < 16) ++n;
        *out = m;
        return PA_OK;
    }
};
Map8Cache g_maps8;

template <typename TQ, int D, int MT>
pa_status launch8(const pa::DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                  pa::sched::Params prm, const Q8Extra& x) {
    using Lay = Q8Layout<D, MT>;
    auto kern = paged_decode_int8_kernel<TQ, D, MT>;
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
                                                       a.head_dim, a.max_q_len, a.max_context_len);
    const int64_t workers = std::min<int64_t>((int64_t)ctas * sms * kWorkerWarps, shape.workers);
    prm.workers = (int)workers;
    const int grid = (int)((workers + kWorkerWarps - 1) / kWorkerWarps);
    if (pa_status s = pa::cuda_status(
            pa::launch_pdl(kern, dim3(grid), dim3(kWorkerWarps * 32), smem, a.stream, mk, mv, prm,
                           x),
            "int8 decode launch"))
        return s;
    // query rows a chunk can have: all its G * max_q_len rows, up to one tile
    const int row_slots = (int)std::min<int64_t>(shape.rows_per_tile,
                                                 (int64_t)(a.num_heads / a.num_kv_heads) *
                                                     a.max_q_len);
    const int64_t rctas = pa::sched::reduce_ctas(a.num_seqs, a.num_kv_heads, shape.max_chunks,
                                                 row_slots);
    if (rctas > 0x7fffffff) return pa::fail(PA_ERR_UNSUPPORTED, "reduce grid too large");
    return pa::cuda_status(pa::launch_pdl(pa::sched::segment_reduce_kernel<TQ, D>,
                                          dim3((unsigned)rctas), dim3(128), 0, a.stream, prm,
                                          (int)shape.max_chunks, row_slots),
                           "segment reduce launch");
}

template <typename TQ>
pa_status launch8_q(const pa::DecodeArgs& a, int mt, const CUtensorMap& mk,
                    const CUtensorMap& mv, const pa::sched::Params& prm, const Q8Extra& x) {
    if (a.head_dim == 128)
        return mt == 1 ? launch8<TQ, 128, 1>(a, mk, mv, prm, x) : launch8<TQ, 128, 2>(a, mk, mv, prm, x);
    return mt == 1 ? launch8<TQ, 64, 1>(a, mk, mv, prm, x) : launch8<TQ, 64, 2>(a, mk, mv, prm, x);
}

}  // namespace

namespace pa {

pa_status launch_decode_int8(const DecodeArgs& a) {
    if (a.partition_size != 0)
        return fail(PA_ERR_UNSUPPORTED, "INT8 caches use the balanced schedule (partition_size 0)");
    if (pa_status s = balanced_check(a)) return s;
    if (((uintptr_t)a.k_scale | (uintptr_t)a.v_scale | (uintptr_t)a.k_zp | (uintptr_t)a.v_zp) % 16)
        return fail(PA_ERR_INVALID_ARG, "k_scale, v_scale, k_zp and v_zp must be 16-byte aligned");
    const BalancedShape shape = balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads,
                                               a.head_dim, a.max_q_len, a.max_context_len);
    CUtensorMap mk, mv;
    if (pa_status s = g_maps8.get(&mk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim))
        return s;
    if (pa_status s = g_maps8.get(&mv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim))
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
    const int mt = shape.rows_per_tile / 16;
    if (a.q_dtype == PA_BF16) return launch8_q<__nv_bfloat16>(a, mt, mk, mv, b, x);
    return launch8_q<__half>(a, mt, mk, mv, b, x);
}

}  // namespace pa
