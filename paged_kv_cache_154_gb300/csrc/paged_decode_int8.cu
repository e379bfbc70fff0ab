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
// scale seen so far, rounded up), so that fp16 P' = P * scale_t / reference
// is never larger than P; a larger reference rescales O exactly, like the
// running max of the softmax.
//
// Work split: the balanced schedule of balanced.cuh with one CTA of four
// warps per share. Warp 0 streams each block's codes, scales and zero points
// into a ring of stages shared by the CTA (TMA for the code tiles, bulk copies
// for the scales); every warp reads the codes it needs straight from the
// stage with ldmatrix and turns them into fp16 (code - zp) in registers.
// With 32-row tiles warp (rh, th) computes query rows 16*rh .. +15 against
// tokens 8*th .. +7 of every block; with 16-row tiles warp (dh, th) computes
// all 16 rows against the same 8 tokens but only head-dim half dh of P V.
// Each warp runs its own online softmax; the two token halves merge at the
// end of every segment. The running max is updated lazily (only when a block
// raises it by more than 2^8), which keeps P <= 256 and makes rescaling O
// rare; l and O always share the same reference, so the result is exact.
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
constexpr int kStages = 6;
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

// D += A(16x8, row) * B(8x8, col), fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(b));
}

__device__ __forceinline__ void ldmatrix_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
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

// byte offset of 16-byte chunk `chunk` of token row `row` in a code tile as
// the tensor map writes it: 128-byte swizzle for d = 128, 64-byte for d = 64
template <int D>
__device__ __forceinline__ uint32_t tile8_offset(int row, int chunk) {
    if constexpr (D == 128) return row * 128 + ((chunk ^ (row & 7)) << 4);
    else return row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4);
}

// Shared memory after the schedule header: the stage ring (each stage a
// multiple of 1024 bytes, as TMA with swizzle needs), the stages' scale
// areas, the Q tile (fp16, padded pitch), the row factors, and the area where
// the token-half-1 warps hand their partial results to the token-half-0 warps.
template <int D, int MT>
struct Q8Layout {
    static constexpr int RT = 16 * MT;
    static constexpr int kCodes = kBS * D;                        // one K (or V) code tile
    static constexpr int kStage = ((2 * kCodes) + 1023) / 1024 * 1024;
    static constexpr int kScalesAt = kStages * kStage;
    static constexpr int kQAt = kScalesAt + kStages * kScaleBytes;
    static constexpr int kQPitch = D * 2 + 16;
    static constexpr int kRowMulAt = kQAt + RT * kQPitch;
    static constexpr int kMergeAt = kRowMulAt + RT * 4;
    static constexpr int kDW = MT == 2 ? D : D / 2;               // output dims per warp
    static constexpr int kNT = kDW / 8;                           // n-tiles per warp
    static constexpr int kMergeFloats = kNT * 128 + 48;           // O fragments, m[16], l[16], ev
    static constexpr int kBody = kMergeAt + 2 * kMergeFloats * 4;
    static_assert(kStage % 1024 == 0, "stages must keep 1024-byte alignment");
    static_assert(kQAt % 16 == 0 && kQPitch % 16 == 0 && kMergeAt % 16 == 0, "16-byte alignment");
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
__global__ void __launch_bounds__(kWorkerWarps * 32, 4)
    paged_decode_int8_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v,
                             const pa::sched::Params p, const Q8Extra x) {
    using namespace pa::sched;
    using Lay = Q8Layout<D, MT>;
    constexpr int S = kStages;
    constexpr int RT = Lay::RT;
    constexpr int KCH = D / 16;          // k-steps of Q K^T (16 dims each)
    constexpr int NT = Lay::kNT;
    constexpr int VCH = NT / 2;          // 16-dim chunks of V per warp
    static_assert(KCH % 4 == 0 && (VCH % 4 == 0 || VCH == 2), "chunk counts");
    // Q fragments stay in registers unless that would push the largest
    // variant past 128 registers (four CTAs per SM); then each block reads
    // them again from the Q tile, which is unchanged for the whole segment.
    constexpr bool kQRegs = !(D == 128 && MT == 2);
    constexpr int QA = kQRegs ? KCH : 1;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = pa::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const smem = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = lane >> 2, qc = lane & 3;
    const int mat = lane >> 3, mrow = lane & 7;
    const int grp = warp & 1, th = warp >> 1;          // row (or dim) half, token half
    const int rbase = MT == 2 ? 16 * grp : 0;          // first tile row of this warp
    const int cbase = MT == 2 ? 0 : grp * VCH;         // first V chunk of this warp
    const int hkv = p.num_kv_heads, G = p.group, n_seqs = p.num_seqs;
    int32_t* const cum = reinterpret_cast<int32_t*>(smem + kWorkerWarps * S * 8);
    uint8_t* const chunks = reinterpret_cast<uint8_t*>(cum + n_seqs + 1);
    const uint32_t full = base, empty = base + 8 * S;
    const int hdr = header_bytes(n_seqs, S);           // a multiple of 1024
    const uint32_t body = base + hdr;
    uint8_t* const bodyp = smem + hdr;
    const uint32_t qtile = body + Lay::kQAt;
    // this lane's ldmatrix address for the warp's A fragments of k-step 0
    // (k-step ks is 32 bytes further on)
    const uint32_t qfrag =
        qtile + (rbase + (mat & 1) * 8 + mrow) * Lay::kQPitch + (mat >> 1) * 16;
    float* const rowmul_p = reinterpret_cast<float*>(bodyp + Lay::kRowMulAt);
    float* const mg = reinterpret_cast<float*>(bodyp + Lay::kMergeAt) + grp * Lay::kMergeFloats;

    build_prefix(cum, chunks, p);
    const int64_t B = cum[n_seqs];
    const int64_t wid = blockIdx.x;                    // one share per CTA
    const int64_t W = share_count(p, B);
    const int64_t f0 = share_start(wid, B, W);
    const int64_t f1 = share_start(wid + 1, B, W);
    const int n = (int)(f1 - f0);
    if (tid == 0) write_merge_record(p, wid, 0, 0, 0);   // none unless set at the end
    if (wid >= W || n <= 0) return;            // uniform over the CTA

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            pa::mbar_init(full + 8 * i, 1);
            pa::mbar_init(empty + 8 * i, kWorkerWarps);
        }
        pa::fence_barrier_init();
        pa::prefetch_tensormap(&tmap_k);
        pa::prefetch_tensormap(&tmap_v);
    }
    __syncthreads();

    // Producer (warp 0): each lane keeps the (block * H_kv + kv head) tile
    // index of virtual block win + lane.
    int win = -32, my_tile = 0;
    auto refresh = [&](int wb) {
        win = wb;
        const int64_t f = f0 + wb + lane;
        my_tile = 0;
        if (f < f1) {
            const Pos q = locate(p, cum, chunks, f);
            int blk = __ldg(p.block_tables + (int64_t)q.s * p.max_blocks + q.b);
            if (blk < 0 || blk >= p.num_blocks) {
                if (p.err) atomicOr(p.err, pa::ERR_BAD_BLOCK);
                blk = 0;
            }
            my_tile = blk * hkv + q.g;
        }
    };
    auto issue = [&](int k) {   // warp 0, warp-uniform
        if (k >= win + 32) refresh(k & ~31);
        const int tile = __shfl_sync(0xffffffffu, my_tile, k - win);
        if (lane == 0) {
            const int st = k % S;
            const uint32_t bar = full + 8 * st;
            const uint32_t dst = body + st * Lay::kStage;
            const uint32_t sd = body + Lay::kScalesAt + st * kScaleBytes;
            pa::mbar_arrive_expect_tx(bar, 2 * Lay::kCodes + kScaleBytes);
            pa::tma_load_2d(dst, &tmap_k, 0, tile * kBS, bar);
            pa::tma_load_2d(dst + Lay::kCodes, &tmap_v, 0, tile * kBS, bar);
            bulk_load(sd, x.k_scale + (int64_t)tile * kBS, 64, bar);
            bulk_load(sd + 64, x.v_scale + (int64_t)tile * kBS, 64, bar);
            bulk_load(sd + 128, x.k_zp + (int64_t)tile * kBS, 16, bar);
            bulk_load(sd + 144, x.v_zp + (int64_t)tile * kBS, 16, bar);
        }
    };
    int issued = 0, consumed = 0;
    if (warp == 0)
        for (; issued < S && issued < n; ++issued) issue(issued);

    Pos cur = locate(p, cum, chunks, f0);
    float o[NT][4];
    float m_run[2], l_run[2], rowmul[2];
    uint32_t qa[QA][4];
    int ev = -126;                       // log2 of this warp's running V-scale reference
    int L = 0, r = 1, q0 = 0, rows = 0, row_off = 0, seg_b0 = cur.b;
    bool seg_first = true, aborted = false;

    // Segment start (all warps): the Q tile in fp16, each row scaled by
    // 2^(14 - e_row) with its dims in the MMA's k order; then every warp takes
    // its A fragments and row factors into registers.
    auto start_segment = [&]() {
        L = __ldg(p.context_lens + cur.s);
        r = query_run(p.qsl, cur.s, &q0);
        row_off = cur.c * RT;
        rows = min(RT, G * r - row_off);
        constexpr int EPL = D / 32;
        constexpr int RPW = RT / kWorkerWarps;      // rows built by each warp
        float v[RPW][EPL];
#pragma unroll
        for (int j = 0; j < RPW; ++j) {
            const int row = warp + kWorkerWarps * j;
#pragma unroll
            for (int e = 0; e < EPL; ++e) v[j][e] = 0.f;
            if (row < rows) {
                const int gr = row_off + row;
                const TQ* src = static_cast<const TQ*>(p.q) +
                                ((int64_t)(q0 + gr / G) * p.num_heads + cur.g * G + gr % G) * D +
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
        for (int j = 0; j < RPW; ++j) {
            const int row = warp + kWorkerWarps * j;
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
                asm volatile("st.shared.b32 [%0], %1;" ::"r"(rowb + (ch * 16 + 8 * b + 2 * a) * 2),
                             "r"(*reinterpret_cast<const uint32_t*>(&h)) : "memory");
            }
            if (lane == 0) rowmul_p[row] = row < rows ? p.scale_log2 * exp2i(ex - 14) : 0.f;
        }
        __syncthreads();
        if constexpr (kQRegs) {
#pragma unroll
            for (int ks = 0; ks < KCH; ++ks)
                pa::ldmatrix_x4(qfrag + ks * 32, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
        }
        rowmul[0] = rowmul_p[rbase + quad];
        rowmul[1] = rowmul_p[rbase + quad + 8];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
        ev = -126;
    };

    // Segment end (all warps): token half 1 hands (O, m, l, ev) to token half
    // 0 through shared memory; token half 0 merges and writes the output
    // (segment held whole) or the partial slot.
    auto finish_segment = [&](bool complete, int slot_idx, int tok_end) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
        }
        if (th == 1) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) mg[(nt * 4 + e) * 32 + lane] = o[nt][e];
            if (qc == 0) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    mg[NT * 128 + quad + 8 * h] = m_run[h];
                    mg[NT * 128 + 16 + quad + 8 * h] = l_run[h];
                }
            }
            if (lane == 0) mg[NT * 128 + 32] = __int_as_float(ev);
        }
        __syncthreads();
        if (th != 0) return;
        const int ev1 = __float_as_int(mg[NT * 128 + 32]);
        Slot sl(p.slots + (2 * wid + slot_idx) * (int64_t)p.slot_bytes, RT);
        if (!complete && warp == 0 && lane == 0) {
            sl.hdr[0] = cur.s;
            sl.hdr[1] = cur.g;
            sl.hdr[2] = cur.c;
            sl.hdr[3] = seg_b0 * kBS;
            sl.hdr[4] = tok_end;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = rbase + quad + 8 * h;
            if (row >= rows) continue;
            const float m1 = mg[NT * 128 + quad + 8 * h];
            const float l1 = mg[NT * 128 + 16 + quad + 8 * h];
            const float M = fmaxf(m_run[h], m1);
            const float Mu = M == -INFINITY ? 0.f : M;
            const float a0 = exp2f(m_run[h] - Mu), a1 = exp2f(m1 - Mu);
            const float w0 = a0 * exp2i(ev), w1 = a1 * exp2i(ev1);   // to true scale
            const float l = l_run[h] * a0 + l1 * a1;
            const float mul = complete ? 1.f / l : 1.f;
            int64_t obase = 0;
            if (complete) {
                const int gr = row_off + row;
                obase = ((int64_t)(q0 + gr / G) * p.num_heads + cur.g * G + gr % G) * D;
            } else if (qc == 0 && (MT == 2 || grp == 0)) {   // dim halves share m, l
                sl.m[row] = M;
                sl.l[row] = l;
            }
#pragma unroll
            for (int cc = 0; cc < VCH; ++cc) {
                // n-tile 2cc holds dims 16c + 4qc and + 2, n-tile 2cc+1 dims + 1 and + 3
                float t[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int nt = 2 * cc + (u & 1), e = 2 * h + (u >> 1);
                    t[u] = (o[nt][e] * w0 + mg[(nt * 4 + e) * 32 + lane] * w1) * mul;
                }
                const float4 v = make_float4(t[0], t[1], t[2], t[3]);
                const int col = 16 * (cbase + cc) + 4 * qc;
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

    for (int k = 0; k < n; ++k) {
        const int st = k % S;
        bool ok = false;
        if (!aborted)
            ok = __all_sync(0xffffffffu,
                            pa::mbar_wait(full + 8 * st, (k / S) & 1, p.err, pa::ERR_WAIT_FULL));
        if (!ok) aborted = true;
        if (ok) {
            if (warp == 0) consumed = k + 1;
            const uint32_t kb = body + st * Lay::kStage, vb = kb + Lay::kCodes;
            const uint8_t* sp = bodyp + Lay::kScalesAt + st * kScaleBytes;
            const float* ksc = reinterpret_cast<const float*>(sp);
            const float* vsc = ksc + 16;
            const int8_t* kzp = reinterpret_cast<const int8_t*>(sp + 128);
            const int8_t* vzp = kzp + 16;
            const int tok0 = cur.b * kBS;
            const int t0 = th * 8 + 2 * qc;             // this lane's first S column (token)

            // ---- S = Q (K codes - zp)^T over this warp's 8 tokens ----
            const int kt = th * 8 + quad;               // token of this lane's K fragment
            const uint32_t zk = zp_bias(kzp[kt], kzp[kt]);
            float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int pp = 0; pp < KCH / 4; ++pp) {
                uint32_t rr[4];
                pa::ldmatrix_x4(kb + tile8_offset<D>(th * 8 + mrow, 4 * pp + mat), rr[0], rr[1],
                                rr[2], rr[3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t u = rr[j] ^ 0x80808080u;
                    const uint32_t b0 = hsub2(prmt(u, kMagic, 0x4140), zk);
                    const uint32_t b1 = hsub2(prmt(u, kMagic, 0x4342), zk);
                    if constexpr (kQRegs) {
                        mma_f16(s, qa[4 * pp + j], b0, b1);
                    } else {
                        pa::ldmatrix_x4(qfrag + (4 * pp + j) * 32, qa[0][0], qa[0][1], qa[0][2],
                                        qa[0][3]);
                        mma_f16(s, qa[0], b0, b1);
                    }
                }
            }

            // ---- scales, mask, online softmax (lazy max) ----
            const float2 ks2 = *reinterpret_cast<const float2*>(ksc + t0);
            const float2 vs2 = *reinterpret_cast<const float2*>(vsc + t0);
            const int valid = L - tok0;
            const float vs0 = t0 < valid ? vs2.x : 0.f, vs1 = t0 + 1 < valid ? vs2.y : 0.f;
            float vmax = fmaxf(vs0, vs1);
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
            const int ev_new = max(ev, ceil_log2(vmax));
            const float vfix = exp2i(ev - ev_new);      // exact rescale of O to the new reference
            ev = ev_new;
            const float inv_vref = exp2i(-ev);
            const int last_q = L - r;
            const bool need_mask = tok0 + kBS - 1 > last_q;
            float alpha[2];
            bool rescale = vfix != 1.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = rbase + quad + 8 * h;
                float a0 = s[2 * h] * ks2.x, a1 = s[2 * h + 1] * ks2.y;
                if (need_mask) {
                    const int bound = min(last_q + (row_off + row) / G, L - 1);
                    if (tok0 + t0 > bound) a0 = -INFINITY;
                    if (tok0 + t0 + 1 > bound) a1 = -INFINITY;
                }
                float mx = fmaxf(a0, a1);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float rm = rowmul[h];             // > 0 for real rows
                const float m_blk = mx == -INFINITY ? -INFINITY : mx * rm;
                float al = 1.f;
                if (m_blk > m_run[h] + kLazyMax) {
                    al = pa::ex2(m_run[h] - m_blk);     // 0 while m_run is -inf
                    m_run[h] = m_blk;
                    rescale = true;
                }
                const float m_use = m_run[h] == -INFINITY ? 0.f : m_run[h];
                const float p0 = pa::ex2(fmaf(a0, rm, -m_use));
                const float p1 = pa::ex2(fmaf(a1, rm, -m_use));
                l_run[h] = l_run[h] * al + (p0 + p1);
                s[2 * h] = p0 * (vs0 * inv_vref);
                s[2 * h + 1] = p1 * (vs1 * inv_vref);
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
            __half2 h01 = __floats2half2_rn(s[0], s[1]);
            __half2 h23 = __floats2half2_rn(s[2], s[3]);
            const uint32_t pa0 = *reinterpret_cast<uint32_t*>(&h01);
            const uint32_t pa1 = *reinterpret_cast<uint32_t*>(&h23);

            // ---- O += P' (V codes - zp) over this warp's 8 tokens ----
            const uint32_t zv = zp_bias(vzp[t0], vzp[t0 + 1]);
            auto pv_chunk = [&](int cc, uint32_t reg) {
                // reg: tokens t0, t0 + 1 x dims 2*quad, 2*quad + 1 of the chunk
                const uint32_t u = reg ^ 0x80808080u;
                mma_f16_k8(o[2 * cc], pa0, pa1, hsub2(prmt(u, kMagic, 0x4240), zv));
                mma_f16_k8(o[2 * cc + 1], pa0, pa1, hsub2(prmt(u, kMagic, 0x4341), zv));
            };
            if constexpr (VCH >= 4) {
#pragma unroll
                for (int pp = 0; pp < VCH / 4; ++pp) {
                    uint32_t rr[4];
                    pa::ldmatrix_x4_trans(
                        vb + tile8_offset<D>(th * 8 + mrow, cbase + 4 * pp + mat), rr[0], rr[1],
                        rr[2], rr[3]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) pv_chunk(4 * pp + j, rr[j]);
                }
            } else {
                uint32_t r0, r1;
                ldmatrix_x2_trans(vb + tile8_offset<D>(th * 8 + mrow, cbase + (mat & 1)), r0, r1);
                pv_chunk(0, r0);
                pv_chunk(1, r1);
            }
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(empty + 8 * st);   // this warp is done with the stage
        }

        // refill the stage that block k - 1 used once every warp has released it
        if (warp == 0 && !aborted && k >= 1 && k - 1 + S < n) {
            const int kp = k - 1;
            const bool fr = __all_sync(
                0xffffffffu, pa::mbar_wait(empty + 8 * (kp % S), (kp / S) & 1, p.err,
                                           pa::ERR_WAIT_EMPTY));
            if (fr) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(kp + S);
                ++issued;
            } else {
                aborted = true;
            }
        }

        ++cur.b;
        const bool seg_done = cur.b == cur.nbs;
        if (seg_done || k == n - 1) {
            if (__syncthreads_or(aborted)) break;       // a CTA-wide decision
            finish_segment(seg_b0 == 0 && seg_done, seg_first ? 0 : 1, min(cur.b * kBS, L));
            if (k == n - 1) {
                if (tid == 0)
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

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------



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
                                                       a.head_dim, a.max_q_len, a.max_context_len,
                                                       pa::kTileInt8);
    // one share per CTA, every CTA resident at once
    const int64_t workers = std::min<int64_t>((int64_t)ctas * sms, shape.workers);
    prm.workers = (int)workers;
    if (pa_status s = pa::cuda_status(
            pa::launch_pdl(kern, dim3((unsigned)workers), dim3(kWorkerWarps * 32), smem, a.stream,
                           mk, mv, prm, x),
            "int8 decode launch"))
        return s;
    const int row_slots = (int)std::min<int64_t>(shape.rows_per_tile, (int64_t)(a.num_heads / a.num_kv_heads) *
                                                          a.max_q_len);
    return pa::cuda_status(pa::sched::launch_segment_reduce<TQ, D>(prm, (int)shape.max_chunks,
                                                                    row_slots, a.stream),
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
    const int mt = shape.rows_per_tile / 16;
    if (a.q_dtype == PA_BF16) return launch8_q<__nv_bfloat16>(a, mt, mk, mv, b, x);
    return launch8_q<__half>(a, mt, mk, mv, b, x);
}

}  // namespace pa
