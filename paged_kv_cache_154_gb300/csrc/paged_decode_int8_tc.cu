// Paged decode attention over an INT8 cache on the 5th-generation tensor
// cores (tcgen05, TMEM), for head_dim 128 and at least 32 query rows per KV
// head (MQA decode, verify runs).
//
// The cache holds codes x_q with one fp32 scale and int8 zero point per
// (token, kv head); a value is (x_q - zero_point) * scale ("cs336 lecture 10",
// Quantization). As in the mma.sync INT8 kernel the products run on
// (x_q - zp) exactly in fp16, with the scales applied outside them:
//
//   S[i][t] = scale_t * sum_j q_ij (x_q[t][j] - zp_t)      (column scale)
//   O[i][j] = sum_t (P[i][t] scale_t) (x_q[t][j] - zp_t)    (scale folded into P)
//
// Here the (x_q - zp) tiles are built once per block in shared memory, in
// the operand layout of the tensor cores, and shared by every query row:
//
//   warp 0      streams each 16-token block's K and V codes (TMA) and its
//               scales and zero points (plain loads, one group of four blocks
//               ahead) into a ring of block stages;
//   warps 1-8   (converters) turn the codes of a 64-token tile (warp pair c:
//               block c, one warp for K, one for V) into fp16 (code - zp)
//               with the 1024-bias trick, written 128-byte swizzled: K as the
//               K-major B operand of Q K^T, V as the MN-major B operand of
//               P V (three tile buffers);
//   warp 9      issues S = Q K^T (tcgen05.mma M128 N64 K16, Q fp16 in shared
//               memory) into one of two S buffers in TMEM and O += P V (M128
//               N128 K16, P read from TMEM);
//   warps 14-15 build Q of every segment piece (fp16, scaled rows) two
//               pieces ahead;
//   warps 10-13 (softmax) one thread per query row, only the warps holding
//               rows of the current segment work: S from TMEM, column scale,
//               causal mask, online softmax with a lazy running max and a
//               running power-of-two reference for the V scales (as in the
//               mma.sync kernel), P' = P * scale_t / reference written over S
//               as fp16 pairs; at a segment end O from TMEM, normalised
//               (segment held whole) or as a partial (m, l, O) slot.
//
// The work split is the balanced schedule (one share of virtual blocks per
// CTA, query rows in chunks of 128); cut segments are merged by the segment
// reduce kernel. q is converted to fp16 after an exact power-of-two scaling
// per row (its largest |q| into [2^14, 2^15)), undone on S. Every wait is
// bounded; a wait that gives up stops every role, and the MMA warp waits for
// its own operations before TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <math.h>
#include <stdlib.h>

#include <algorithm>
#include <type_traits>

#include "balanced.cuh"
#include "pa_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace {

using pa::sched::kBS;
using pa::sched::Pos;
constexpr int D = 128;
constexpr int kRows = 128;               // query rows per segment chunk (MMA M)
constexpr int kTok = 64;                 // keys per tile (S columns)
constexpr int kTileBlocks = kTok / kBS;  // 4
constexpr int kThreads = 512;            // producer, 8 converters, MMA, 4 softmax, 2 Q builders
constexpr int kMmaWarp = 9;
constexpr int kNS = 12;                  // block stages of the code ring
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyMax = 8.f;
constexpr uint32_t kMagic = 0x64646464u;
constexpr int kNB = 3;                   // operand tiles / S buffers in flight

// shared memory after the schedule header (offsets from a 1024-byte boundary)
constexpr int kQBytes = 32 * 1024;                  // Q fp16: [2 halves][128 rows][128 B]
constexpr int kQOff = 0;                            // two Q buffers
constexpr int kOpBytes = 16 * 1024;                 // one operand: [2 halves][64 tokens][128 B]
constexpr int kOpOff = 2 * kQBytes;                 // kNB x (K operand, V operand)
constexpr int kCodeStage = 4096;                    // K codes 2 KB, V codes 2 KB (TMA, swizzled)
constexpr int kCodeOff = kOpOff + 2 * kNB * kOpBytes;
constexpr int kScaleStage = 160;                    // k scale[16], v scale[16], k zp[16], v zp[16]
constexpr int kScaleOff = kCodeOff + kNS * kCodeStage;
// per operand buffer, one entry per key column: k scale, additive mask (0 or
// -inf: the token is past the context or the tile), v scale (0 when masked);
// then the largest v scale of each block's valid tokens
constexpr int kColBytes = (3 * kTok + 4) * 4;
constexpr int kTileScaleOff = kScaleOff + kNS * kScaleStage;
constexpr int kRowMulOff = kTileScaleOff + kNB * kColBytes;    // per Q buffer: rowmul[128]
constexpr int kBarOff = kRowMulOff + 2 * kRows * 4;
// barriers: code full / empty per stage; per buffer b: operands ready, S and
// P buffer free (P V of the buffer's tile done), S full, P full; per Q buffer:
// Q ready; per O buffer: O free; the final drain
constexpr int kBFull = 0, kBEmpty = kNS, kBOpReady = 2 * kNS, kBSpFree = 2 * kNS + kNB,
              kBSFull = 2 * kNS + 2 * kNB, kBPFull = 2 * kNS + 3 * kNB, kBQReady = 2 * kNS + 4 * kNB,
              kBOFree = 2 * kNS + 4 * kNB + 2, kBFin = 2 * kNS + 4 * kNB + 4;
constexpr int kNumBars = 2 * kNS + 4 * kNB + 5;
constexpr int kBodyBytes = kBarOff + 8 * kNumBars + 16;
// TMEM: O of segment parity o at 128o, S (and P over it) of buffer b at 256 + 64b (b < kNB)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 256;
static_assert(kCodeOff % 1024 == 0 && kOpOff % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(kScaleOff % 16 == 0 && kTileScaleOff % 16 == 0 && kColBytes % 16 == 0 &&
              kRowMulOff % 16 == 0 && kBarOff % 8 == 0, "alignment");

__host__ __device__ constexpr int header_bytes(int num_seqs) {
    return ((num_seqs + 1) * 4 + num_seqs + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int smem_bytes(int num_seqs) {
    return header_bytes(num_seqs) + kBodyBytes + 1024;
}
// the schedule header (prefix sums of the sequences) shares the 227 KB with
// the body: calls with more sequences take the mma.sync INT8 kernel
constexpr int kMaxSeqs = 2048;
static_assert(smem_bytes(kMaxSeqs) + 128 <= 232448, "shared memory budget");

struct TcExtra {
    const float* k_scale;
    const float* v_scale;
    const int8_t* k_zp;
    const int8_t* v_zp;
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

// fp16 pair (1152 + zp, 1152 + zp): subtracted from (1024 + (code ^ 0x80))
// it leaves code - zp exactly
__device__ __forceinline__ uint32_t zp_bias(int zp) {
    const __half h = __int2half_rn(1152 + zp);
    const __half2 hh = __halves2half2(h, h);
    return *reinterpret_cast<const uint32_t*>(&hh);
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

// packed two-lane fp32 arithmetic (one instruction for two values)
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float4 lds4(const float* p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(pa::smem_addr(p)));
    return v;
}

// byte offset of 16-byte chunk c (0..7) of row `row` in a 128-byte-wide,
// 128-byte-swizzled matrix (8-row atoms of 1024 bytes)
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return row * 128 + ((c ^ (row & 7)) << 4);
}

// The tiles of a share, in order: within each segment piece (the blocks of
// one segment inside the share) tiles of up to four blocks.
struct TileWalk {
    Pos cur;          // segment of the tile; cur.b = its first block
    int left;         // blocks of the share from this tile on
    int piece_end;    // one past the last block of the piece
    int seg_b0;       // first block of the piece
    int j;            // segment piece index within the share
    int t;            // tile index within the share
    int nb;           // blocks of this tile
    __device__ void init(const pa::sched::Params& p, const int32_t* cum, const uint8_t* chunks,
                         int64_t f0, int n) {
        cur = pa::sched::locate(p, cum, chunks, f0);
        left = n;
        seg_b0 = cur.b;
        piece_end = min(cur.nbs, cur.b + n);
        j = 0;
        t = 0;
        nb = min(kTileBlocks, piece_end - cur.b);
        if (nb <= 0) left = 0;   // inconsistent schedule: no tiles rather than no progress
    }
    __device__ bool first() const { return cur.b == seg_b0; }
    __device__ bool last() const { return cur.b + nb == piece_end; }
    __device__ bool valid() const { return left > 0; }
    __device__ void next(const pa::sched::Params& p, const int32_t* cum, const uint8_t* chunks) {
        left -= nb;
        ++t;
        if (left <= 0) return;
        if (cur.b + nb == piece_end) {
            pa::sched::next_segment(p, cur, cum, chunks);
            seg_b0 = 0;
            piece_end = min(cur.nbs, left);
            ++j;
        } else {
            cur.b += nb;
        }
        nb = min(kTileBlocks, piece_end - cur.b);
        if (nb <= 0) left = 0;
    }
};

template <typename TQ>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_int8_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                const __grid_constant__ CUtensorMap tmap_v,
                                const pa::sched::Params p, const TcExtra x) {
    using namespace pa::sched;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = pa::smem_addr(smem_raw);
    const uint32_t base0 = (raw + 1023u) & ~1023u;
    uint8_t* const smem0 = smem_raw + (base0 - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_seqs = p.num_seqs;
    int32_t* const cum = reinterpret_cast<int32_t*>(smem0);
    uint8_t* const chunks = reinterpret_cast<uint8_t*>(cum + n_seqs + 1);
    const int hdr = header_bytes(n_seqs);
    const uint32_t base = base0 + hdr;                 // body (1024-aligned)
    uint8_t* const smem = smem0 + hdr;
    const uint32_t bars = base + kBarOff;
    uint32_t* const tmem_holder = reinterpret_cast<uint32_t*>(smem + kBarOff + 8 * kNumBars);
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(smem + kBarOff + 8 * kNumBars + 8);
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };

    build_prefix(cum, chunks, p);                      // also waits for the previous kernel
    const int64_t B = cum[n_seqs];
    const int64_t wid = blockIdx.x;                    // one share per CTA
    const int64_t W = share_count(p, B);
    const int64_t f0 = share_start(wid, B, W);
    const int64_t f1 = share_start(wid + 1, B, W);
    const int n = (int)(f1 - f0);
    if (tid == 0) write_merge_record(p, wid, 0, 0, 0);   // none unless set at the end
    if (wid >= W || n <= 0) return;            // uniform over the CTA

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t cnt = 1;
            if (i >= kBOpReady && i < kBOpReady + kNB) cnt = 8;          // the converter warps
            if (i >= kBEmpty && i < kBEmpty + kNS) cnt = 2;              // a block's K and V warps
            if (i >= kBFull && i < kBFull + kNS) cnt = 2;                // code copies, scale stores
            if (i >= kBPFull && i < kBFin) cnt = 4;                      // the softmax warps
            if (i >= kBQReady && i < kBQReady + 2) cnt = 2;              // the Q builders
            pa::mbar_init(bar(i), cnt);
        }
        *abort_flag = 0;
        pa::fence_barrier_init();
        pa::prefetch_tensormap(&tmap_k);
        pa::prefetch_tensormap(&tmap_v);
    }
    if (warp == kMmaWarp) {
        pa::tc::tmem_alloc(pa::smem_addr(tmem_holder), kTmemCols);
        pa::tc::tmem_relinquish();
    }
    pa::tc::fence_before_sync();
    __syncthreads();
    pa::tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    const int hkv = p.num_kv_heads;

    if (warp == 0) {
        // ---------------- producer: codes, scales and zero points of every block ----------------
        // Blocks in groups of four. Lane l keeps the (block * H_kv + kv head)
        // index of share-local block win + l (one round of loads per 32
        // blocks). Each copy request costs the copy engine about a hundred
        // cycles, so only the code tiles go by TMA (two per block); the
        // scales and zero points (160 bytes a block) are plain loads, issued
        // one group ahead and stored into the stage, which then takes a
        // second arrival.
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
        // lane l: block l / 8 of the group, 16 bytes (part l % 8) of its k scales
        // (parts 0-3) or v scales (4-7); lanes 0-7 also the k (even) or v (odd)
        // zero points of block l / 2
        auto tile_of = [&](int k) {               // block k must lie in the window
            return __shfl_sync(0xffffffffu, my_tile, (k - win) & 31);
        };
        auto load_scales = [&](int g0, uint4& sv, uint4& zv) {
            const int nbg = min(4, n - g0);
            const int ts = tile_of(g0 + min(lane >> 3, nbg - 1));
            const int tz = tile_of(g0 + min((lane & 7) >> 1, nbg - 1));
            sv = make_uint4(0, 0, 0, 0);
            zv = make_uint4(0, 0, 0, 0);
            if ((lane >> 3) < nbg) {
                const int part = lane & 7;
                const float* src = (part < 4 ? x.k_scale : x.v_scale) + (int64_t)ts * kBS + 4 * (part & 3);
                sv = __ldg(reinterpret_cast<const uint4*>(src));
            }
            if (lane < 8 && (lane >> 1) < nbg)
                zv = __ldg(reinterpret_cast<const uint4*>((lane & 1 ? x.v_zp : x.k_zp) + (int64_t)tz * kBS));
        };
        int issued = 0;
        refresh(0);
        uint4 sv_cur, zv_cur;
        load_scales(0, sv_cur, zv_cur);
        for (int k0 = 0; k0 < n; k0 += 4) {
            const int nb = min(4, n - k0);
            // the stages are free once their converters are done with blocks k - kNS
            bool ok = true;
            if (lane < nb && k0 + lane >= kNS) {
                const int k = k0 + lane;
                ok = pa::mbar_wait(bar(kBEmpty + k % kNS), ((k / kNS) - 1) & 1, p.err, pa::ERR_WAIT_EMPTY);
            }
            ok = __all_sync(0xffffffffu, ok);
            if (!ok || *abort_flag) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            // the converters read the stages with ordinary loads; the copies write them
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const int ti = tile_of(k0 + (lane < nb ? lane : 0));
            if (lane < nb) {
                const int st = (k0 + lane) % kNS;
                const uint32_t full = bar(kBFull + st);
                const uint32_t dst = base + kCodeOff + st * kCodeStage;
                pa::mbar_arrive_expect_tx(full, kCodeStage);
                pa::tma_load_2d(dst, &tmap_k, 0, ti * kBS, full);
                pa::tma_load_2d(dst + kCodeStage / 2, &tmap_v, 0, ti * kBS, full);
            }
            // this group's scales and zero points (loaded one group ago) into the stages
            if ((lane >> 3) < nb) {
                const int st = (k0 + (lane >> 3)) % kNS, part = lane & 7;
                uint8_t* d = smem + kScaleOff + st * kScaleStage + (part < 4 ? 16 * part : 64 + 16 * (part - 4));
                *reinterpret_cast<uint4*>(d) = sv_cur;
            }
            if (lane < 8 && (lane >> 1) < nb) {
                const int st = (k0 + (lane >> 1)) % kNS;
                *reinterpret_cast<uint4*>(smem + kScaleOff + st * kScaleStage + 128 + 16 * (lane & 1)) = zv_cur;
            }
            __syncwarp();
            if (lane < nb) pa::mbar_arrive(bar(kBFull + (k0 + lane) % kNS));
            issued = k0 + nb;
            // the next group's indices and scales
            if (k0 + 4 < n) {
                if (k0 + 4 + min(4, n - k0 - 4) > win + 32) refresh(k0 + 4);
                load_scales(k0 + 4, sv_cur, zv_cur);
            }
        }
        // no copy may be in flight when the CTA ends: the last kNS issued
        // blocks are waited once more (earlier ones were consumed before
        // their stage was reused)
        if (lane == 0)
            for (int k = issued > kNS ? issued - kNS : 0; k < issued; ++k)
                if (!pa::mbar_wait(bar(kBFull + k % kNS), (k / kNS) & 1, nullptr, 0)) {
                    if (p.err) atomicOr(p.err, pa::ERR_WAIT_DRAIN);
                    break;
                }
    } else if (warp <= 8) {
        // ---------------- converters: warp (c, kv) turns the K (kv = 0) or V codes of
        // block c of each tile into fp16 operands ----------------
        const int c = (warp - 1) >> 1, kvw = (warp - 1) & 1;
        TileWalk w;
        w.init(p, cum, chunks, f0, n);
        int k0 = 0;                                    // share-local index of the tile's first block
        int L = 0;
        for (; w.valid(); w.next(p, cum, chunks)) {
            if (w.first()) L = __ldg(p.context_lens + w.cur.s);
            const int t = w.t, b = t % kNB, nb = w.nb;
            if (t >= kNB) {   // the operand buffer is free once the P V product of tile t - kNB is done
                const bool ok = __all_sync(0xffffffffu, pa::mbar_wait(bar(kBSpFree + b),
                                                                      ((t / kNB) - 1) & 1, p.err,
                                                                      pa::ERR_WAIT_FULL));
                if (!ok || *abort_flag) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
            }
            const uint32_t kop = base + kOpOff + b * 2 * kOpBytes, vop = kop + kOpBytes;
            float* const ks_col = reinterpret_cast<float*>(smem + kTileScaleOff + b * kColBytes);
            float* const madd_col = ks_col + kTok;
            float* const vs_col = madd_col + kTok;
            float* const vmax_blk = vs_col + kTok;
            const int k = k0 + c, st = k % kNS;
            if (c < nb) {
                const bool ok = __all_sync(0xffffffffu, pa::mbar_wait(bar(kBFull + st), (k / kNS) & 1,
                                                                      p.err, pa::ERR_WAIT_FULL));
                if (!ok || *abort_flag) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
                const uint32_t kc = base + kCodeOff + st * kCodeStage, vc = kc + kCodeStage / 2;
                const uint8_t* sp = smem + kScaleOff + st * kScaleStage;
                const int8_t* kzp = reinterpret_cast<const int8_t*>(sp + 128);
                const int8_t* vzp = kzp + 16;
                // 16 tokens x 8 chunks of 16 codes: item e = lane + 32 i (loads first)
                const uint32_t src = kvw ? vc : kc, dst = kvw ? vop : kop;
                const int8_t* zp = kvw ? vzp : kzp;
                uint32_t u[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = lane + 32 * i;
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(u[i][0]), "=r"(u[i][1]), "=r"(u[i][2]), "=r"(u[i][3])
                                 : "r"(src + sw128(e >> 3, e & 7)));
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int e = lane + 32 * i, tr = e >> 3, cc = e & 7;
                    const uint32_t zb = zp_bias(zp[tr]);
                    uint32_t h[8];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t v = u[i][q] ^ 0x80808080u;
                        h[2 * q] = hsub2(prmt(v, kMagic, 0x4140), zb);      // codes 4q, 4q + 1
                        h[2 * q + 1] = hsub2(prmt(v, kMagic, 0x4342), zb);  // codes 4q + 2, 4q + 3
                    }
                    // dims 16 cc .. + 15: half cc / 4, 16-byte chunks 2 (cc % 4) and + 1
                    const int row = 16 * c + tr;
                    const uint32_t d0 = dst + (cc >> 2) * (kTok * 128) + sw128(row, 2 * (cc & 3));
                    const uint32_t d1 = dst + (cc >> 2) * (kTok * 128) + sw128(row, 2 * (cc & 3) + 1);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(d0), "r"(h[0]),
                                 "r"(h[1]), "r"(h[2]), "r"(h[3])
                                 : "memory");
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(d1), "r"(h[4]),
                                 "r"(h[5]), "r"(h[6]), "r"(h[7])
                                 : "memory");
                }
                // key columns of this block: scales, and the mask of tokens past the context
                const bool valid = lane < 16 && w.cur.b * kBS + 16 * c + lane < L;
                if (kvw == 0) {
                    if (lane < 16) {
                        ks_col[16 * c + lane] = valid ? reinterpret_cast<const float*>(sp)[lane] : 0.f;
                        madd_col[16 * c + lane] = valid ? 0.f : -INFINITY;
                    }
                } else {
                    const float vsv = valid ? reinterpret_cast<const float*>(sp + 64)[lane] : 0.f;
                    if (lane < 16) vs_col[16 * c + lane] = vsv;
                    float vm = vsv;
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
                    if (lane == 0) vmax_blk[c] = vm;
                }
            } else {
                // no block c in this tile: its columns are masked; zero its K
                // (or V) rows (stale shared memory might hold NaN patterns, and
                // a masked column is S * 0 - inf)
                const uint32_t dst = kvw ? vop : kop;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int e = lane + 32 * i, hh = e >> 7, tr = (e >> 3) & 15, cc = e & 7;
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};"
                                 ::"r"(dst + hh * (kTok * 128) + (16 * c + tr) * 128 + cc * 16), "r"(0u)
                                 : "memory");
                }
                if (kvw == 0) {
                    if (lane < 16) {
                        ks_col[16 * c + lane] = 0.f;
                        madd_col[16 * c + lane] = -INFINITY;
                    }
                } else {
                    if (lane < 16) vs_col[16 * c + lane] = 0.f;
                    if (lane == 0) vmax_blk[c] = 0.f;
                }
            }
            // the operands are read by the tensor cores (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                pa::mbar_arrive(bar(kBOpReady + b));
                if (c < nb) pa::mbar_arrive(bar(kBEmpty + st));
            }
            k0 += nb;
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue (the whole warp; one elected lane issues) ----------------
        // QK(t + 1) is issued before PV(t) when its operands are ready, so each
        // softmax finds its next S ready; otherwise PV(t) goes first (it frees
        // an operand buffer for the converters). QK(t) writes S buffer t % kNB
        // once PV(t - kNB) (which read P from it) is done; the first PV of
        // segment piece j overwrites O buffer j & 1 once the epilogue of piece
        // j - 2 has read it.
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        const uint32_t sb = __shfl_sync(0xffffffffu, base, 0);
        const uint32_t bb = sb + kBarOff;
        constexpr uint32_t idesc_qk = pa::tc::idesc_f16(false, false, false, kRows, kTok);
        constexpr uint32_t idesc_pv = pa::tc::idesc_f16(false, false, true, kRows, D);
        auto wait = [&](int i, uint32_t parity) -> bool {
            const uint32_t b_ = bb + 8u * (uint32_t)i;
            if (__all_sync(0xffffffffu, pa::mbar_try_wait(b_, parity))) return true;
            const bool ok = __all_sync(0xffffffffu, pa::mbar_wait(b_, parity, p.err, pa::ERR_WAIT_FULL));
            return ok && __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
        };
        // descriptors: a descriptor of address a + o is the one of a plus o >> 4
        const uint64_t dq = pa::tc::smem_desc_sw128(sb + kQOff, 16, 1024);
        const uint64_t dk = pa::tc::smem_desc_sw128(sb + kOpOff, 16, 1024);
        const uint64_t dv = pa::tc::smem_desc_sw128(sb + kOpOff + kOpBytes, kTok * 128, 1024);
        auto issue_qk = [&](const TileWalk& w) -> bool {   // S[t % kNB] = Q_j K(t)^T
            const int t = w.t, b = t % kNB, j = w.j;
            if (!wait(kBOpReady + b, (t / kNB) & 1)) return false;
            if (t >= kNB && !wait(kBSpFree + b, ((t / kNB) - 1) & 1)) return false;
            if (w.first() && !wait(kBQReady + (j & 1), (j >> 1) & 1)) return false;
            pa::tc::fence_after_sync();
            const uint64_t a0 = dq + (uint64_t)(((j & 1) * kQBytes) >> 4);
            const uint64_t b0 = dk + (uint64_t)((b * 2 * kOpBytes) >> 4);
            const uint32_t d = tm + kSCol + 64 * b;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t qa = ((kk >> 2) * (kRows * 128) + (kk & 3) * 32) >> 4;
                const uint32_t ka = ((kk >> 2) * (kTok * 128) + (kk & 3) * 32) >> 4;
                pa::tc::mma_f16_ss_warp(d, a0 + qa, b0 + ka, idesc_qk, kk > 0 ? 1u : 0u);
            }
            pa::tc::commit_warp(bb + 8u * (kBSFull + b));
            return true;
        };
        auto issue_pv = [&](const TileWalk& w) -> bool {   // O_j += P(t) V(t)
            const int t = w.t, b = t % kNB, j = w.j;
            if (!wait(kBPFull + b, (t / kNB) & 1)) return false;
            if (w.first() && j >= 2 && !wait(kBOFree + (j & 1), ((j >> 1) - 1) & 1)) return false;
            pa::tc::fence_after_sync();
            const uint64_t v0 = dv + (uint64_t)((b * 2 * kOpBytes) >> 4);
            const uint32_t o = tm + 128 * (j & 1), pc = tm + kSCol + 64 * b;
            const uint32_t acc0 = w.first() ? 0u : 1u;
#pragma unroll
            for (int kb = 0; kb < kTileBlocks; ++kb)
                if (kb < w.nb)
                    pa::tc::mma_f16_ts_warp(o, pc + 8 * kb, v0 + (uint64_t)((kb * kBS * 128) >> 4),
                                            idesc_pv, kb > 0 ? 1u : acc0);
            pa::tc::commit_warp(bb + 8u * (kBSpFree + b));
            return true;
        };
        TileWalk wq, wp;
        wq.init(p, cum, chunks, f0, n);
        wp = wq;
        bool ok = issue_qk(wq);
        wq.next(p, cum, chunks);
        while (ok && wp.valid()) {
            const bool qk_first =
                wq.valid() && __all_sync(0xffffffffu, pa::mbar_try_wait(bb + 8u * (kBOpReady + wq.t % kNB),
                                                                         (wq.t / kNB) & 1));
            if (!qk_first) {
                ok = issue_pv(wp);
                wp.next(p, cum, chunks);
            }
            if (ok && wq.valid()) {
                ok = issue_qk(wq);
                wq.next(p, cum, chunks);
            }
            if (ok && qk_first) {
                ok = issue_pv(wp);
                wp.next(p, cum, chunks);
            }
        }
        if (!ok && lane == 0) *abort_flag = 1;
        // every MMA this warp issued has finished before TMEM is freed
        pa::tc::commit_warp(bb + 8u * kBFin);
        if (!__all_sync(0xffffffffu, pa::mbar_wait(bb + 8u * kBFin, 0, nullptr, 0)) && lane == 0 && p.err)
            atomicOr(p.err, pa::ERR_WAIT_DRAIN);
    } else if (warp >= 14) {
        // ---------------- Q builders (warps 14, 15): Q of every piece, two pieces ahead ----------------
        // fp16 rows scaled by 2^(14 - e), e = floor(log2 max|q|) of the row;
        // a half-warp per row (lane: one 16-byte chunk of 8 elements), four
        // rows per round, loads of up to eight rounds in flight; padding rows
        // zero. Piece j goes to Q buffer j & 1 once the epilogue of piece
        // j - 2 is done (all its products of S have completed).
        const int qt = (warp - 14) * 32 + lane;            // 0..63
        const int ch = qt & 15, sub = qt >> 4;             // chunk, row within a round of 4
        const int G = p.group;
        float* const rowmul_s = reinterpret_cast<float*>(smem + kRowMulOff);
        TileWalk wq;
        wq.init(p, cum, chunks, f0, n);
        for (int j = 0; wq.valid(); ++j) {
            if (j >= 2 && (!__all_sync(0xffffffffu, pa::mbar_wait(bar(kBOFree + (j & 1)), ((j >> 1) - 1) & 1,
                                                                   p.err, pa::ERR_WAIT_FULL)) ||
                           *abort_flag)) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            const int qb = j & 1;
            int q0;
            const int r = query_run(p.qsl, wq.cur.s, &q0);
            const int rows = min(kRows, G * r - wq.cur.c * kRows);
            const uint32_t qbase = base + kQOff + qb * kQBytes;
            for (int r0 = 0; r0 < kRows; r0 += 32) {      // eight rounds of four rows
                uint4 v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = r0 + 4 * i + sub;
                    v[i] = make_uint4(0, 0, 0, 0);
                    if (row < rows) {
                        const int gr = wq.cur.c * kRows + row;
                        v[i] = __ldg(reinterpret_cast<const uint4*>(
                                         static_cast<const TQ*>(p.q) +
                                         ((int64_t)(q0 + gr / G) * p.num_heads + wq.cur.g * G + gr % G) * D) +
                                     ch);
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = r0 + 4 * i + sub;
                    const TQ* e = reinterpret_cast<const TQ*>(&v[i]);
                    float mx = 0.f;
#pragma unroll
                    for (int u = 0; u < 8; ++u) mx = fmaxf(mx, fabsf((float)e[u]));
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                    int ex = 0;
                    if (mx > 0.f) ex = max(-100, min(100, (int)((__float_as_uint(mx) >> 23) & 0xff) - 127));
                    const float up = exp2i(14 - ex);
                    uint32_t h[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const __half2 hh = __floats2half2_rn((float)e[2 * u] * up, (float)e[2 * u + 1] * up);
                        h[u] = *reinterpret_cast<const uint32_t*>(&hh);
                    }
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};"
                                 ::"r"(qbase + (ch >> 3) * (kRows * 128) + sw128(row, ch & 7)), "r"(h[0]),
                                 "r"(h[1]), "r"(h[2]), "r"(h[3])
                                 : "memory");
                    // padding rows: Q = 0, S = 0, factor 1
                    if (ch == 0) rowmul_s[qb * kRows + row] = row < rows ? p.scale_log2 * exp2i(ex - 14) : 1.f;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(bar(kBQReady + qb));
            while (wq.valid() && wq.j == j) wq.next(p, cum, chunks);
        }
    } else {
        // ---------------- softmax (warps 10-13): one thread per query row ----------------
        const int lane_base = 32 * (warp & 3);
        const int row = lane_base + lane;                  // tile row = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)lane_base << 16);
        const int G = p.group;
        float* const rowmul_s = reinterpret_cast<float*>(smem + kRowMulOff);

        TileWalk w;
        w.init(p, cum, chunks, f0, n);
        int L = 0, r = 1, q0 = 0, rows = 0, bound = 0, bound_min = 0, ev = -126;
        float m_run = -INFINITY, l_run = 0.f, rowmul = 0.f;
        bool active = false, aborted = false;
        for (; w.valid(); w.next(p, cum, chunks)) {
            const int t = w.t, b = t % kNB, j = w.j;
            if (w.first()) {
                // Q and the row factors of this piece are built
                if (!__all_sync(0xffffffffu, pa::mbar_wait(bar(kBQReady + (j & 1)), (j >> 1) & 1, p.err,
                                                           pa::ERR_WAIT_FULL)) || *abort_flag) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
                L = __ldg(p.context_lens + w.cur.s);
                r = query_run(p.qsl, w.cur.s, &q0);
                rows = min(kRows, G * r - w.cur.c * kRows);
                active = lane_base < rows;
                const int jq = (w.cur.c * kRows + min(row, rows - 1)) / G;
                bound = row < rows ? min(L - r + jq, L - 1) : L - 1;
                // the smallest bound of the piece's rows (columns past L are masked already)
                bound_min = min(L - r + (w.cur.c * kRows) / G, L - 1);
                rowmul = rowmul_s[(j & 1) * kRows + row];
                m_run = -INFINITY;
                l_run = 0.f;
                ev = -126;
            }
            bool ok = __all_sync(0xffffffffu, pa::mbar_wait(bar(kBSFull + b), (t / kNB) & 1, p.err,
                                                            pa::ERR_WAIT_FULL)) &&
                      __all_sync(0xffffffffu, pa::mbar_wait(bar(kBOpReady + b), (t / kNB) & 1, p.err,
                                                            pa::ERR_WAIT_FULL));
            if (!ok || *abort_flag) {
                if (lane == 0) *abort_flag = 1;
                aborted = true;
                break;
            }
            pa::tc::fence_after_sync();
            if (active) {
                const uint32_t s_tm = trow + kSCol + 64 * b;
                const float* col = reinterpret_cast<const float*>(smem + kTileScaleOff + b * kColBytes);
                float sv[kTok];
                pa::tc::ld_64cols(s_tm, *reinterpret_cast<uint32_t(*)[64]>(sv));
                // a = S * k_scale + mask (0, or -inf for tokens past the context or the tile)
#pragma unroll
                for (int c = 0; c < kTok; c += 4) {
                    const float4 k4 = lds4(col + c), m4 = lds4(col + kTok + c);
                    fma2(sv[c], sv[c + 1], sv[c], sv[c + 1], k4.x, k4.y, m4.x, m4.y);
                    fma2(sv[c + 2], sv[c + 3], sv[c + 2], sv[c + 3], k4.z, k4.w, m4.z, m4.w);
                }
                // query i of a verify run sees keys up to L - r + i
                const int tok0 = w.cur.b * kBS;
                if (tok0 + kTok - 1 > bound_min) {
#pragma unroll
                    for (int c = 0; c < kTok; ++c)
                        if (tok0 + c > bound) sv[c] = -INFINITY;
                }
                float m4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
                for (int c = 4; c < kTok; c += 8)
#pragma unroll
                    for (int u = 0; u < 4; ++u) m4[u] = max3(m4[u], sv[c + 2 * u], sv[c + 2 * u + 1]);
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                const float m_blk = mx == -INFINITY ? -INFINITY : mx * rowmul;
                const float4 vb4 = lds4(col + 3 * kTok);
                const float vmax = fmaxf(fmaxf(vb4.x, vb4.y), fmaxf(vb4.z, vb4.w));
                // V-scale reference 2^ev and running max m: l (kept in the
                // reference's units, like O) and O follow both exactly
                const int ev_new = max(ev, ceil_log2(vmax));
                const float vfix = exp2i(ev - ev_new);
                ev = ev_new;
                float am = 1.f;
                if (m_blk > m_run + kLazyMax) {
                    am = pa::ex2(m_run - m_blk);           // 0 while m_run is -inf
                    m_run = m_blk;
                }
                const float alpha = am * vfix;
                l_run *= alpha;
                // p' = 2^(a rowmul - m - ev), l += p', P' = p' * v_scale (<= 256)
                const float nm = (m_run == -INFINITY ? 0.f : -m_run) - (float)ev;
                float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {              // 32 keys = 16 columns of P' at a time
                    uint32_t pk[16];
#pragma unroll
                    for (int cc = 0; cc < 32; cc += 4) {
                        const int c = 32 * h + cc;
                        const float4 v4 = lds4(col + 2 * kTok + c);
                        float e0, e1, e2, e3;
                        fma2(e0, e1, sv[c], sv[c + 1], rowmul, rowmul, nm, nm);
                        fma2(e2, e3, sv[c + 2], sv[c + 3], rowmul, rowmul, nm, nm);
                        e0 = pa::ex2(e0);
                        e1 = pa::ex2(e1);
                        e2 = pa::ex2(e2);
                        e3 = pa::ex2(e3);
                        add2(ls0, ls1, ls0, ls1, e0, e1);
                        add2(ls0, ls1, ls0, ls1, e2, e3);
                        mul2(e0, e1, e0, e1, v4.x, v4.y);
                        mul2(e2, e3, e2, e3, v4.z, v4.w);
                        const __half2 h01 = __floats2half2_rn(e0, e1), h23 = __floats2half2_rn(e2, e3);
                        pk[cc >> 1] = *reinterpret_cast<const uint32_t*>(&h01);
                        pk[(cc >> 1) + 1] = *reinterpret_cast<const uint32_t*>(&h23);
                    }
                    pa::tc::st_16cols_nowait(s_tm + 16 * h, pk);
                }
                pa::tc::wait_st();
                l_run += ls0 + ls1;
                // O_j may be rescaled once PV(t - 1) is done (same piece only;
                // PV(t) waits for this warp's P)
                if (!w.first() && __any_sync(0xffffffffu, alpha != 1.f)) {
                    const bool ok2 = __all_sync(0xffffffffu,
                                                pa::mbar_wait(bar(kBSpFree + ((t - 1) % kNB)),
                                                              ((t - 1) / kNB) & 1, p.err,
                                                              pa::ERR_WAIT_FULL));
                    if (!ok2 || *abort_flag) {
                        if (lane == 0) *abort_flag = 1;
                        aborted = true;
                        break;
                    }
                    pa::tc::fence_after_sync();
                    const uint32_t o_tm = trow + 128 * (j & 1);
#pragma unroll 1
                    for (int q = 0; q < D / 16; ++q) {
                        uint32_t ov[16];
                        pa::tc::ld_16cols(o_tm + 16 * q, ov);
#pragma unroll
                        for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        pa::tc::st_16cols(o_tm + 16 * q, ov);
                    }
                }
            }
            pa::tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(bar(kBPFull + b));
            if (!w.last()) continue;

            // ---- end of a segment piece: O of rows this thread owns ----
            if (active) {
                const bool ok3 = __all_sync(0xffffffffu, pa::mbar_wait(bar(kBSpFree + b), (t / kNB) & 1,
                                                                       p.err, pa::ERR_WAIT_FULL));
                if (!ok3 || *abort_flag) {
                    if (lane == 0) *abort_flag = 1;
                    aborted = true;
                    break;
                }
                pa::tc::fence_after_sync();
                const bool complete = w.seg_b0 == 0 && w.piece_end == w.cur.nbs;
                Slot sl(p.slots + (2 * wid + (j == 0 ? 0 : 1)) * (int64_t)p.slot_bytes, kRows);
                if (!complete && row == 0) {
                    sl.hdr[0] = w.cur.s;
                    sl.hdr[1] = w.cur.g;
                    sl.hdr[2] = w.cur.c;
                    sl.hdr[3] = w.seg_b0 * kBS;
                    sl.hdr[4] = min(w.piece_end * kBS, L);
                }
                // O and l are in units of the V-scale reference 2^ev: it cancels
                // in O / l; a partial keeps true-scale l and O
                const float to_true = exp2i(ev);
                const float mul = complete ? 1.f / l_run : to_true;
                int64_t obase = 0;
                if (row < rows) {
                    if (complete) {
                        const int gr = w.cur.c * kRows + row;
                        obase = ((int64_t)(q0 + gr / G) * p.num_heads + w.cur.g * G + gr % G) * D;
                    } else {
                        sl.m[row] = m_run;
                        sl.l[row] = l_run * to_true;
                    }
                }
                const uint32_t o_tm = trow + 128 * (j & 1);
#pragma unroll 1
                for (int q = 0; q < D / 16; ++q) {
                    uint32_t ou[16];
                    pa::tc::ld_16cols(o_tm + 16 * q, ou);
                    const float* ov = reinterpret_cast<const float*>(ou);
                    if (row >= rows) continue;
                    if (!complete) {
                        float* dst = sl.o + (int64_t)row * D + 16 * q;
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(dst + i) =
                                make_float4(ov[i] * mul, ov[i + 1] * mul, ov[i + 2] * mul, ov[i + 3] * mul);
                    } else if (p.out_f32) {
                        float* dst = static_cast<float*>(p.out) + obase + 16 * q;
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(dst + i) =
                                make_float4(ov[i] * mul, ov[i + 1] * mul, ov[i + 2] * mul, ov[i + 3] * mul);
                    } else {
                        TQ* dst = static_cast<TQ*>(p.out) + obase + 16 * q;
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            if constexpr (std::is_same<TQ, __half>::value)
                                *reinterpret_cast<__half2*>(dst + i) = __floats2half2_rn(ov[i] * mul, ov[i + 1] * mul);
                            else
                                *reinterpret_cast<__nv_bfloat162*>(dst + i) =
                                    __floats2bfloat162_rn(ov[i] * mul, ov[i + 1] * mul);
                        }
                    }
                }
            }
            pa::tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(bar(kBOFree + (j & 1)));
            if (w.left == w.nb && row == 0)                // the share's last piece
                record_last_segment(p, wid, f1, B, w.piece_end == w.cur.nbs, w.seg_b0,
                                    w.cur.nbs - w.piece_end, j == 0, q0, rows);
        }
        (void)aborted;
    }
    pa::tc::fence_before_sync();
    __syncthreads();
    pa::tc::fence_after_sync();
    if (warp == kMmaWarp) pa::tc::tmem_dealloc(tmem, kTmemCols);
}

template <typename TQ>
pa_status launch_tc(const pa::DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                    pa::sched::Params prm, const TcExtra& x, int64_t workers, int max_chunks) {
    auto kern = paged_decode_int8_tc_kernel<TQ>;
    static bool attr_set = false;   // per instantiation; benign race (idempotent)
    if (!attr_set) {
        if (pa_status s = pa::cuda_status(
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem_bytes(kMaxSeqs)),
                "int8 tensor-core decode: set shared memory size"))
            return s;
        attr_set = true;
    }
    prm.workers = (int)workers;
    if (pa_status s = pa::cuda_status(
            pa::launch_pdl(kern, dim3((unsigned)workers), dim3(kThreads), smem_bytes(a.num_seqs),
                           a.stream, mk, mv, prm, x),
            "int8 tensor-core decode launch"))
        return s;
    const int row_slots = (int)std::min<int64_t>(kRows, (int64_t)(a.num_heads / a.num_kv_heads) * a.max_q_len);
    return pa::cuda_status(pa::sched::launch_segment_reduce<TQ, D>(prm, max_chunks, row_slots, a.stream),
                           "segment reduce launch");
}

}  // namespace

namespace pa {

// INT8 cache, head_dim 128, at least 32 query rows per KV head (MQA decode,
// verify runs), at most kMaxSeqs sequences, and PA_INT8_TC set: the
// tensor-core kernel, one CTA (one share) per SM. Opt-in: on the mixed MQA
// step it is still slower than the mma.sync kernel (its single softmax warp
// per 32-row piece and the per-tile hand-offs between six warp roles bound
// it), so the mma.sync kernel stays the default.
bool int8_tc_applies(const DecodeArgs& a) {
    const int64_t rows = (int64_t)(a.num_heads / a.num_kv_heads) * a.max_q_len;
    return a.kv_dtype == PA_INT8 && a.head_dim == 128 && a.partition_size == 0 && rows >= 32 &&
           a.num_seqs <= kMaxSeqs && !a.ctx_start && !a.lse_out && !a.unmasked &&
           std::getenv("PA_INT8_TC") != nullptr;
}

pa_status launch_decode_int8_tc(const DecodeArgs& a) {
    if (pa_status s = balanced_check(a)) return s;
    const BalancedShape ws = balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads, a.head_dim,
                                            a.max_q_len, a.max_context_len, kTileInt8);
    int dev = 0, sms = 0;
    if (pa_status s = cuda_status(cudaGetDevice(&dev), "cudaGetDevice")) return s;
    if (pa_status s = cuda_status(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                                  "SM count"))
        return s;
    const int G = a.num_heads / a.num_kv_heads;
    const int64_t max_chunks = ((int64_t)G * a.max_q_len + kRows - 1) / kRows;
    // virtual blocks: every (sequence, kv head, 128-row chunk) over its blocks
    const int64_t vblocks = (int64_t)a.num_seqs * a.num_kv_heads * max_chunks *
                            ((a.max_context_len + kBS - 1) / kBS);
    const int64_t workers = std::max<int64_t>(1, std::min<int64_t>(sms, vblocks));
    const int64_t slot = pa::sched::slot_bytes(kRows, D);
    // the partial slots of 128-row pieces, in the workspace the caller sized
    // for the balanced schedule
    if (ws.cum_bytes + 2 * workers * slot > ws.workspace_bytes)
        return fail(PA_ERR_UNSUPPORTED, "int8 tensor-core decode: workspace too small for its slots");
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
    b.slots = static_cast<uint8_t*>(a.slots) + ws.cum_bytes;
    b.err = device_error_word();
    b.max_blocks = a.max_blocks_per_seq;
    b.num_heads = a.num_heads;
    b.num_kv_heads = a.num_kv_heads;
    b.group = G;
    b.num_seqs = a.num_seqs;
    b.num_blocks = a.num_blocks;
    b.rows_per_tile = kRows;
    b.slot_bytes = (int)slot;
    b.scale_log2 = a.scale * kLog2e;
    b.out_f32 = a.out_dtype == PA_F32;
    const TcExtra x{a.k_scale, a.v_scale, a.k_zp, a.v_zp};
    if (a.q_dtype == PA_BF16) return launch_tc<__nv_bfloat16>(a, mk, mv, b, x, workers, (int)max_chunks);
    return launch_tc<__half>(a, mk, mv, b, x, workers, (int)max_chunks);
}

}  // namespace pa
