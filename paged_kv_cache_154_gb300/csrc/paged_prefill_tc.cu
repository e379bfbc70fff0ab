// Paged prefill attention on the 5th-generation tensor cores (tcgen05, TMEM).
//
// A long query run (a prefill chunk, "大模型推理优化全攻略" / "LLM推理优化深度实战":
// chunked prefill) turns attention over the paged cache into a dense
// contraction: per KV head, G q heads x r query tokens against the
// sequence's keys, causally masked ("cs336 lecture 10": query i of a run of
// r at position L - r + i sees keys 0 .. L - r + i). This kernel computes it
// per 128-row tile (the rows of one (sequence, kv head) in chunks of 128) over
// key tiles of 64 tokens (four 16-token blocks, gathered through the block
// table by TMA):
//
//   S = Q K^T          tcgen05.mma M128 N64, A = Q, B = K (both K-major in
//                      shared memory, 128-byte swizzle), S in TMEM (two
//                      buffers, so the product of tile t + 1 runs while the
//                      softmax works on tile t);
//   P = softmax(S)     four warps, one thread per row: S read from TMEM, fp32
//                      online softmax with a running max moved only when a
//                      tile raises it by more than 2^8 (O is then rescaled in
//                      TMEM), P written as two 16-bit parts P_hi + P_lo so the
//                      weights keep ~16 mantissa bits (two P buffers);
//   O += P V           tcgen05.mma M128 N128, A = P (K-major), B = V
//                      (MN-major: V's rows are tokens, the contraction index),
//                      O in TMEM for the whole key range;
//   out = O / l        read from TMEM at the end.
//
// Roles: warp 0 streams K/V blocks into a 4-stage ring (TMA), lane 0 of warp 1
// issues the MMAs and commits them to mbarriers, warps 2-5 do the softmax and
// the epilogue. Every wait is bounded; a wait that gives up stops the tile
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
constexpr int kRows = 128;              // query rows per tile (MMA M)
constexpr int kTok = 64;                // keys per tile (S columns)
constexpr int kTileBlocks = kTok / kBS; // 4
constexpr int kThreads = 192;           // 6 warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyMax = 8.f;

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kStages = 4;                      // K/V ring
constexpr int kQOff = 0;                        // [2 sub][128 rows][128 B]
constexpr int kKVOff = 32 * 1024;               // kStages x (K 16 KB, V 16 KB)
constexpr int kKVStage = 32 * 1024;
constexpr int kKBytes = 16 * 1024;              // [2 sub][64 rows][128 B]
constexpr int kSubKV = 8 * 1024;                // one 64-dim half of a K (or V) tile
constexpr int kPOff = kKVOff + kStages * kKVStage;   // 2 buffers x (P_hi, P_lo) [128 rows][128 B]
constexpr int kPBytes = 16 * 1024;
constexpr int kPBuf = 2 * kPBytes;
constexpr int kBarOff = kPOff + 2 * kPBuf;      // mbarriers and flags
constexpr int kSmem = kBarOff + 256 + 1024;     // + alignment slack
// barrier slots: K/V full and empty per stage; S full, P full, O done per buffer
constexpr int kBarKVFull = 0, kBarKVEmpty = kStages, kBarSFull = 2 * kStages,
              kBarPFull = 2 * kStages + 2, kBarODone = 2 * kStages + 4, kBarFin = 2 * kStages + 6;
constexpr int kNumBars = 2 * kStages + 7;
// TMEM columns: S in two buffers of 64, O in 128
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kOCol = 128;

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
    int max_chunks;
    float scale_log2;
    int out_f32;
};

// byte offset of 16-byte chunk c (0..7) of row `row` inside a 128-byte-wide,
// 128-byte-swizzled matrix (8-row atoms of 1024 bytes)
__device__ __forceinline__ uint32_t sw128(int row, int c) {
    return row * 128 + ((c ^ (row & 7)) << 4);
}

template <typename T>
struct Cvt;
template <>
struct Cvt<__nv_bfloat16> {
    static constexpr bool kBF16 = true;
    __device__ static uint32_t pack(float a, float b, float& ra, float& rb) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        ra = a - __low2float(v);
        rb = b - __high2float(v);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ static uint32_t pack(float a, float b) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ static void store2(void* p, float a, float b) {
        *static_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
    }
};
template <>
struct Cvt<__half> {
    static constexpr bool kBF16 = false;
    __device__ static uint32_t pack(float a, float b, float& ra, float& rb) {
        __half2 v = __floats2half2_rn(a, b);
        ra = a - __low2float(v);
        rb = b - __high2float(v);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ static uint32_t pack(float a, float b) {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ static void store2(void* p, float a, float b) {
        *static_cast<__half2*>(p) = __floats2half2_rn(a, b);
    }
};

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
    using C = Cvt<T>;
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

    // task: (chunk, sequence, kv head), later chunks (longer key ranges) first
    const int sh = p.num_seqs * p.num_kv_heads;
    const int c = p.max_chunks - 1 - (int)(blockIdx.x / sh);
    const int s = (int)(blockIdx.x % sh) / p.num_kv_heads;
    const int g = (int)(blockIdx.x % sh) % p.num_kv_heads;
    const int L = __ldg(p.context_lens + s);
    int q0, r;
    if (p.qsl) {
        q0 = __ldg(p.qsl + s);
        r = __ldg(p.qsl + s + 1) - q0;
    } else {
        q0 = s;
        r = 1;
    }
    const int G = p.group;
    const int row_off = c * kRows;
    const int rows = min(kRows, G * r - row_off);
    if (rows <= 0) return;                                       // uniform over the CTA
    const int jmax = min(r - 1, (row_off + rows - 1) / G);
    const int end_blocks = min((L + kBS - 1) / kBS, (L - r + jmax) / kBS + 1);
    const int tiles = (end_blocks + kTileBlocks - 1) / kTileBlocks;

    if (threadIdx.x == 0) {
        // P-ready takes one arrival from each of the four softmax warps
        for (int i = 0; i < kNumBars; ++i)
            pa::mbar_init(bars + 8 * i, (i == kBarPFull || i == kBarPFull + 1) ? 4 : 1);
        *abort_flag = 0;
        pa::fence_barrier_init();
        pa::prefetch_tensormap(&tmap_k);
        pa::prefetch_tensormap(&tmap_v);
    }
    if (warp == 1) {
        pa::tc::tmem_alloc(pa::smem_addr(tmem_holder), kTmemCols);
        pa::tc::tmem_relinquish();
    }
    // Q tile: 128 rows x 128 dims, 128-byte swizzled K-major (two 64-dim halves)
    for (int e = threadIdx.x; e < kRows * 16; e += kThreads) {
        const int row = e >> 4, ch = e & 15;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < rows) {
            const int gr = row_off + row;
            const T* src = static_cast<const T*>(p.q) +
                           ((int64_t)(q0 + gr / G) * p.num_heads + g * G + gr % G) * D;
            v = __ldg(reinterpret_cast<const uint4*>(src) + ch);
        }
        const uint32_t dst = base + kQOff + (ch >> 3) * (kRows * 128) + sw128(row, ch & 7);
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
        int issued = 0;
        for (int t = 0; t < tiles; ++t) {
            const int st = t % kStages;
            if (t >= kStages) {   // the stage is free once the P V product of tile t - kStages is done
                const bool ok = __all_sync(
                    0xffffffffu,
                    pa::mbar_wait(bars + 8 * (kBarKVEmpty + st), ((t / kStages) - 1) & 1, p.err,
                                  pa::ERR_WAIT_EMPTY));
                if (!ok || *abort_flag) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
            }
            const int nblk = min(kTileBlocks, end_blocks - t * kTileBlocks);
            int row = 0;
            if (lane < nblk) {
                int blk = __ldg(p.block_tables + (int64_t)s * p.max_blocks + t * kTileBlocks + lane);
                if (blk < 0 || blk >= p.num_blocks) {
                    if (p.err) atomicOr(p.err, pa::ERR_BAD_BLOCK);
                    blk = 0;
                }
                row = (blk * p.num_kv_heads + g) * kBS;
            }
            const uint32_t bar = bars + 8 * (kBarKVFull + st);
            if (lane == 0) pa::mbar_arrive_expect_tx(bar, nblk * 4 * (kBS * 128));
            const uint32_t kst = base + kKVOff + st * kKVStage;
            for (int j = 0; j < nblk; ++j) {
                const int rj = __shfl_sync(0xffffffffu, row, j);
                if (lane == 0) {
#pragma unroll
                    for (int sub = 0; sub < 2; ++sub) {
                        pa::tma_load_2d(kst + sub * kSubKV + j * (kBS * 128), &tmap_k, sub * 64, rj,
                                        bar);
                        pa::tma_load_2d(kst + kKBytes + sub * kSubKV + j * (kBS * 128), &tmap_v,
                                        sub * 64, rj, bar);
                    }
                }
            }
            issued = t + 1;
        }
        // drain: no copy may be in flight when the CTA ends; the last kStages
        // issued tiles are waited once more (each completes whether or not it
        // was consumed; earlier ones were consumed before their stage was reused)
        if (lane == 0)
            for (int t = issued > kStages ? issued - kStages : 0; t < issued; ++t)
                if (!pa::mbar_wait(bars + 8 * (kBarKVFull + t % kStages), (t / kStages) & 1,
                                   nullptr, 0)) {
                    if (p.err) atomicOr(p.err, pa::ERR_WAIT_DRAIN);
                    break;
                }
    } else if (warp == 1) {
        // ---------------- MMA issue (one thread) ----------------
        // order on the tensor pipe: QK(0), then per tile t: QK(t + 1), PV(t)
        if (lane == 0) {
            constexpr uint32_t idesc_qk = pa::tc::idesc_f16(C::kBF16, false, false, kRows, kTok);
            constexpr uint32_t idesc_pv = pa::tc::idesc_f16(C::kBF16, false, true, kRows, D);
            auto issue_qk = [&](int t) -> bool {   // S[t & 1] = Q K(t)^T
                const int st = t % kStages;
                bool ok = pa::mbar_wait(bars + 8 * (kBarKVFull + st), (t / kStages) & 1, p.err,
                                        pa::ERR_WAIT_FULL);
                if (ok && t >= 2)   // S[t & 1] is free once the softmax of tile t - 2 is done
                    ok = pa::mbar_wait(bars + 8 * (kBarPFull + (t & 1)), ((t >> 1) - 1) & 1, p.err,
                                       pa::ERR_WAIT_FULL);
                if (!ok || *abort_flag) return false;
                pa::tc::fence_after_sync();
                const uint32_t kst = base + kKVOff + st * kKVStage;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = pa::tc::smem_desc_sw128(
                        base + kQOff + (kk >> 2) * (kRows * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = pa::tc::smem_desc_sw128(
                        kst + (kk >> 2) * kSubKV + (kk & 3) * 32, 16, 1024);
                    pa::tc::mma_f16_ss(tmem + 64 * (t & 1), a, b, idesc_qk, kk > 0 ? 1u : 0u);
                }
                pa::tc::commit(bars + 8 * (kBarSFull + (t & 1)));
                return true;
            };
            bool ok = issue_qk(0);
            for (int t = 0; ok && t < tiles; ++t) {
                if (t + 1 < tiles && !issue_qk(t + 1)) {
                    ok = false;
                    break;
                }
                ok = pa::mbar_wait(bars + 8 * (kBarPFull + (t & 1)), (t >> 1) & 1, p.err,
                                   pa::ERR_WAIT_FULL);
                if (!ok || *abort_flag) {
                    ok = false;
                    break;
                }
                pa::tc::fence_after_sync();
                const int st = t % kStages;
                const uint32_t kst = base + kKVOff + st * kKVStage;
                const uint32_t pbuf = base + kPOff + (t & 1) * kPBuf;
                const int nblk = min(kTileBlocks, end_blocks - t * kTileBlocks);
                for (int kb = 0; kb < nblk; ++kb) {
                    const uint64_t bv = pa::tc::smem_desc_sw128(
                        kst + kKBytes + kb * (kBS * 128), kSubKV, 1024);
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        const uint64_t a =
                            pa::tc::smem_desc_sw128(pbuf + part * kPBytes + kb * 32, 16, 1024);
                        pa::tc::mma_f16_ss(tmem + kOCol, a, bv, idesc_pv,
                                           (t > 0 || kb > 0 || part > 0) ? 1u : 0u);
                    }
                }
                pa::tc::commit(bars + 8 * (kBarODone + (t & 1)));
                pa::tc::commit(bars + 8 * (kBarKVEmpty + st));
            }
            if (!ok) *abort_flag = 1;
            // every MMA this thread issued has finished before TMEM is freed
            pa::tc::commit(bars + 8 * kBarFin);
            if (!pa::mbar_wait(bars + 8 * kBarFin, 0, nullptr, 0) && p.err)
                atomicOr(p.err, pa::ERR_WAIT_DRAIN);
        }
        __syncwarp();
    } else {
        // ---------------- softmax and epilogue: one thread per row ----------------
        const int lane_base = 32 * (warp & 3);
        const int row = lane_base + lane;                    // tile row = TMEM lane
        const int gr = row_off + row;
        const bool valid = row < rows;
        const int jq = valid ? gr / G : 0;
        const int bound = valid ? min(L - r + jq, L - 1) : -1;
        const uint32_t trow = tmem + ((uint32_t)lane_base << 16);
        float m_run = -INFINITY, l_run = 0.f;
        const int sm_tid = threadIdx.x - 64;                 // 0..127
        int done = 0;
        for (int t = 0; t < tiles; ++t) {
            const bool ok = __all_sync(
                0xffffffffu, pa::mbar_wait(bars + 8 * (kBarSFull + (t & 1)), (t >> 1) & 1, p.err,
                                           pa::ERR_WAIT_FULL));
            if (!ok || *abort_flag) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            pa::tc::fence_after_sync();
            float sv[kTok];
            const uint32_t scol = 64 * (t & 1);
            pa::tc::ld_32cols(trow + scol, *reinterpret_cast<float(*)[32]>(sv));
            pa::tc::ld_32cols(trow + scol + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
            const int tok0 = t * kTok;
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < kTok; ++j) {
                float v = sv[j] * p.scale_log2;
                if (tok0 + j > bound) v = -INFINITY;
                sv[j] = v;
                mx = fmaxf(mx, v);
            }
            float alpha = 1.f;
            bool moved = false;
            if (mx > m_run + kLazyMax) {
                alpha = pa::ex2(m_run - mx);                   // 0 while m_run is -inf
                m_run = mx;
                moved = true;
            }
            const float m_use = m_run == -INFINITY ? 0.f : m_run;
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < kTok; ++j) {
                sv[j] = pa::ex2(sv[j] - m_use);
                sum += sv[j];
            }
            l_run = l_run * alpha + sum;
            // P buffer t & 1 is free once the P V product of tile t - 2 is done
            if (t >= 2) {
                const bool ok2 = __all_sync(
                    0xffffffffu, pa::mbar_wait(bars + 8 * (kBarODone + (t & 1)),
                                               ((t >> 1) - 1) & 1, p.err, pa::ERR_WAIT_FULL));
                if (!ok2 || *abort_flag) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
            }
            // O may be rescaled once the P V product of tile t - 1 is done
            if (t >= 1 && __any_sync(0xffffffffu, moved)) {
                const bool ok3 = __all_sync(
                    0xffffffffu, pa::mbar_wait(bars + 8 * (kBarODone + ((t - 1) & 1)),
                                               ((t - 1) >> 1) & 1, p.err, pa::ERR_WAIT_FULL));
                if (!ok3 || *abort_flag) {
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
                pa::tc::fence_after_sync();
                {
                    // rescale this warp's rows of O in TMEM (alpha = 1 for the others)
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        float ov[32];
                        pa::tc::ld_32cols(trow + kOCol + 32 * q, ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] *= alpha;
                        pa::tc::st_32cols(trow + kOCol + 32 * q, ov);
                    }
                }
            }
            // P_hi and P_lo of this row: 64 keys = 8 chunks of 16 bytes each
#pragma unroll
            for (int ch = 0; ch < kTok / 8; ++ch) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float ra, rb;
                    hi[u] = C::pack(sv[8 * ch + 2 * u], sv[8 * ch + 2 * u + 1], ra, rb);
                    lo[u] = C::pack(ra, rb);
                }
                const uint32_t off = base + kPOff + (t & 1) * kPBuf + sw128(row, ch);
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(off), "r"(hi[0]),
                             "r"(hi[1]), "r"(hi[2]), "r"(hi[3])
                             : "memory");
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(off + kPBytes),
                             "r"(lo[0]), "r"(lo[1]), "r"(lo[2]), "r"(lo[3])
                             : "memory");
            }
            // V rows past the context (in the sequence's last block) may hold
            // anything: zero them so that P = 0 never meets a NaN
            const int nblk = min(kTileBlocks, end_blocks - t * kTileBlocks);
            const int tok_end = tok0 + nblk * kBS;
            if (L < tok_end) {
                const int z0 = L - tok0, zrows = tok_end - L;      // local token rows to zero
                for (int e = sm_tid; e < zrows * 16; e += 128) {
                    const int lr = z0 + e / 16, ch = e % 16;
                    const uint32_t dst = base + kKVOff + (t % kStages) * kKVStage + kKBytes +
                                         (ch >> 3) * kSubKV + lr * 128 + ((ch & 7) << 4);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0u)
                                 : "memory");
                }
            }
            // each warp releases its part (no CTA-wide barrier a stalled warp could hold)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            pa::tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(bars + 8 * (kBarPFull + (t & 1)));
            done = t + 1;
        }
        // epilogue: O / l for this row
        if (done == tiles && tiles > 0) {
            const bool ok = __all_sync(
                0xffffffffu, pa::mbar_wait(bars + 8 * (kBarODone + ((tiles - 1) & 1)),
                                           ((tiles - 1) >> 1) & 1, p.err, pa::ERR_WAIT_FULL));
            if (ok) {
                pa::tc::fence_after_sync();
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                const int64_t orow =
                    valid ? ((int64_t)(q0 + gr / G) * p.num_heads + g * G + gr % G) : 0;
#pragma unroll
                for (int qd = 0; qd < D / 32; ++qd) {
                    float ov[32];
                    pa::tc::ld_32cols(trow + kOCol + 32 * qd, ov);
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
                            for (int i = 0; i < 32; i += 2) C::store2(dst + i, ov[i] * inv, ov[i + 1] * inv);
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

template <typename T>
pa_status launch(const pa::DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                 const PrefillParams& prm, int64_t grid) {
    auto kern = paged_prefill_tc_kernel<T>;
    static bool attr_set = false;   // per instantiation; benign race (idempotent)
    if (!attr_set) {
        if (pa_status s = pa::cuda_status(
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem),
                "prefill: set shared memory size"))
            return s;
        attr_set = true;
    }
    return pa::cuda_status(
        pa::launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), kSmem, a.stream, mk, mv, prm),
        "prefill launch");
}

}  // namespace

namespace pa {

// Long query runs over a 16-bit cache with head_dim 128 (and no token offset
// or log-sum-exp output): at least 256 query rows per KV head.
bool prefill_tc_applies(const DecodeArgs& a) {
    const int64_t rows = (int64_t)(a.num_heads / a.num_kv_heads) * a.max_q_len;
    return (a.kv_dtype == PA_BF16 || a.kv_dtype == PA_F16) && a.head_dim == 128 &&
           a.partition_size == 0 && !a.ctx_start && !a.lse_out && !a.unmasked && rows >= 256 &&
           std::getenv("PA_PREFILL_MMA_SYNC") == nullptr;
}

pa_status launch_prefill_tc(const DecodeArgs& a) {
    const int G = a.num_heads / a.num_kv_heads;
    const int64_t max_chunks = ((int64_t)G * a.max_q_len + kRows - 1) / kRows;
    const int64_t grid = max_chunks * a.num_seqs * a.num_kv_heads;
    if (grid > 0x7fffffff) return fail(PA_ERR_UNSUPPORTED, "prefill grid too large");
    CUtensorMap mk, mv;
    if (pa_status s = cache_tensor_map(&mk, a.k_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 2))
        return s;
    if (pa_status s = cache_tensor_map(&mv, a.v_cache, a.num_blocks, a.num_kv_heads, a.head_dim, 2))
        return s;
    PrefillParams prm{};
    prm.out = a.out;
    prm.q = a.q;
    prm.block_tables = a.block_tables;
    prm.context_lens = a.context_lens;
    prm.qsl = a.query_start_loc;
    prm.err = device_error_word();
    prm.max_blocks = a.max_blocks_per_seq;
    prm.num_heads = a.num_heads;
    prm.num_kv_heads = a.num_kv_heads;
    prm.group = G;
    prm.num_seqs = a.num_seqs;
    prm.num_blocks = a.num_blocks;
    prm.max_chunks = (int)max_chunks;
    prm.scale_log2 = a.scale * kLog2e;
    prm.out_f32 = a.out_dtype == PA_F32;
    if (a.kv_dtype == PA_BF16) return launch<__nv_bfloat16>(a, mk, mv, prm, grid);
    return launch<__half>(a, mk, mv, prm, grid);
}

}  // namespace pa
