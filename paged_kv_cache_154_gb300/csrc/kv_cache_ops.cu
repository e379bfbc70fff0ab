// KV-cache writes: append through a slot mapping (F16/BF16 copy, INT8 or
// FP8 quantisation) and copy-on-write block copies.
//
// Append restates the decode workflow of "cs336 lecture 10" (KV Cache:
// append the new K, V to the cache) and the block table of "KV Cache ...
// PagedAttention" §七 (slot = physical block * 16 + offset). The INT8 path
// restates the same lecture's Quantization formula x_q = round(x/scale) +
// zero_point with one (scale, zero point) per (token, kv head) row, as
// "LLM推理优化深度实战" §5.2 asks (per head, not global). Block copies restate
// §2.1 of that page (copy a shared block only when it is modified).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pa_internal.h"

namespace {

constexpr int kBlock = 16;

// One thread per 16-byte vector of a (token, kv head) row, K and V together.
__global__ void append_kv16_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                   uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                   const int64_t* __restrict__ slots, int num_tokens,
                                   int num_kv_heads, int vec_per_row, int64_t num_slots,
                                   unsigned int* err) {
    const int64_t per_token = (int64_t)num_kv_heads * vec_per_row;
    const int64_t total = (int64_t)num_tokens * per_token;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_token;
        const int64_t rem = i - t * per_token;
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (err) atomicOr(err, pa::ERR_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot / kBlock, off = slot % kBlock;
        const int64_t g = rem / vec_per_row, v = rem - g * vec_per_row;
        const int64_t dst = ((blk * num_kv_heads + g) * kBlock + off) * vec_per_row + v;
        k_cache[dst] = __ldg(key + i);
        v_cache[dst] = __ldg(value + i);
    }
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

// One warp per (token, kv head, K-or-V) row. EPL elements per lane
// (head_dim = 32 * EPL). Arithmetic is IEEE fp32: correctly rounded
// division (__fdiv_rn), round-half-to-even (rintf), no contraction.
template <typename T, int EPL>
__global__ void append_kv_int8_kernel(const T* __restrict__ key, const T* __restrict__ value,
                                      int8_t* __restrict__ k_cache, int8_t* __restrict__ v_cache,
                                      float* __restrict__ k_scale, float* __restrict__ v_scale,
                                      int8_t* __restrict__ k_zp, int8_t* __restrict__ v_zp,
                                      const int64_t* __restrict__ slots, int num_tokens,
                                      int num_kv_heads, int64_t num_slots, unsigned int* err) {
    constexpr int D = 32 * EPL;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t rows = (int64_t)num_tokens * num_kv_heads * 2;
    if (warp >= rows) return;
    const int which = (int)(warp & 1);          // 0 = K, 1 = V
    const int64_t tg = warp >> 1;               // token * num_kv_heads + g
    const int64_t t = tg / num_kv_heads;
    const int64_t g = tg - t * num_kv_heads;
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (lane == 0 && err) atomicOr(err, pa::ERR_BAD_SLOT);
        return;
    }
    const T* src = (which ? value : key) + tg * D + lane * EPL;
    float x[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) x[e] = to_f32<T>(src[e]);
    // range widened to contain 0, as the oracle does
    float mn = 0.0f, mx = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        mn = x[e] < mn ? x[e] : mn;
        mx = x[e] > mx ? x[e] : mx;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float a = __shfl_xor_sync(0xffffffffu, mn, o);
        const float b = __shfl_xor_sync(0xffffffffu, mx, o);
        mn = a < mn ? a : mn;
        mx = b > mx ? b : mx;
    }
    float scale = __fdiv_rn(__fsub_rn(mx, mn), 255.0f);
    if (scale == 0.0f) scale = 1.0f;
    const float zf = __fsub_rn(-128.0f, rintf(__fdiv_rn(mn, scale)));
    int zp = (int)zf;
    zp = zp < -128 ? -128 : (zp > 127 ? 127 : zp);
    const int64_t blk = slot / kBlock, off = slot % kBlock;
    const int64_t row = (blk * num_kv_heads + g) * kBlock + off;
    uint32_t packed[(EPL + 3) / 4] = {};
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        int c = (int)rintf(__fdiv_rn(x[e], scale)) + zp;
        c = c < -128 ? -128 : (c > 127 ? 127 : c);
        packed[e / 4] |= (uint32_t)(uint8_t)(int8_t)c << (8 * (e % 4));
    }
    int8_t* dst = (which ? v_cache : k_cache) + row * D + lane * EPL;
    if constexpr (EPL == 4) {
        *reinterpret_cast<uint32_t*>(dst) = packed[0];
    } else {
        static_assert(EPL == 2, "head_dim 64 or 128");
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed[0];
    }
    if (lane == 0) {
        (which ? v_scale : k_scale)[row] = scale;
        (which ? v_zp : k_zp)[row] = (int8_t)zp;
    }
}

// FP8 E4M3 append ("LLM推理优化深度实战" §5.2: FP8 KV cache, one scale per
// KV head): one thread per 16 consecutive elements of a (token, kv head) row,
// K and V together. code = E4M3(x / scale[head]): the IEEE fp32 quotient
// (__fdiv_rn), converted with round-to-nearest-even and saturation at +-448.
template <typename T>
__global__ void append_kv_fp8_kernel(const T* __restrict__ key, const T* __restrict__ value,
                                     uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                                     const float* __restrict__ k_scale,
                                     const float* __restrict__ v_scale,
                                     const int64_t* __restrict__ slots, int num_tokens,
                                     int num_kv_heads, int head_dim, int64_t num_slots,
                                     unsigned int* err) {
    const int per_row = head_dim / 16;
    const int64_t per_token = (int64_t)num_kv_heads * per_row;
    const int64_t total = (int64_t)num_tokens * per_token;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_token;
        const int64_t rem = i - t * per_token;
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (err) atomicOr(err, pa::ERR_BAD_SLOT);
            continue;
        }
        const int g = (int)(rem / per_row), c = (int)(rem - (int64_t)g * per_row);
        const int64_t blk = slot / kBlock, off = slot % kBlock;
        const int64_t src = (t * num_kv_heads + g) * head_dim + c * 16;
        const int64_t dst = ((blk * num_kv_heads + g) * kBlock + off) * head_dim + c * 16;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const T* in = (which ? value : key) + src;
            const float s = __ldg((which ? v_scale : k_scale) + g);
            const uint4 raw0 = __ldg(reinterpret_cast<const uint4*>(in));
            const uint4 raw1 = __ldg(reinterpret_cast<const uint4*>(in) + 1);
            const T* h0 = reinterpret_cast<const T*>(&raw0);
            const T* h1 = reinterpret_cast<const T*>(&raw1);
            uint32_t out[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                uint32_t word = 0;
#pragma unroll
                for (int pr = 0; pr < 2; ++pr) {
                    const int e = 4 * w + 2 * pr;
                    const T* h = e < 8 ? h0 + e : h1 + (e - 8);
                    const float2 y = make_float2(__fdiv_rn(to_f32<T>(h[0]), s),
                                                 __fdiv_rn(to_f32<T>(h[1]), s));
                    const __nv_fp8x2_storage_t q =
                        __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
                    word |= (uint32_t)q << (16 * pr);
                }
                out[w] = word;
            }
            *reinterpret_cast<uint4*>((which ? v_cache : k_cache) + dst) =
                make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
}

struct CopyParams {
    uint4* arrays[6];
    int64_t vecs_per_block[6];
};

// grid = (n_pairs, 6): one CTA copies one block of one array.
__global__ void copy_blocks_kernel(CopyParams p, const int32_t* __restrict__ pairs, int n_pairs,
                                   int64_t num_blocks, unsigned int* err) {
    const int pair = blockIdx.x, arr = blockIdx.y;
    uint4* base = p.arrays[arr];
    if (!base) return;
    const int64_t src = __ldg(pairs + 2 * pair), dst = __ldg(pairs + 2 * pair + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && err) atomicOr(err, pa::ERR_BAD_BLOCK);
        return;
    }
    const int64_t n = p.vecs_per_block[arr];
    const uint4* s = base + src * n;
    uint4* d = base + dst * n;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
}

}  // namespace

namespace pa {

pa_status launch_append_kv(const AppendArgs& a) {
    unsigned int* err = device_error_word();
    const int64_t num_slots = (int64_t)a.num_blocks * a.block_size;
    if (a.kv_dtype == PA_FP8_E4M3) {
        const int64_t total = (int64_t)a.num_tokens * a.num_kv_heads * (a.head_dim / 16);
        const int threads = 256;
        const int64_t blocks = (total + threads - 1) / threads;
        const int grid = (int)(blocks < 65535 ? blocks : 65535);
        if (((uintptr_t)a.k_scale | (uintptr_t)a.v_scale) % 4)
            return fail(PA_ERR_INVALID_ARG, "k_scale / v_scale must be 4-byte aligned");
        if (a.src_dtype == PA_BF16)
            append_kv_fp8_kernel<__nv_bfloat16><<<grid, threads, 0, a.stream>>>(
                static_cast<const __nv_bfloat16*>(a.key),
                static_cast<const __nv_bfloat16*>(a.value), static_cast<uint8_t*>(a.k_cache),
                static_cast<uint8_t*>(a.v_cache), a.k_scale, a.v_scale, a.slots, a.num_tokens,
                a.num_kv_heads, a.head_dim, num_slots, err);
        else
            append_kv_fp8_kernel<__half><<<grid, threads, 0, a.stream>>>(
                static_cast<const __half*>(a.key), static_cast<const __half*>(a.value),
                static_cast<uint8_t*>(a.k_cache), static_cast<uint8_t*>(a.v_cache), a.k_scale,
                a.v_scale, a.slots, a.num_tokens, a.num_kv_heads, a.head_dim, num_slots, err);
    } else if (a.kv_dtype != PA_INT8) {
        const int vec_per_row = a.head_dim * 2 / 16;
        const int64_t total = (int64_t)a.num_tokens * a.num_kv_heads * vec_per_row;
        const int threads = 256;
        const int64_t blocks = (total + threads - 1) / threads;
        const int grid = (int)(blocks < 65535 ? blocks : 65535);
        append_kv16_kernel<<<grid, threads, 0, a.stream>>>(
            static_cast<const uint4*>(a.key), static_cast<const uint4*>(a.value),
            static_cast<uint4*>(a.k_cache), static_cast<uint4*>(a.v_cache), a.slots,
            a.num_tokens, a.num_kv_heads, vec_per_row, num_slots, err);
    } else {
        const int64_t rows = (int64_t)a.num_tokens * a.num_kv_heads * 2;
        const int threads = 256;
        const int64_t grid = (rows * 32 + threads - 1) / threads;
        if (grid > 0x7fffffff) return fail(PA_ERR_UNSUPPORTED, "too many tokens for one launch");
#define PA_LAUNCH_Q8(T, EPL)                                                                   \
    append_kv_int8_kernel<T, EPL><<<(unsigned)grid, threads, 0, a.stream>>>(                   \
        static_cast<const T*>(a.key), static_cast<const T*>(a.value),                          \
        static_cast<int8_t*>(a.k_cache), static_cast<int8_t*>(a.v_cache), a.k_scale,           \
        a.v_scale, a.k_zp, a.v_zp, a.slots, a.num_tokens, a.num_kv_heads, num_slots, err)
        if (a.src_dtype == PA_BF16) {
            if (a.head_dim == 128) PA_LAUNCH_Q8(__nv_bfloat16, 4);
            else PA_LAUNCH_Q8(__nv_bfloat16, 2);
        } else {
            if (a.head_dim == 128) PA_LAUNCH_Q8(__half, 4);
            else PA_LAUNCH_Q8(__half, 2);
        }
#undef PA_LAUNCH_Q8
    }
    return cuda_status(cudaGetLastError(), "append_kv launch");
}

pa_status launch_copy_blocks(const CopyArgs& a) {
    CopyParams p{};
    for (int i = 0; i < 6; ++i) {
        p.arrays[i] = static_cast<uint4*>(a.arrays[i]);
        p.vecs_per_block[i] = a.bytes_per_block[i] / 16;
    }
    dim3 grid(a.n_pairs, 6);
    copy_blocks_kernel<<<grid, 256, 0, a.stream>>>(p, a.pairs, a.n_pairs, a.num_blocks,
                                                   device_error_word());
    return cuda_status(cudaGetLastError(), "copy_blocks launch");
}

}  // namespace pa
