// C-ABI entry points for the device operations: argument checks on the host,
// optional range validation of device arrays (PA_VALIDATE=1), the device
// error word, and dispatch to the kernel launchers.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace {

thread_local char g_msg[512] = "";

// One word per device; kernels OR error codes into it instead of trapping.
__device__ unsigned int g_device_error;

}  // namespace

namespace pa {

pa_status fail(pa_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return s;
}

pa_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return PA_OK;
    return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

unsigned int* device_error_word() {
    static std::mutex mu;
    static std::vector<unsigned int*> per_device;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)per_device.size() <= dev) per_device.resize(dev + 1, nullptr);
    if (!per_device[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        per_device[dev] = static_cast<unsigned int*>(p);
    }
    return per_device[dev];
}

bool validate_enabled() {
    const char* v = getenv("PA_VALIDATE");
    return v && v[0] && strcmp(v, "0") != 0;
}

}  // namespace pa

using pa::fail;

namespace {

bool is_kv_dtype(pa_dtype t) {
    return t == PA_F16 || t == PA_BF16 || t == PA_INT8 || t == PA_FP8_E4M3;
}

pa_status check_shape(int32_t num_kv_heads, int32_t head_dim, int32_t block_size) {
    if (block_size != 16)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d (only 16 is supported)", block_size);
    if (head_dim != 64 && head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d (64 or 128 supported)", head_dim);
    if (num_kv_heads <= 0) return fail(PA_ERR_INVALID_ARG, "num_kv_heads %d", num_kv_heads);
    return PA_OK;
}

template <typename T>
pa_status to_host(std::vector<T>& h, const T* d, size_t n, cudaStream_t st) {
    h.resize(n);
    if (n == 0) return PA_OK;
    if (pa_status s = pa::cuda_status(cudaStreamSynchronize(st), "validate: sync")) return s;
    return pa::cuda_status(cudaMemcpy(h.data(), d, n * sizeof(T), cudaMemcpyDeviceToHost),
                           "validate: copy to host");
}

}  // namespace

extern "C" const char* pa_last_error(void) { return g_msg; }
extern "C" const char* pa_version(void) { return "paged-kv-gb300 0.1 (sm_103a)"; }

extern "C" pa_status pa_copy_blocks(void* k_cache, void* v_cache, void* k_scale,
                                    void* v_scale, void* k_zp, void* v_zp,
                                    const int32_t* d_pairs, int32_t n_pairs,
                                    int32_t num_blocks, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t block_size,
                                    pa_dtype kv_dtype, void* stream) {
    if (n_pairs < 0) return fail(PA_ERR_INVALID_ARG, "n_pairs < 0");
    if (n_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !d_pairs) return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (!is_kv_dtype(kv_dtype)) return fail(PA_ERR_INVALID_ARG, "kv_dtype %d", (int)kv_dtype);
    if (pa_status s = check_shape(num_kv_heads, head_dim, block_size)) return s;
    const bool q8 = kv_dtype == PA_INT8;
    if (q8 && (!k_scale || !v_scale || !k_zp || !v_zp))
        return fail(PA_ERR_INVALID_ARG, "INT8 cache needs k_scale, v_scale, k_zp, v_zp");
    cudaStream_t st = (cudaStream_t)stream;
    if (pa::validate_enabled()) {
        std::vector<int32_t> h;
        if (pa_status s = to_host(h, d_pairs, 2 * (size_t)n_pairs, st)) return s;
        std::vector<uint8_t> role(num_blocks, 0);   // 1 = source, 2 = destination
        for (int32_t i = 0; i < 2 * n_pairs; ++i) {
            int32_t b = h[i];
            if (b < 0 || b >= num_blocks)
                return fail(PA_ERR_VALIDATION, "copy pair %d names block %d outside [0,%d)", i / 2,
                            b, num_blocks);
            uint8_t want = (i % 2) ? 2 : 1;
            if (role[b] && (role[b] != want || want == 2))
                return fail(PA_ERR_VALIDATION, "block %d is used twice in the copy list", b);
            role[b] = want;
        }
    }
    const int64_t tile = (int64_t)num_kv_heads * block_size;
    pa::CopyArgs a{};
    a.arrays[0] = k_cache;
    a.arrays[1] = v_cache;
    a.bytes_per_block[0] = a.bytes_per_block[1] = tile * head_dim * pa::dtype_bytes(kv_dtype);
    if (q8) {
        a.arrays[2] = k_scale;
        a.arrays[3] = v_scale;
        a.arrays[4] = k_zp;
        a.arrays[5] = v_zp;
        a.bytes_per_block[2] = a.bytes_per_block[3] = tile * 4;
        a.bytes_per_block[4] = a.bytes_per_block[5] = tile;
    }
    for (int i = 0; i < 6; ++i)
        if (a.arrays[i] && ((uintptr_t)a.arrays[i] % 16 != 0))
            return fail(PA_ERR_INVALID_ARG, "cache array %d is not 16-byte aligned", i);
    a.pairs = d_pairs;
    a.n_pairs = n_pairs;
    a.num_blocks = num_blocks;
    a.stream = st;
    return pa::launch_copy_blocks(a);
}

extern "C" pa_status pa_append_kv(const void* key, const void* value, pa_dtype src_dtype,
                                  void* k_cache, void* v_cache, pa_dtype kv_dtype,
                                  float* k_scale, float* v_scale, int8_t* k_zp,
                                  int8_t* v_zp, const int64_t* slot_mapping,
                                  int32_t num_tokens, int32_t num_blocks,
                                  int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, void* stream) {
    if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (src_dtype != PA_F16 && src_dtype != PA_BF16)
        return fail(PA_ERR_UNSUPPORTED, "src_dtype %d (F16 or BF16)", (int)src_dtype);
    if (!is_kv_dtype(kv_dtype)) return fail(PA_ERR_INVALID_ARG, "kv_dtype %d", (int)kv_dtype);
    if ((kv_dtype == PA_F16 || kv_dtype == PA_BF16) && kv_dtype != src_dtype)
        return fail(PA_ERR_UNSUPPORTED, "a %s cache takes %s rows only",
                    kv_dtype == PA_F16 ? "F16" : "BF16", kv_dtype == PA_F16 ? "F16" : "BF16");
    if (kv_dtype == PA_FP8_E4M3 && (!k_scale || !v_scale))
        return fail(PA_ERR_INVALID_ARG, "FP8 cache needs per-head k_scale and v_scale");
    if (pa_status s = check_shape(num_kv_heads, head_dim, block_size)) return s;
    if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks %d", num_blocks);
    if (kv_dtype == PA_INT8 && (!k_scale || !v_scale || !k_zp || !v_zp))
        return fail(PA_ERR_INVALID_ARG, "INT8 cache needs k_scale, v_scale, k_zp, v_zp");
    if (((uintptr_t)key | (uintptr_t)value | (uintptr_t)k_cache | (uintptr_t)v_cache) % 16)
        return fail(PA_ERR_INVALID_ARG, "key, value and caches must be 16-byte aligned");
    cudaStream_t st = (cudaStream_t)stream;
    if (pa::validate_enabled()) {
        std::vector<int64_t> h;
        if (pa_status s = to_host(h, slot_mapping, (size_t)num_tokens, st)) return s;
        const int64_t lim = (int64_t)num_blocks * block_size;
        for (int32_t i = 0; i < num_tokens; ++i) {
            if (h[i] >= lim)
                return fail(PA_ERR_VALIDATION, "slot %lld of token %d outside the pool (%lld slots)",
                            (long long)h[i], i, (long long)lim);
        }
    }
    pa::AppendArgs a{key, value, src_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                     k_zp, v_zp, slot_mapping, num_tokens, num_blocks, num_kv_heads,
                     head_dim, block_size, st};
    return pa::launch_append_kv(a);
}

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_tokens,
                                           int32_t num_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t max_q_len,
                                           int32_t max_context_len, int32_t partition_size) {
    if (num_seqs <= 0 || num_q_tokens <= 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || max_q_len <= 0 || max_context_len <= 0 || partition_size < 0 ||
        num_heads % num_kv_heads != 0)
        return 0;
    if (partition_size == 0)
        return (size_t)(pa::kArrivalBytes + pa::balanced_shape(num_seqs, num_heads, num_kv_heads,
                                                               head_dim, max_q_len, max_context_len)
                                                .workspace_bytes);
    const int64_t parts = (max_context_len + (int64_t)partition_size - 1) / partition_size;
    if (parts <= 1) return 0;
    const size_t rows = (size_t)num_q_tokens * num_heads * parts;
    return (size_t)pa::kArrivalBytes + align256(rows * head_dim * sizeof(float)) +
           2 * align256(rows * sizeof(float));
}

namespace pa {

// Host-side checks shared by the decode entry points; may rewrite max_q_len
// (1 without query_start_loc).
pa_status check_decode_args(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype,
                            const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
                            const float* k_scale, const float* v_scale, const int8_t* k_zp,
                            const int8_t* v_zp, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* context_lens,
                            const int32_t* query_start_loc, int32_t num_seqs,
                            int32_t num_q_tokens, int32_t* max_q_len, int32_t num_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t num_blocks, int32_t max_context_len) {
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "NULL pointer");
    if (pa_status s = check_shape(num_kv_heads, head_dim, block_size)) return s;
    if (num_heads <= 0 || num_heads % num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "num_heads %d is not a multiple of num_kv_heads %d",
                    num_heads, num_kv_heads);
    if (!is_kv_dtype(kv_dtype)) return fail(PA_ERR_INVALID_ARG, "kv_dtype %d", (int)kv_dtype);
    if (q_dtype != PA_F16 && q_dtype != PA_BF16)
        return fail(PA_ERR_UNSUPPORTED, "q_dtype %d (F16 or BF16)", (int)q_dtype);
    if ((kv_dtype == PA_F16 || kv_dtype == PA_BF16) && q_dtype != kv_dtype)
        return fail(PA_ERR_UNSUPPORTED, "q_dtype must equal kv_dtype for F16/BF16 caches");
    if (kv_dtype == PA_FP8_E4M3 && (!k_scale || !v_scale))
        return fail(PA_ERR_INVALID_ARG, "FP8 cache needs per-head k_scale and v_scale");
    if (out_dtype != PA_F32 && out_dtype != q_dtype)
        return fail(PA_ERR_UNSUPPORTED, "out_dtype must be F32 or the q dtype");
    if (kv_dtype == PA_INT8 && (!k_scale || !v_scale || !k_zp || !v_zp))
        return fail(PA_ERR_INVALID_ARG, "INT8 cache needs k_scale, v_scale, k_zp, v_zp");
    if (!query_start_loc) {
        if (num_q_tokens != num_seqs)
            return fail(PA_ERR_INVALID_ARG, "without query_start_loc num_q_tokens must equal num_seqs");
        *max_q_len = 1;
    }
    if (*max_q_len < 1 || num_q_tokens < num_seqs)
        return fail(PA_ERR_INVALID_ARG, "max_q_len %d / num_q_tokens %d", *max_q_len, num_q_tokens);
    if (max_context_len < *max_q_len)
        return fail(PA_ERR_INVALID_ARG, "max_context_len %d < max_q_len %d", max_context_len,
                    *max_q_len);
    if (num_blocks <= 0) return fail(PA_ERR_INVALID_ARG, "num_blocks %d", num_blocks);
    if ((int64_t)max_blocks_per_seq * block_size < max_context_len)
        return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq %d cannot hold %d tokens",
                    max_blocks_per_seq, max_context_len);
    if (((uintptr_t)k_cache | (uintptr_t)v_cache) % 16)
        return fail(PA_ERR_INVALID_ARG, "k_cache and v_cache must be 16-byte aligned");
    if (((uintptr_t)q | (uintptr_t)out) % 16)
        return fail(PA_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    return PA_OK;
}

// PA_VALIDATE=1: context lengths, query runs and block-table entries of every
// sequence, read back from the device.
pa_status validate_decode_arrays(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens, const int32_t* query_start_loc,
                                 int32_t num_seqs, int32_t num_q_tokens, int32_t max_q_len,
                                 int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                                 cudaStream_t st) {
    std::vector<int32_t> lens, bt, qsl;
    if (pa_status s = to_host(lens, context_lens, (size_t)num_seqs, st)) return s;
    if (pa_status s = to_host(bt, block_tables, (size_t)num_seqs * max_blocks_per_seq, st))
        return s;
    if (query_start_loc)
        if (pa_status s = to_host(qsl, query_start_loc, (size_t)num_seqs + 1, st)) return s;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t r = query_start_loc ? qsl[s + 1] - qsl[s] : 1;
        int32_t L = lens[s];
        if (query_start_loc && (qsl[s] < 0 || qsl[s + 1] > num_q_tokens))
            return fail(PA_ERR_VALIDATION, "query_start_loc of sequence %d out of range", s);
        if (r < 1 || r > max_q_len || L < r || L > max_context_len)
            return fail(PA_ERR_VALIDATION, "sequence %d: context_len %d, query run %d", s, L, r);
        for (int32_t b = 0; b < (L + block_size - 1) / block_size; ++b) {
            int32_t e = bt[(size_t)s * max_blocks_per_seq + b];
            if (e < 0 || e >= num_blocks)
                return fail(PA_ERR_VALIDATION, "block_tables[%d][%d] = %d outside [0,%d)", s, b,
                            e, num_blocks);
        }
    }
    return PA_OK;
}

}  // namespace pa

extern "C" pa_status pa_decode(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype,
                               const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
                               const float* k_scale, const float* v_scale, const int8_t* k_zp,
                               const int8_t* v_zp, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                               const int32_t* query_start_loc, int32_t num_seqs,
                               int32_t num_q_tokens, int32_t max_q_len, int32_t num_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, float scale, int32_t max_context_len,
                               int32_t partition_size, void* workspace,
                               size_t workspace_bytes, void* stream) {
    if (num_seqs < 0) return fail(PA_ERR_INVALID_ARG, "num_seqs < 0");
    if (num_seqs == 0) return PA_OK;
    if (pa_status s = pa::check_decode_args(
            out, out_dtype, q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale, k_zp, v_zp,
            block_tables, max_blocks_per_seq, context_lens, query_start_loc, num_seqs,
            num_q_tokens, &max_q_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
            max_context_len))
        return s;
    const int32_t P = partition_size;
    if (P < 0 || P % block_size != 0)
        return fail(PA_ERR_INVALID_ARG, "partition_size %d is not a multiple of %d", P, block_size);
    const int64_t parts = P > 0 ? (max_context_len + (int64_t)P - 1) / P : 1;
    if (parts > 65535) return fail(PA_ERR_UNSUPPORTED, "too many partitions (%lld)", (long long)parts);
    const size_t need = pa_decode_workspace_size(num_seqs, num_q_tokens, num_heads, num_kv_heads,
                                                 head_dim, max_q_len, max_context_len,
                                                 partition_size);
    if (need > 0 && (!workspace || workspace_bytes < need || (uintptr_t)workspace % 256))
        return fail(PA_ERR_INVALID_ARG, "workspace needs %zu bytes, 256-byte aligned (got %zu)",
                    need, workspace_bytes);
    cudaStream_t st = (cudaStream_t)stream;
    if (pa::validate_enabled())
        if (pa_status s = pa::validate_decode_arrays(block_tables, max_blocks_per_seq,
                                                     context_lens, query_start_loc, num_seqs,
                                                     num_q_tokens, max_q_len, block_size,
                                                     num_blocks, max_context_len, st))
            return s;
    pa::DecodeArgs a{};
    a.out = out;
    a.out_dtype = out_dtype;
    a.q = q;
    a.q_dtype = q_dtype;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.kv_dtype = kv_dtype;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.k_zp = k_zp;
    a.v_zp = v_zp;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.query_start_loc = query_start_loc;
    a.num_seqs = num_seqs;
    a.num_q_tokens = num_q_tokens;
    a.max_q_len = max_q_len;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.max_context_len = max_context_len;
    a.partition_size = P;
    a.num_partitions = (int32_t)parts;
    // the arrival counters first (kept zero), then this call's scratch
    if (P == 0) {
        a.arrivals = static_cast<unsigned int*>(workspace);
        a.slots = static_cast<char*>(workspace) + pa::kArrivalBytes;
    } else if (parts > 1) {
        const size_t rows = (size_t)num_q_tokens * num_heads * parts;
        char* w = static_cast<char*>(workspace) + pa::kArrivalBytes;
        a.o_part = reinterpret_cast<float*>(w);
        a.m_part = reinterpret_cast<float*>(w + align256(rows * head_dim * sizeof(float)));
        a.l_part = reinterpret_cast<float*>(w + align256(rows * head_dim * sizeof(float)) +
                                            align256(rows * sizeof(float)));
    }
    a.stream = st;
    return pa::launch_decode(a);
}

static_assert(PA_DEVERR_WAIT_FULL == pa::ERR_WAIT_FULL && PA_DEVERR_WAIT_EMPTY == pa::ERR_WAIT_EMPTY &&
                  PA_DEVERR_WAIT_DRAIN == pa::ERR_WAIT_DRAIN &&
                  PA_DEVERR_BAD_BLOCK == pa::ERR_BAD_BLOCK && PA_DEVERR_BAD_SLOT == pa::ERR_BAD_SLOT &&
                  PA_DEVERR_BAD_GROUP == pa::ERR_BAD_GROUP &&
                  PA_DEVERR_WORKSPACE == pa::ERR_WORKSPACE,
              "device error bits of pa.h and the kernels agree");

extern "C" pa_status pa_device_error(void* stream, uint32_t* code) {
    if (!code) return fail(PA_ERR_INVALID_ARG, "code is NULL");
    *code = 0;
    unsigned int* w = pa::device_error_word();
    if (!w) return fail(PA_ERR_CUDA, "cannot resolve the device error word");
    cudaStream_t st = (cudaStream_t)stream;
    unsigned int h = 0;
    if (pa_status s = pa::cuda_status(cudaStreamSynchronize(st), "pa_device_error: sync")) return s;
    if (pa_status s = pa::cuda_status(cudaMemcpy(&h, w, sizeof h, cudaMemcpyDeviceToHost),
                                      "pa_device_error: read"))
        return s;
    if (h) {
        unsigned int zero = 0;
        cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice);
        *code = h;
        return fail(PA_ERR_DEVICE, "device error word 0x%x", h);
    }
    return PA_OK;
}
