// pa_decode_no_alloc: pa_decode for callers that cannot allocate device
// memory. The split-KV workspace lives in a file-scope device array of fixed
// size instead of caller memory; everything else is pa_decode unchanged.
//
// Size: 40 MiB holds the largest workspace of any call with at most 16 query
// rows per KV head (q heads per KV head x the longest query run), whatever
// the batch: 24 KiB of arrival counters, up to 32 KiB of prefix sums and
// 2 x 2048 partial slots of 8,352 bytes (head_dim 128) -- about 32.7 MiB.
#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = (size_t)40 << 20;   // 40 MiB per device

// Held by every GPU that loads this library, for the life of the process.
static __device__ __align__(256) unsigned char g_decode_workspace[kStaticWorkspaceBytes];

// Device address of g_decode_workspace on the current device. In host code
// the symbol names a host-side stand-in, never the device array, so the
// address is resolved once per device (with that device current) and cached.
pa_status workspace_address(void** out) {
    static std::mutex mu;
    static std::vector<void*> per_device;
    int dev = 0;
    if (pa_status s = pa::cuda_status(cudaGetDevice(&dev), "pa_decode_no_alloc: cudaGetDevice"))
        return s;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)per_device.size() <= dev) per_device.resize(dev + 1, nullptr);
    if (!per_device[dev]) {
        void* p = nullptr;
        if (pa_status s = pa::cuda_status(cudaGetSymbolAddress(&p, g_decode_workspace),
                                          "pa_decode_no_alloc: cudaGetSymbolAddress"))
            return s;
        per_device[dev] = p;
    }
    *out = per_device[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_no_alloc(
    void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype, const void* k_cache,
    const void* v_cache, pa_dtype kv_dtype, const float* k_scale, const float* v_scale,
    const int8_t* k_zp, const int8_t* v_zp, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, const int32_t* query_start_loc,
    int32_t num_seqs, int32_t num_q_tokens, int32_t max_q_len, int32_t num_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks,
    float scale, int32_t max_context_len, int32_t partition_size, void* stream) {
    const size_t need = pa_decode_workspace_size(num_seqs, num_q_tokens, num_heads, num_kv_heads,
                                                 head_dim, max_q_len, max_context_len,
                                                 partition_size);
    if (need > kStaticWorkspaceBytes)
        return pa::fail(PA_ERR_UNSUPPORTED,
                        "pa_decode_no_alloc: this call needs %zu bytes of split-KV workspace, "
                        "more than the built-in %zu; use pa_decode with caller memory",
                        need, kStaticWorkspaceBytes);
    void* ws = nullptr;
    if (need > 0) {
        if (pa_status s = workspace_address(&ws)) return s;
        // The arrival counters must be zero when a call starts. A call whose
        // bounded wait gave up can leave some part-counted, and the caller has
        // no pointer to this array to clear them, so every call clears them
        // itself, in stream order before its kernels (a memset, no allocation).
        if (pa_status s = pa::cuda_status(
                cudaMemsetAsync(ws, 0, (size_t)pa::kArrivalBytes, static_cast<cudaStream_t>(stream)),
                "pa_decode_no_alloc: clear the arrival counters"))
            return s;
    }
    return pa_decode(out, out_dtype, q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                     k_zp, v_zp, block_tables, max_blocks_per_seq, context_lens,
                     query_start_loc, num_seqs, num_q_tokens, max_q_len, num_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, scale, max_context_len,
                     partition_size, ws, need, stream);
}
