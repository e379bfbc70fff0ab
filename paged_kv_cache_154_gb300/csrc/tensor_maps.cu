// TMA tensor maps of the paged caches (host side), shared by the decode
// kernels: a cache viewed as rows of head_dim elements,
// [num_blocks * num_kv_heads * 16 rows][head_dim], one box per (block, kv
// head) tile of 16 rows. A few recently used maps are kept so that a decode
// step does not re-encode them.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pa_internal.h"

namespace {

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

// 16-bit elements: box 16 rows x 64 columns with 128-byte swizzle (head_dim
// 128 takes two boxes). 8-bit codes: box 16 rows x head_dim, 128-byte swizzle
// for head_dim 128 and 64-byte swizzle for head_dim 64 (one swizzle span per
// row either way).
pa_status make_map(CUtensorMap* m, const void* cache, int num_blocks, int hkv, int d,
                   int elem_bytes) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return pa::fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const uint64_t rows = (uint64_t)num_blocks * hkv * 16;
    if (rows > 0x7fffffffull) return pa::fail(PA_ERR_UNSUPPORTED, "cache has too many rows for TMA");
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * elem_bytes};
    cuuint32_t box[2] = {elem_bytes == 2 ? 64u : (cuuint32_t)d, 16u};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType type =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapSwizzle swz = (elem_bytes == 1 && d == 64) ? CU_TENSOR_MAP_SWIZZLE_64B
                                                                : CU_TENSOR_MAP_SWIZZLE_128B;
    CUresult r = fn(m, type, 2, const_cast<void*>(cache), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return pa::fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PA_OK;
}

// the whole-tile view of a 16-bit, head_dim 128 cache (see pa_internal.h)
pa_status make_map_tile(CUtensorMap* m, const void* cache, int num_blocks, int hkv) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return pa::fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const uint64_t rows = (uint64_t)num_blocks * hkv * 16;
    if (rows > 0x7fffffffull) return pa::fail(PA_ERR_UNSUPPORTED, "cache has too many rows for TMA");
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, 2};
    cuuint64_t strides[2] = {256, 128};   // bytes: next row, next half
    cuuint32_t box[3] = {64u, 16u, 2u};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(cache), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return pa::fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled (tile view) failed (%d)", (int)r);
    return PA_OK;
}

struct Entry {
    const void* ptr;
    int num_blocks, num_kv_heads, head_dim, elem_bytes, device;
    CUtensorMap map;
};
std::mutex g_mu;
Entry g_entries[32];
int g_n = 0, g_next = 0;

}  // namespace

namespace pa {

pa_status cache_tensor_map_tile(CUtensorMap* out, const void* ptr, int num_blocks,
                                int num_kv_heads) {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_n; ++i) {
        const Entry& e = g_entries[i];
        // elem_bytes -2 marks the tile view
        if (e.ptr == ptr && e.num_blocks == num_blocks && e.num_kv_heads == num_kv_heads &&
            e.head_dim == 128 && e.elem_bytes == -2 && e.device == dev) {
            *out = e.map;
            return PA_OK;
        }
    }
    CUtensorMap m;
    if (pa_status s = make_map_tile(&m, ptr, num_blocks, num_kv_heads)) return s;
    g_entries[g_next] = Entry{ptr, num_blocks, num_kv_heads, 128, -2, dev, m};
    g_next = (g_next + 1) % 32;
    if (g_n < 32) ++g_n;
    *out = m;
    return PA_OK;
}

pa_status cache_tensor_map(CUtensorMap* out, const void* ptr, int num_blocks, int num_kv_heads,
                           int head_dim, int elem_bytes) {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_n; ++i) {
        const Entry& e = g_entries[i];
        if (e.ptr == ptr && e.num_blocks == num_blocks && e.num_kv_heads == num_kv_heads &&
            e.head_dim == head_dim && e.elem_bytes == elem_bytes && e.device == dev) {
            *out = e.map;
            return PA_OK;
        }
    }
    CUtensorMap m;
    if (pa_status s = make_map(&m, ptr, num_blocks, num_kv_heads, head_dim, elem_bytes)) return s;
    g_entries[g_next] = Entry{ptr, num_blocks, num_kv_heads, head_dim, elem_bytes, dev, m};
    g_next = (g_next + 1) % 32;
    if (g_n < 32) ++g_n;
    *out = m;
    return PA_OK;
}

}  // namespace pa
