// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Records a formatted message for pa_last_error() and returns `s`.
pa_status fail(pa_status s, const char* fmt, ...);
// Maps a CUDA error to PA_ERR_CUDA with a message; PA_OK on cudaSuccess.
pa_status cuda_status(cudaError_t e, const char* what);

// Pointer to this device's error word (kernels OR codes into it instead of
// trapping). Null if it cannot be resolved.
unsigned int* device_error_word();

// Error codes OR-ed into the device error word.
enum : unsigned int {
    ERR_WAIT_FULL = 1u << 0,    // consumer gave up waiting for a staged tile
    ERR_WAIT_EMPTY = 1u << 1,   // producer gave up waiting for a free stage
    ERR_WAIT_DRAIN = 1u << 2,   // exit drain gave up on an in-flight copy
    ERR_BAD_BLOCK = 1u << 3,    // a block-table entry outside the pool
    ERR_BAD_SLOT = 1u << 4,     // a slot outside the pool
    ERR_BAD_GROUP = 1u << 5,    // a shared-prefix group range or prefix length out of bounds
    ERR_WORKSPACE = 1u << 6,    // a split-segment arrival counter was not zero at the start
};

inline int dtype_bytes(pa_dtype t) {
    switch (t) {
        case PA_F16: case PA_BF16: return 2;
        case PA_F32: return 4;
        case PA_INT8: case PA_FP8_E4M3: return 1;
    }
    return 0;
}

bool validate_enabled();

// Launch with programmatic stream serialization: the kernel may begin while
// the previous kernel in the stream finishes; it must call
// grid_dependency_wait() (ptx.cuh) before touching memory that kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

struct AppendArgs {
    const void* key;
    const void* value;
    pa_dtype src_dtype;
    void* k_cache;
    void* v_cache;
    pa_dtype kv_dtype;
    float* k_scale;
    float* v_scale;
    int8_t* k_zp;
    int8_t* v_zp;
    const int64_t* slots;
    int32_t num_tokens;
    int32_t num_blocks;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    cudaStream_t stream;
};
pa_status launch_append_kv(const AppendArgs& a);

struct CopyArgs {
    void* arrays[6];          // k, v, k_scale, v_scale, k_zp, v_zp (unused = null)
    int64_t bytes_per_block[6];
    const int32_t* pairs;
    int32_t n_pairs;
    int32_t num_blocks;
    cudaStream_t stream;
};
pa_status launch_copy_blocks(const CopyArgs& a);

struct DecodeArgs {
    void* out;
    pa_dtype out_dtype;
    const void* q;
    pa_dtype q_dtype;
    const void* k_cache;
    const void* v_cache;
    pa_dtype kv_dtype;
    const float* k_scale;
    const float* v_scale;
    const int8_t* k_zp;
    const int8_t* v_zp;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* context_lens;
    const int32_t* query_start_loc;
    int32_t num_seqs;
    int32_t num_q_tokens;
    int32_t max_q_len;
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t num_blocks;
    float scale;
    int32_t max_context_len;
    int32_t partition_size;
    int32_t num_partitions;
    float* o_part;           // partitioned schedule (partition_size > 0)
    float* m_part;
    float* l_part;
    void* slots;             // balanced schedule (partition_size == 0)
    unsigned int* arrivals;  // balanced schedule: 3 x kBalancedMaxWorkers counters, zero before the
                             // call and left zero by it; null: merge cut segments in a
                             // separate reduce kernel
    // balanced schedule of a 16-bit cache only (null / 0 otherwise):
    const int32_t* ctx_start;  // [num_seqs] first attended token, a multiple of 16
    float* lse_out;            // [num_q_tokens][num_heads] base-2 log-sum-exp per output row
    int unmasked;              // every query row sees every key < context_len
    int max_workers;           // balanced 16-bit decode: at most this many worker warps (0: none)
    cudaStream_t stream;
};
pa_status launch_decode(const DecodeArgs& a);

// TMA tensor map of a cache ([num_blocks][num_kv_heads][16][head_dim] of
// elem_bytes-byte elements), cached per (pointer, shape, device)
// (tensor_maps.cu).
pa_status cache_tensor_map(CUtensorMap* out, const void* ptr, int num_blocks, int num_kv_heads,
                           int head_dim, int elem_bytes);
// 16-bit cache with head_dim 128 viewed in three dimensions -- 64 columns,
// rows, the two 64-column halves of a row -- so that one box of 16 rows x 2
// halves (4 KiB) moves a whole (block, kv head) tile in one copy, laid out in
// shared memory as [half][16 rows][128 B] with the 128-byte swizzle (the
// layout two 2-D boxes give).
pa_status cache_tensor_map_tile(CUtensorMap* out, const void* ptr, int num_blocks,
                                int num_kv_heads);

// Host-side argument checks of the decode entry points (capi.cu).
pa_status check_decode_args(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype,
                            const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
                            const float* k_scale, const float* v_scale, const int8_t* k_zp,
                            const int8_t* v_zp, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* context_lens,
                            const int32_t* query_start_loc, int32_t num_seqs,
                            int32_t num_q_tokens, int32_t* max_q_len, int32_t num_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t num_blocks, int32_t max_context_len);
pa_status validate_decode_arrays(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens, const int32_t* query_start_loc,
                                 int32_t num_seqs, int32_t num_q_tokens, int32_t max_q_len,
                                 int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                                 cudaStream_t st);

// Balanced schedule (partition_size == 0): at most this many worker warps
// (and partial-slot pairs), and at most this many sequences per call (their
// prefix sums live in shared memory).
constexpr int kBalancedMaxWorkers = 2048;
constexpr int kBalancedMaxSeqs = 8192;
// The first bytes of every decode workspace: three regions of one arrival
// counter per worker (see DecodeArgs::arrivals), at the same offset whatever
// the call's shape so that one buffer can serve calls of different sizes.
constexpr int64_t kArrivalBytes = 3 * 4 * kBalancedMaxWorkers;

struct BalancedShape {
    int rows_per_tile;       // query rows per worker tile of this kernel family
    int64_t max_chunks;      // row tiles per (sequence, kv head), at most
    int64_t workers;         // cap on workers (partial-slot pairs)
    int64_t cum_bytes;       // workspace prefix sums, 256-byte aligned
    int64_t slot_bytes;      // one partial slot
    int64_t virtual_blocks;  // upper bound of the schedule's work units
    int64_t workspace_bytes;
};

// Kernel families of the balanced schedule.
enum TileKind { kTile16Bit = 0, kTileInt8 = 1, kTileFp8 = 2 };

// Query rows per tile: 16 while a KV head has at most 16 rows (G q heads x
// the longest query run), else 64 for the 16-bit kernels (four warps of 16
// rows share each block); the INT8 and FP8 kernels always use 16 (one warp
// per tile, further rows as further chunks).
inline int tile_rows(int64_t rows, int kind) {
    if (rows <= 16 || kind == kTileFp8 || kind == kTileInt8) return 16;
    return 64;
}

// The workspace is sized for every kernel family: the worker cap from the
// smallest tile (most work units) and the slot from the largest.
inline BalancedShape balanced_shape(int num_seqs, int num_heads, int num_kv_heads,
                                    int head_dim, int max_q_len, int max_context_len,
                                    int kind = kTile16Bit) {
    BalancedShape b{};
    const int64_t rows = (int64_t)(num_heads / num_kv_heads) * max_q_len;
    b.rows_per_tile = tile_rows(rows, kind);
    b.max_chunks = (rows + b.rows_per_tile - 1) / b.rows_per_tile;
    const int64_t small = tile_rows(rows, kTileFp8), large = tile_rows(rows, kTile16Bit);
    b.virtual_blocks = (int64_t)num_seqs * num_kv_heads * ((rows + small - 1) / small) *
                       ((max_context_len + 15) / 16);
    b.workers = b.virtual_blocks < kBalancedMaxWorkers ? b.virtual_blocks : kBalancedMaxWorkers;
    b.cum_bytes = ((int64_t)4 * (num_seqs + 1) + 255) / 256 * 256;
    b.slot_bytes = (32 + 4 * large * (head_dim + 2) + 15) / 16 * 16;
    b.workspace_bytes = b.cum_bytes + 2 * b.workers * b.slot_bytes;
    return b;
}

// INT8 decode with tokens in the M dimension of tensor-core products
// (paged_decode_int8_tc.cu): for more than 16 query rows per KV head at
// head_dim 128; int8_tc_applies says whether a call takes it.
struct DecodeArgs;
bool int8_tc_applies(const DecodeArgs& a);
pa_status launch_decode_int8_tc(const DecodeArgs& a);

// Limits of the balanced schedule that the host can check.
inline pa_status balanced_check(const DecodeArgs& a) {
    if (a.num_seqs > kBalancedMaxSeqs)
        return fail(PA_ERR_UNSUPPORTED, "more than %d sequences in one call with partition_size 0",
                    kBalancedMaxSeqs);
    const BalancedShape b = balanced_shape(a.num_seqs, a.num_heads, a.num_kv_heads, a.head_dim,
                                           a.max_q_len, a.max_context_len,
                                           a.kv_dtype == PA_INT8       ? kTileInt8
                                           : a.kv_dtype == PA_FP8_E4M3 ? kTileFp8
                                                                       : kTile16Bit);
    if (b.max_chunks > 255 || b.virtual_blocks > 0x7fffffffll)
        return fail(PA_ERR_UNSUPPORTED, "decode call too large for one balanced launch");
    return PA_OK;
}

}  // namespace pa
