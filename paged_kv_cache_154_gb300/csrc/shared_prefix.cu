// Shared-prefix ("read-once") decode for copy-on-write forks.
//
// Forks of one prompt hold the same physical blocks for their common prefix
// ("KV Cache ... PagedAttention" §2.1: forks share blocks by reference count
// and copy only on write; the best-of-N workload forks one prompt N ways).
// Plain paged decode reads those blocks once per fork. Here each group of
// forks reads them once for all its query rows:
//
//   1. prefix phase: one pseudo-sequence per group, whose query rows are all
//      the group's rows and whose keys are the first prefix_len[g] tokens
//      (every one of them earlier than every query, so no causal mask),
//   2. suffix phase: every sequence over its own tokens [prefix_len, L),
//      with the usual causal offset for verify runs,
//   3. merge: each row combines the two states by their log-sum-exp,
//      out = (2^(a - M) o_a + 2^(b - M) o_b) / (2^(a - M) + 2^(b - M)),
//      the same rule the split-KV reduce applies to partitions.
//
// Phases 1 and 2 are the balanced 16-bit decode kernel (balanced.cuh) with
// the ctx_start / unmasked / lse_out extensions; both write fp32 rows and
// their log-sum-exp into the workspace, and the merge writes the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <math.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "pa_internal.h"
#include "ptx.cuh"

namespace pa {
int64_t prefix_tc_ctas(const DecodeArgs& a, int sms);
}

namespace {

constexpr int kBS = 16;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct PrepArgs {
    const int32_t* group_start;   // [n_groups + 1]
    const int32_t* prefix_len;    // [n_groups]
    const int32_t* qsl;           // [num_seqs + 1] or null
    const int32_t* block_tables;  // [num_seqs][max_blocks]
    int32_t max_blocks;
    int32_t num_seqs;
    int32_t n_groups;
    int64_t rows;                 // num_q_tokens * num_heads
    int32_t* g_qsl;               // out [n_groups + 1]
    int32_t* g_ctx;               // out [n_groups]
    int32_t* g_tables;            // out [n_groups][max_blocks]
    int32_t* ctx_start;           // out [num_seqs]
    float* lse_a;                 // out [rows] = -inf
    float* lse_b;                 // out [rows] = -inf
    unsigned int* err;
};

// One CTA per group (plus a grid-stride fill of the log-sum-exp arrays): the
// group's pseudo-sequence (query range, prefix length, block table = the
// first member's), and every member's first attended token.
__global__ void __launch_bounds__(128) prefix_prep_kernel(const PrepArgs a) {
    pa::grid_dependency_wait();
    pa::grid_dependents_launch();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.rows; i += stride) {
        a.lse_a[i] = -INFINITY;
        a.lse_b[i] = -INFINITY;
    }
    const int g = blockIdx.x;
    if (g >= a.n_groups) return;
    // out-of-range group arrays are clamped (and reported), never followed
    int s0 = __ldg(a.group_start + g), s1 = __ldg(a.group_start + g + 1);
    int P = __ldg(a.prefix_len + g);
    if (s0 < 0 || s0 >= a.num_seqs || s1 < s0 || s1 > a.num_seqs || P < 0 ||
        P > a.max_blocks * kBS) {
        if (threadIdx.x == 0 && a.err) atomicOr(a.err, pa::ERR_BAD_GROUP);
        s0 = min(max(s0, 0), a.num_seqs - 1);
        s1 = min(max(s1, s0), a.num_seqs);
        P = min(max(P, 0), a.max_blocks * kBS);
    }
    if (threadIdx.x == 0) {
        a.g_qsl[g] = a.qsl ? __ldg(a.qsl + s0) : s0;
        a.g_ctx[g] = P;
        if (g == a.n_groups - 1) a.g_qsl[g + 1] = a.qsl ? __ldg(a.qsl + s1) : s1;
    }
    for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) a.ctx_start[s] = P;
    const int nb = P / kBS;
    for (int b = threadIdx.x; b < nb; b += blockDim.x)
        a.g_tables[(int64_t)g * a.max_blocks + b] =
            __ldg(a.block_tables + (int64_t)s0 * a.max_blocks + b);
}

// One warp per output row (query token, q head): merge the prefix state
// (o_a, lse_a) and the suffix state (o_b, lse_b); a side whose log-sum-exp is
// -inf saw no key and is left out (its o is never read).
template <typename TO, int D>
__global__ void __launch_bounds__(128)
    prefix_merge_kernel(void* out, int out_f32, const float* o_a, const float* lse_a,
                        const float* o_b, const float* lse_b, int64_t rows) {
    constexpr int EPL = D / 32;
    pa::grid_dependency_wait();
    pa::grid_dependents_launch();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float la = __ldg(lse_a + row), lb = __ldg(lse_b + row);
    const float M = fmaxf(la, lb);
    const float wa = la == -INFINITY ? 0.f : exp2f(la - M);
    const float wb = lb == -INFINITY ? 0.f : exp2f(lb - M);
    const float inv = 1.f / (wa + wb);
    float v[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] = 0.f;
    const int64_t base = row * D + lane * EPL;
    if (wa > 0.f) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[e] += wa * __ldg(o_a + base + e);
    }
    if (wb > 0.f) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[e] += wb * __ldg(o_b + base + e);
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const float x = v[e] * inv;
        if (out_f32) {
            static_cast<float*>(out)[base + e] = x;
        } else if constexpr (std::is_same<TO, __half>::value) {
            static_cast<__half*>(out)[base + e] = __float2half_rn(x);
        } else {
            static_cast<__nv_bfloat16*>(out)[base + e] = __float2bfloat16_rn(x);
        }
    }
}

// A second stream of this device and two events: the suffix phase runs on
// it beside the prefix phase when the prefix phase leaves SMs free (its
// tensor-core kernel holds one CTA per SM). Created once per device, kept
// for the life of the process; the fork and the join are stream-ordered
// event records and waits, which graph capture turns into edges.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

// held from an event record to the wait that reads it, so calls from
// several host threads do not interleave their records
std::mutex& side_mutex() {
    static std::mutex mu;
    return mu;
}

pa_status side_stream(SideStream* out) {
    static std::mutex mu;
    static std::vector<SideStream> per_device;
    int dev = 0;
    if (pa_status s = pa::cuda_status(cudaGetDevice(&dev), "cudaGetDevice")) return s;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)per_device.size() <= dev) per_device.resize(dev + 1);
    SideStream& ss = per_device[dev];
    if (!ss.stream) {
        SideStream t;
        if (pa_status s = pa::cuda_status(
                cudaStreamCreateWithFlags(&t.stream, cudaStreamNonBlocking), "side stream"))
            return s;
        if (pa_status s = pa::cuda_status(
                cudaEventCreateWithFlags(&t.fork, cudaEventDisableTiming), "side stream event"))
            return s;
        if (pa_status s = pa::cuda_status(
                cudaEventCreateWithFlags(&t.join, cudaEventDisableTiming), "side stream event"))
            return s;
        ss = t;
    }
    *out = ss;
    return PA_OK;
}

// Workspace: the arrival counters (kept zero; the two phases use them one
// after the other), the two decode calls' own scratch, the two phases' fp32
// rows and log-sum-exps, and the pseudo-sequence arrays.
struct SpLayout {
    size_t arr, ws_a, ws_b, o_a, lse_a, o_b, lse_b, g_qsl, g_ctx, g_tables, ctx_start, total;
};

SpLayout sp_layout(int32_t num_seqs, int32_t num_q_tokens, int32_t num_heads,
                   int32_t num_kv_heads, int32_t head_dim, int32_t max_q_len,
                   int32_t max_context_len, int32_t num_groups, int32_t max_group_q_len,
                   int32_t max_prefix_len, int32_t max_blocks_per_seq) {
    SpLayout l{};
    const size_t rows = (size_t)num_q_tokens * num_heads;
    const pa::BalancedShape sa = pa::balanced_shape(num_groups, num_heads, num_kv_heads, head_dim,
                                                    max_group_q_len, std::max(1, max_prefix_len));
    const pa::BalancedShape sb = pa::balanced_shape(num_seqs, num_heads, num_kv_heads, head_dim,
                                                    max_q_len, max_context_len);
    size_t at = 0;
    auto take = [&](size_t bytes) {
        const size_t here = at;
        at += align256(bytes);
        return here;
    };
    l.arr = take((size_t)pa::kArrivalBytes);
    l.ws_a = take((size_t)sa.workspace_bytes);
    l.ws_b = take((size_t)sb.workspace_bytes);
    l.o_a = take(rows * head_dim * sizeof(float));
    l.lse_a = take(rows * sizeof(float));
    l.o_b = take(rows * head_dim * sizeof(float));
    l.lse_b = take(rows * sizeof(float));
    l.g_qsl = take(((size_t)num_groups + 1) * sizeof(int32_t));
    l.g_ctx = take((size_t)num_groups * sizeof(int32_t));
    l.g_tables = take((size_t)num_groups * max_blocks_per_seq * sizeof(int32_t));
    l.ctx_start = take((size_t)num_seqs * sizeof(int32_t));
    l.total = at;
    return l;
}

// PA_VALIDATE=1: the groups tile the batch in order, every prefix is a whole
// number of blocks that every member holds with the same physical ids, and
// every prefix token precedes every query of its group.
pa_status validate_groups(const int32_t* group_start, const int32_t* prefix_len, int32_t ng,
                          const int32_t* block_tables, int32_t max_blocks,
                          const int32_t* context_lens, const int32_t* qsl, int32_t num_seqs,
                          int32_t max_group_q_len, int32_t max_prefix_len, cudaStream_t st) {
    std::vector<int32_t> gs(ng + 1), pl(ng), lens(num_seqs), bt((size_t)num_seqs * max_blocks),
        q(qsl ? num_seqs + 1 : 0);
    if (pa_status s = pa::cuda_status(cudaStreamSynchronize(st), "validate: sync")) return s;
    auto get = [](std::vector<int32_t>& h, const int32_t* d) {
        return h.empty() ? cudaSuccess
                         : cudaMemcpy(h.data(), d, h.size() * sizeof(int32_t),
                                      cudaMemcpyDeviceToHost);
    };
    if (get(gs, group_start) != cudaSuccess || get(pl, prefix_len) != cudaSuccess ||
        get(lens, context_lens) != cudaSuccess || get(bt, block_tables) != cudaSuccess ||
        (qsl && get(q, qsl) != cudaSuccess))
        return pa::fail(PA_ERR_CUDA, "validate: copy to host");
    if (gs[0] != 0 || gs[ng] != num_seqs)
        return pa::fail(PA_ERR_VALIDATION, "group_start must run from 0 to num_seqs");
    for (int32_t g = 0; g < ng; ++g) {
        if (gs[g + 1] <= gs[g]) return pa::fail(PA_ERR_VALIDATION, "group %d is empty", g);
        const int32_t P = pl[g];
        if (P < 0 || P % kBS || P > max_prefix_len)
            return pa::fail(PA_ERR_VALIDATION, "prefix_len[%d] = %d", g, P);
        int32_t nq = 0;
        for (int32_t s = gs[g]; s < gs[g + 1]; ++s) {
            const int32_t r = qsl ? q[s + 1] - q[s] : 1;
            nq += r;
            if (P > lens[s] - r + 1)
                return pa::fail(PA_ERR_VALIDATION,
                                "prefix_len[%d] = %d reaches a query of sequence %d", g, P, s);
            for (int32_t b = 0; b < P / kBS; ++b)
                if (bt[(size_t)s * max_blocks + b] != bt[(size_t)gs[g] * max_blocks + b])
                    return pa::fail(PA_ERR_VALIDATION,
                                    "sequence %d does not share prefix block %d of group %d", s,
                                    b, g);
        }
        if (nq > max_group_q_len)
            return pa::fail(PA_ERR_VALIDATION, "group %d has %d query tokens > max_group_q_len",
                            g, nq);
    }
    return PA_OK;
}

}  // namespace

extern "C" size_t pa_decode_shared_prefix_workspace_size(
    int32_t num_seqs, int32_t num_q_tokens, int32_t num_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t max_q_len, int32_t max_context_len, int32_t num_groups,
    int32_t max_group_q_len, int32_t max_prefix_len, int32_t max_blocks_per_seq) {
    if (num_seqs <= 0 || num_q_tokens <= 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || max_q_len <= 0 || max_context_len <= 0 || num_groups <= 0 ||
        max_group_q_len <= 0 || max_prefix_len < 0 || max_blocks_per_seq <= 0 ||
        num_heads % num_kv_heads != 0)
        return 0;
    return sp_layout(num_seqs, num_q_tokens, num_heads, num_kv_heads, head_dim, max_q_len,
                     max_context_len, num_groups, max_group_q_len, max_prefix_len,
                     max_blocks_per_seq)
        .total;
}

extern "C" pa_status pa_decode_shared_prefix(
    void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype, const void* k_cache,
    const void* v_cache, pa_dtype kv_dtype, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, const int32_t* query_start_loc,
    int32_t num_seqs, int32_t num_q_tokens, int32_t max_q_len, int32_t num_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
    int32_t max_context_len, const int32_t* group_start, const int32_t* prefix_len,
    int32_t num_groups, int32_t max_group_q_len, int32_t max_prefix_len, void* workspace,
    size_t workspace_bytes, void* stream) {
    if (num_seqs < 0) return pa::fail(PA_ERR_INVALID_ARG, "num_seqs < 0");
    if (num_seqs == 0) return PA_OK;
    if (kv_dtype != PA_F16 && kv_dtype != PA_BF16)
        return pa::fail(PA_ERR_UNSUPPORTED, "shared-prefix decode needs an F16 or BF16 cache");
    if (pa_status s = pa::check_decode_args(
            out, out_dtype, q, q_dtype, k_cache, v_cache, kv_dtype, nullptr, nullptr, nullptr,
            nullptr, block_tables, max_blocks_per_seq, context_lens, query_start_loc, num_seqs,
            num_q_tokens, &max_q_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
            max_context_len))
        return s;
    if (!group_start || !prefix_len) return pa::fail(PA_ERR_INVALID_ARG, "NULL group arrays");
    if (num_groups < 1 || num_groups > num_seqs)
        return pa::fail(PA_ERR_INVALID_ARG, "num_groups %d (1..num_seqs)", num_groups);
    if (max_group_q_len < max_q_len || max_group_q_len > num_q_tokens)
        return pa::fail(PA_ERR_INVALID_ARG, "max_group_q_len %d (max_q_len..num_q_tokens)",
                        max_group_q_len);
    if (max_prefix_len < 0 || max_prefix_len % block_size || max_prefix_len > max_context_len)
        return pa::fail(PA_ERR_INVALID_ARG, "max_prefix_len %d", max_prefix_len);
    const SpLayout lay = sp_layout(num_seqs, num_q_tokens, num_heads, num_kv_heads, head_dim,
                                   max_q_len, max_context_len, num_groups, max_group_q_len,
                                   max_prefix_len, max_blocks_per_seq);
    if (!workspace || workspace_bytes < lay.total || (uintptr_t)workspace % 256)
        return pa::fail(PA_ERR_INVALID_ARG, "workspace needs %zu bytes, 256-byte aligned (got %zu)",
                        lay.total, workspace_bytes);
    cudaStream_t st = (cudaStream_t)stream;
    if (pa::validate_enabled()) {
        if (pa_status s = pa::validate_decode_arrays(block_tables, max_blocks_per_seq,
                                                     context_lens, query_start_loc, num_seqs,
                                                     num_q_tokens, max_q_len, block_size,
                                                     num_blocks, max_context_len, st))
            return s;
        if (pa_status s = validate_groups(group_start, prefix_len, num_groups, block_tables,
                                          max_blocks_per_seq, context_lens, query_start_loc,
                                          num_seqs, max_group_q_len, max_prefix_len, st))
            return s;
    }
    char* w = static_cast<char*>(workspace);
    float* o_a = reinterpret_cast<float*>(w + lay.o_a);
    float* lse_a = reinterpret_cast<float*>(w + lay.lse_a);
    float* o_b = reinterpret_cast<float*>(w + lay.o_b);
    float* lse_b = reinterpret_cast<float*>(w + lay.lse_b);
    int32_t* g_qsl = reinterpret_cast<int32_t*>(w + lay.g_qsl);
    int32_t* g_ctx = reinterpret_cast<int32_t*>(w + lay.g_ctx);
    int32_t* g_tables = reinterpret_cast<int32_t*>(w + lay.g_tables);
    int32_t* ctx_start = reinterpret_cast<int32_t*>(w + lay.ctx_start);
    const int64_t rows = (int64_t)num_q_tokens * num_heads;

    PrepArgs pa_{group_start, prefix_len, query_start_loc, block_tables, max_blocks_per_seq,
                 num_seqs, num_groups, rows, g_qsl, g_ctx, g_tables, ctx_start, lse_a, lse_b,
                 pa::device_error_word()};
    if (pa_status s = pa::cuda_status(
            pa::launch_pdl(prefix_prep_kernel, dim3((unsigned)num_groups), dim3(128), 0, st, pa_),
            "shared-prefix prep launch"))
        return s;

    // phase 1: the groups' prefixes, every key visible to every row of the group
    pa::DecodeArgs a{};
    a.out = o_a;
    a.out_dtype = PA_F32;
    a.q = q;
    a.q_dtype = q_dtype;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.kv_dtype = kv_dtype;
    a.block_tables = g_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.context_lens = g_ctx;
    a.query_start_loc = g_qsl;
    a.num_seqs = num_groups;
    a.num_q_tokens = num_q_tokens;
    a.max_q_len = max_group_q_len;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.max_context_len = std::max(1, max_prefix_len);
    a.partition_size = 0;
    a.num_partitions = 1;
    a.slots = w + lay.ws_a;
    a.arrivals = reinterpret_cast<unsigned int*>(w + lay.arr);
    a.lse_out = lse_a;
    a.unmasked = 1;
    a.stream = st;
    // With the prefix phase on the tensor-core kernel (one CTA per SM, SMs
    // to spare), the suffix phase runs beside it on the side stream, with
    // its workers capped to the free SMs (three CTAs of four warps each).
    int dev = 0, sms = 0;
    if (pa_status s = pa::cuda_status(cudaGetDevice(&dev), "cudaGetDevice")) return s;
    if (pa_status s = pa::cuda_status(
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count"))
        return s;
    const int64_t tc_ctas = pa::prefix_tc_ctas(a, sms);
    const int64_t free_sms = sms - tc_ctas;
    SideStream side{};
    const bool beside = tc_ctas > 0 && free_sms >= sms / 16;
    if (beside) {
        if (pa_status s = side_stream(&side)) return s;
        std::lock_guard<std::mutex> lock(side_mutex());
        if (pa_status s = pa::cuda_status(cudaEventRecord(side.fork, st), "fork record")) return s;
        if (pa_status s = pa::cuda_status(cudaStreamWaitEvent(side.stream, side.fork, 0),
                                          "fork wait"))
            return s;
    }
    if (pa_status s = pa::launch_decode(a)) return s;

    // phase 2: every sequence from the end of its group's prefix
    a.out = o_b;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start_loc = query_start_loc;
    a.num_seqs = num_seqs;
    a.max_q_len = max_q_len;
    a.max_context_len = max_context_len;
    a.slots = w + lay.ws_b;
    // the private suffixes are short (a few blocks per share), where the
    // reduce kernel merges faster than the decode kernel's tail
    a.arrivals = nullptr;
    a.ctx_start = ctx_start;
    a.lse_out = lse_b;
    a.unmasked = 0;
    if (beside) {
        a.stream = side.stream;
        a.max_workers = (int)(free_sms * 3 * 4);
    }
    if (pa_status s = pa::launch_decode(a)) return s;
    if (beside) {   // the merge waits for the suffix phase
        std::lock_guard<std::mutex> lock(side_mutex());
        if (pa_status s = pa::cuda_status(cudaEventRecord(side.join, side.stream), "join record"))
            return s;
        if (pa_status s = pa::cuda_status(cudaStreamWaitEvent(st, side.join, 0), "join wait"))
            return s;
    }

    // phase 3: merge the two states of every row
    const unsigned grid = (unsigned)((rows + 3) / 4);
    const int of32 = out_dtype == PA_F32;
    cudaError_t e;
    if (q_dtype == PA_BF16)
        e = head_dim == 128
                ? pa::launch_pdl(prefix_merge_kernel<__nv_bfloat16, 128>, dim3(grid), dim3(128),
                                 0, st, out, of32, o_a, lse_a, o_b, lse_b, rows)
                : pa::launch_pdl(prefix_merge_kernel<__nv_bfloat16, 64>, dim3(grid), dim3(128),
                                 0, st, out, of32, o_a, lse_a, o_b, lse_b, rows);
    else
        e = head_dim == 128
                ? pa::launch_pdl(prefix_merge_kernel<__half, 128>, dim3(grid), dim3(128), 0, st,
                                 out, of32, o_a, lse_a, o_b, lse_b, rows)
                : pa::launch_pdl(prefix_merge_kernel<__half, 64>, dim3(grid), dim3(128), 0, st,
                                 out, of32, o_a, lse_a, o_b, lse_b, rows);
    return pa::cuda_status(e, "shared-prefix merge launch");
}
