/*
 * pa.h -- C ABI of the paged KV-cache decode-attention library (libpa.so).
 *
 * Decode-phase attention over a KV cache split into fixed 16-token blocks
 * held in one physical pool and mapped per sequence by a block table.
 * Sources (page title, then section):
 *   [p1] "大模型推理优化全攻略" (zhengtianqi.github.io) §2.1 why a KV cache,
 *        §2.3 PagedAttention (16-token blocks, on-demand allocation)
 *   [p2] "LLM推理优化深度实战" (ybb.press) §2.1 PagedAttention, copy-on-write,
 *        best-of-N sharing; §2.2 GQA; §5.2 KV-cache quantisation
 *   [p3] "KV Cache ... PagedAttention" (devpress.csdn.net) §二 attention
 *        formula and KV memory formula; §七 block table and block manager
 *   [p4] "cs336 lecture 10" notes: KV Cache workflow (decode step), GQA/MQA,
 *        Quantization formula, speculative decoding (verify)
 *
 * Conventions for every call:
 *   - Every call returns a pa_status; no C++ exception crosses the ABI.
 *     On failure, pa_last_error() returns a message (thread-local, valid
 *     until the next call on the same thread).
 *   - Argument errors are detected on the host before any launch.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream). Launch failures return PA_ERR_CUDA; faults
 *     that happen later surface at the caller's next synchronisation.
 *   - The library allocates no device memory. Every device pointer is
 *     caller-owned memory; the caller keeps it alive until the work on
 *     `stream` has finished.
 *   - Contents of device arrays (block-table entries, lengths, slots) are the
 *     caller's contract. With the environment variable PA_VALIDATE=1 the
 *     device calls copy them to the host first (synchronising `stream`) and
 *     range-check them, returning PA_ERR_VALIDATION on a bad entry.
 *
 * Memory layout (this library's choice; the pages fix none):
 *   k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim],
 *                      element type kv_dtype (F16, BF16 or INT8 codes).
 *                      Each (block, kv head) tile is contiguous.
 *   k_scale, v_scale : INT8 only, fp32 [num_blocks][num_kv_heads][block_size]
 *   k_zp, v_zp       : INT8 only, int8 [num_blocks][num_kv_heads][block_size]
 *   slot             : phys_block * block_size + offset (int64); < 0 = skip
 *   block_tables     : int32 [num_seqs][max_blocks_per_seq]; entry b of row s
 *                      is the physical block holding tokens 16b .. 16b+15 of
 *                      sequence s ([p3] §七: logical block -> physical block)
 *   q, out           : [num_q_tokens][num_heads][head_dim], rows of sequence s
 *                      at query_start_loc[s] .. query_start_loc[s+1]-1
 *   GQA/MQA          : q head h reads kv head h / (num_heads / num_kv_heads)
 *                      ([p4] GQA: heads split into contiguous groups; MQA is
 *                      num_kv_heads == 1)
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* bad pointer, size, shape or id */
    PA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. block_size != 16) */
    PA_ERR_OUT_OF_BLOCKS = 3, /* the pool cannot cover an append; nothing changed */
    PA_ERR_BAD_REFCOUNT = 4,  /* refcount underflow (double free) */
    PA_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    PA_ERR_VALIDATION = 6,    /* PA_VALIDATE found a bad device-array entry */
    PA_ERR_DEVICE = 7         /* a kernel reported an error word (see pa_device_error) */
} pa_status;

/* PA_FP8_E4M3: 8-bit float codes (1 sign, 4 exponent bits with bias 7, 3
 * fraction bits, no infinities, largest finite 448) with one fp32 scale per
 * KV head ([p2] §5.2: FP8 KV cache with per-head scaling factors found on
 * calibration data); the value of a code is E4M3(code) * scale[head]. */
typedef enum pa_dtype {
    PA_F16 = 0, PA_BF16 = 1, PA_F32 = 2, PA_INT8 = 3, PA_FP8_E4M3 = 4
} pa_dtype;

/* Message for the last failing call on this thread ("" if none). */
const char* pa_last_error(void);
/* Library version string. */
const char* pa_version(void);

/* ======================================================================
 * Host block pool ([p3] §七 KVBlockManager; refcounts and copy-on-write per
 * [p2] §2.1). Owns host metadata only, never device memory. Not thread-safe:
 * one pool per thread, or external locking.
 * ==================================================================== */
typedef struct pa_pool pa_pool;

/* Create a pool of num_blocks physical blocks. The free list starts as
 * free_order[0..num_blocks-1] (a permutation of 0..num_blocks-1) or, if
 * free_order is NULL, as 0..num_blocks-1; blocks are taken from its END and
 * returned to its end ([p3]'s list(range(n)) / pop() / extend()).
 * block_size must be 16. */
pa_status pa_pool_create(int32_t num_blocks, int32_t block_size,
                         const int32_t* free_order, pa_pool** out);
void pa_pool_destroy(pa_pool* pool);

/* New empty sequence; ids are 0, 1, 2, ... in creation order, never reused. */
pa_status pa_seq_create(pa_pool* pool, int32_t* seq_id);

/* Child sharing every block of parent (refcount + 1 on each): best-of-N
 * parallel sampling shares the prompt's blocks ([p2] §2.1). */
pa_status pa_seq_fork(pa_pool* pool, int32_t parent, int32_t* child);

/* Reserve n_tokens new token slots at the end of sequence `seq` and write
 * their slots to slots_out[0..n_tokens-1]. A new block is taken exactly when
 * the token count reaches the capacity ([p3] append_token). If the tail
 * block is partly filled and shared (refcount > 1), it is copied first: a
 * fresh block replaces it in this sequence's table, the old block's refcount
 * drops by one, and the pair (old, fresh) is written to cow_pair_out[0..1]
 * with *n_cow = 1 (else *n_cow = 0). The copy block is taken before any new
 * tail block. The caller must run pa_copy_blocks on the returned pairs
 * before pa_append_kv writes the slots. All-or-nothing: on
 * PA_ERR_OUT_OF_BLOCKS nothing changes. */
pa_status pa_seq_append_slots(pa_pool* pool, int32_t seq, int32_t n_tokens,
                              int64_t* slots_out, int32_t* cow_pair_out,
                              int32_t* n_cow);

/* A decode step's reservations in one call: for i = 0 .. n-1 in order,
 * pa_seq_append_slots(seqs[i], n_tokens[i]), its slots written contiguously
 * to slots_out (sum of n_tokens entries) and its copy-on-write pair, if any,
 * appended to cow_pairs_out (int32 [n][2], may be NULL if no sequence needs
 * one) with the number of pairs in *n_cow. On an error the sequences before
 * the failing one keep their reservations (each reservation is itself
 * all-or-nothing) and *n_cow counts their pairs. */
pa_status pa_seq_append_slots_batch(pa_pool* pool, const int32_t* seqs,
                                    const int32_t* n_tokens, int32_t n,
                                    int64_t* slots_out, int32_t* cow_pairs_out,
                                    int32_t* n_cow);

/* Release a sequence: refcount - 1 on each block; blocks reaching 0 go back
 * to the end of the free list in table order ([p3] release). */
pa_status pa_seq_free(pa_pool* pool, int32_t seq);

/* Number of tokens held by a sequence. */
pa_status pa_seq_len(pa_pool* pool, int32_t seq, int32_t* len);

/* Block tables of n sequences into tables_out[n][max_blocks] (entries past a
 * sequence's blocks are -1) and their lengths into lens_out[n] (may be NULL).
 * PA_ERR_INVALID_ARG if a sequence holds more than max_blocks blocks. */
pa_status pa_pool_block_tables(pa_pool* pool, const int32_t* seqs, int32_t n,
                               int32_t max_blocks, int32_t* tables_out,
                               int32_t* lens_out);

/* free = blocks on the free list, used = refcount > 0, shared = refcount > 1
 * (KV-cache utilisation, [p2] §7.3). Any output pointer may be NULL. */
pa_status pa_pool_stats(pa_pool* pool, int32_t* free_blocks, int32_t* used,
                        int32_t* shared);

/* Reference count of one physical block. */
pa_status pa_pool_refcount(pa_pool* pool, int32_t block, int32_t* ref);

/* ---- Prefix cache ([p1] §2.4: requests sharing a prefix reuse its KV,
 * found by a hash of the prefix tokens, least recently used entries evicted;
 * [p3]: hash(prefix_tokens) -> KV blocks). Per whole block: a full block is
 * named by the complete token prefix that ends with it (looked up by a hash
 * of (prefix of the previous block, this block's 16 token ids) and then
 * compared token by token, so equal names mean equal prefixes). Off until
 * enabled; the calls above behave exactly as before while it is off. ---- */

/* Turn the prefix cache on (or change its size): up to max_cached_blocks
 * registered blocks that no sequence holds are kept for reuse, oldest
 * released first out. Allocation uses the free list first and evicts the
 * oldest cached block only when the free list is empty; pa_pool_stats'
 * free count does not include cached blocks. */
pa_status pa_pool_enable_prefix_cache(pa_pool* pool, int32_t max_cached_blocks);

/* A new sequence that starts with the longest chain of cached whole blocks
 * matching token_ids[0 .. n_tokens) -- at most (n_tokens - 1) / 16 blocks, so
 * at least one token is left to compute. *n_cached_out = tokens covered (a
 * multiple of 16): the sequence holds them (refcounts raised) and its length
 * is that; append the rest with pa_seq_append_tokens and write their K/V. */
pa_status pa_seq_create_with_prefix(pa_pool* pool, const int32_t* token_ids,
                                    int32_t n_tokens, int32_t* seq_out,
                                    int32_t* n_cached_out);

/* pa_seq_append_slots for tokens whose ids are known: every block the append
 * fills is registered under its prefix (unless a block already holds that
 * prefix), so later requests can reuse it. A sequence that ever took a plain
 * pa_seq_append_slots registers nothing after that. Requires the prefix
 * cache to be enabled. */
pa_status pa_seq_append_tokens(pa_pool* pool, int32_t seq, const int32_t* token_ids,
                               int32_t n_tokens, int64_t* slots_out,
                               int32_t* cow_pair_out, int32_t* n_cow);

/* cached_free = registered blocks no sequence holds (the LRU list),
 * registered = blocks registered under a prefix, hit_blocks / lookup_blocks
 * = blocks found / looked up by pa_seq_create_with_prefix. Any output may be
 * NULL. */
pa_status pa_pool_prefix_stats(pa_pool* pool, int32_t* cached_free, int32_t* registered,
                               int64_t* hit_blocks, int64_t* lookup_blocks);

/* Fork groups for pa_decode_shared_prefix ([p2] §2.1: best-of-N forks share
 * the prompt's blocks by reference count). Walks seqs[0..n) in order; a run
 * of adjacent sequences whose first physical block is the same forms one
 * group. prefix_len_out[g] is the number of leading tokens that every member
 * holds in the same physical blocks and that come before every member's
 * first query: whole 16-token blocks only, at most (L - r + 1) / 16 blocks
 * for a member with L tokens and a query run of r (q_lens[i], or 1 when
 * q_lens is NULL). A group of one sequence gets prefix 0.
 *   group_start_out  host int32 [n + 1]: group g is seqs[group_start[g] ..
 *                    group_start[g + 1])
 *   prefix_len_out   host int32 [n]
 *   num_groups_out   number of groups written
 * PA_ERR_INVALID_ARG for an unknown sequence or a query run outside
 * [1, L]. Forks that are not adjacent in seqs land in different groups. */
pa_status pa_pool_prefix_groups(pa_pool* pool, const int32_t* seqs, int32_t n,
                                const int32_t* q_lens, int32_t* group_start_out,
                                int32_t* prefix_len_out, int32_t* num_groups_out);

/* ======================================================================
 * Device operations. Pointers are device memory unless stated.
 * ==================================================================== */

/* Copy-on-write block copies ([p2] §2.1: copy a shared block only when it
 * is modified). For each i < n_pairs, copies physical block d_pairs[2i] to
 * d_pairs[2i+1] in k_cache and v_cache and, for INT8, in k_scale, v_scale,
 * k_zp, v_zp (pass NULL for those otherwise). d_pairs: device int32
 * [n_pairs][2]. Sources and destinations must be distinct blocks, and no
 * destination may also be a source. n_pairs == 0 is a no-op. */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, void* k_scale,
                         void* v_scale, void* k_zp, void* v_zp,
                         const int32_t* d_pairs, int32_t n_pairs,
                         int32_t num_blocks, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size,
                         pa_dtype kv_dtype, void* stream);

/* Append the new tokens' K and V to the cache through slot_mapping ([p4]
 * decode workflow: append the new K, V to the KV cache; [p3] §二 K_cache =
 * [K1 .. Kt]). key, value: [num_tokens][num_kv_heads][head_dim] of
 * src_dtype (F16 or BF16). For kv_dtype F16/BF16 (== src_dtype) the rows are
 * copied bit for bit. For kv_dtype INT8 each (token, kv head) row is
 * quantised ([p4] Quantization, x_q = round(x/scale) + zero_point): with
 * mn = min(row, 0), mx = max(row, 0) in fp32, scale = (mx - mn)/255 (1 if
 * 0), zp = clamp(-128 - rint(mn/scale)), code = clamp(rint(x/scale) + zp),
 * IEEE fp32 division and round-half-to-even; scale and zp are stored per
 * (token, kv head) ([p2] §5.2: per-head rather than global scales).
 * For kv_dtype FP8_E4M3, k_scale / v_scale are the caller's per-head scales,
 * fp32 [num_kv_heads] (read only; k_zp, v_zp unused): code =
 * E4M3(x / scale[head]) with the IEEE fp32 quotient rounded to the nearest
 * E4M3 value, ties to even, magnitudes past 448 saturating to +-448.
 * slot_mapping: device int64 [num_tokens]; a negative slot skips the token. */
pa_status pa_append_kv(const void* key, const void* value, pa_dtype src_dtype,
                       void* k_cache, void* v_cache, pa_dtype kv_dtype,
                       float* k_scale, float* v_scale, int8_t* k_zp,
                       int8_t* v_zp, const int64_t* slot_mapping,
                       int32_t num_tokens, int32_t num_blocks,
                       int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size, void* stream);

/* Bytes of workspace pa_decode needs for these sizes (0 if none). With
 * partition_size 0 (the balanced schedule) this is 24576 bytes of arrival
 * counters, the per-sequence prefix sums (4 x (num_seqs + 1) bytes rounded
 * up to 256) and 2 x min(2048, num_seqs x num_kv_heads x
 * ceil(max_context_len/16)) partial slots of 32 + 4 x R x (head_dim + 2)
 * bytes (rounded up to 16), R = (num_heads / num_kv_heads) x max_q_len
 * (at least 64 rows once R > 16); with partition_size > 0 see pa_decode.
 * Returns 0 for invalid sizes. Host-only: needs no GPU. */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_tokens,
                                int32_t num_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t max_q_len,
                                int32_t max_context_len, int32_t partition_size);

/* Decode attention ([p3] §二 softmax(Q K^T / sqrt(d)) V over the cached
 * keys; [p4] decode workflow: score the new token's q against every cached
 * K and take the weighted sum of the cached V).
 *   out            [num_q_tokens][num_heads][head_dim], out_dtype F32 or
 *                  the q dtype
 *   q              [num_q_tokens][num_heads][head_dim], q_dtype F16/BF16;
 *                  for F16/BF16 caches q_dtype must equal kv_dtype
 *   context_lens   int32 [num_seqs]: tokens in each sequence INCLUDING the
 *                  ones appended this step (append runs before attention)
 *   query_start_loc int32 [num_seqs + 1] or NULL (then one query token per
 *                  sequence and num_q_tokens == num_seqs). A run of r query
 *                  tokens (speculative verify, [p4]: the target model checks
 *                  the draft tokens in one pass) puts query i at position
 *                  L - r + i; it sees keys 0 .. L - r + i (causal).
 *   max_q_len      the largest r (1 when query_start_loc is NULL)
 *   max_context_len the largest context length (host value)
 *   scale          softmax scale, usually 1/sqrt(head_dim)
 *   partition_size 0 (default) selects the balanced schedule: a persistent
 *                  grid in which every warp streams an equal contiguous share
 *                  of all (sequence, KV head, block) work; a share that
 *                  covers a (sequence, KV head) whole writes its output, and
 *                  where share boundaries cut one, the pieces' partials
 *                  (m, l, O) are merged with the log-sum-exp rule (by the
 *                  decode kernel itself for F16/BF16 caches with at most 16
 *                  query rows per KV head, else by a reduce kernel). An INT8
 *                  call at head_dim 128 averaging at least 64 query rows per
 *                  KV head (num_heads / num_kv_heads x num_q_tokens /
 *                  num_seqs) with at most 1536 sequences runs on the tensor
 *                  cores with one share per SM, shares cut by cost; its
 *                  partial slots hold 96 rows, and it uses as many SMs as the
 *                  workspace size above has room for. A multiple
 *                  of 16 up to 4096 selects fixed split-KV partitions of that
 *                  many tokens (one CTA per partition, KV head and sequence).
 *   workspace      device memory of pa_decode_workspace_size() bytes,
 *                  256-byte aligned (NULL allowed if that size is 0). Its
 *                  first 24576 bytes are 6144 uint32 arrival counters: they
 *                  must be ZERO before the first call that uses the buffer
 *                  (cudaMemset once, at allocation), and every call leaves
 *                  them zero, so one buffer serves any sequence of calls of
 *                  any sizes on one stream. With partition_size 0 the
 *                  decode kernel counts the blocks of each cut (sequence,
 *                  KV head) as its pieces finish, and the piece that
 *                  completes the count merges them. A counter that a call
 *                  finds above its total sets PA_DEVERR_WORKSPACE in the
 *                  device error word; a stale count below the total is not
 *                  always detected (it can make a merge run before all of
 *                  its pieces are written). So after a call whose device
 *                  error word is non-zero (a bounded wait gave up and left
 *                  counts short), zero the counters again before the next
 *                  call. The rest needs no initialisation. Layout after the counters with
 *                  partition_size > 0 and P = ceil(max_context_len /
 *                  partition_size):
 *                    o_part fp32 [num_q_tokens][num_heads][P][head_dim]
 *                           (each partition's normalised output)
 *                    m_part fp32 [num_q_tokens][num_heads][P] (base-2 log
 *                           domain: max of logit * log2(e))
 *                    l_part fp32 [num_q_tokens][num_heads][P]
 *                  each region starting on a 256-byte boundary. With
 *                  partition_size 0: partial slots, each int32 {sequence,
 *                  kv head, first token, end token} then fp32 m[R], l[R]
 *                  (base-2 units) and O[R][head_dim] (not normalised).
 * Requirements: head_dim 64 or 128, block_size 16, num_heads a multiple of
 * num_kv_heads, context_lens[s] >= (query run length of s) >= 1, at most
 * 8192 sequences per call with partition_size 0. */
pa_status pa_decode(void* out, pa_dtype out_dtype, const void* q,
                    pa_dtype q_dtype, const void* k_cache, const void* v_cache,
                    pa_dtype kv_dtype, const float* k_scale,
                    const float* v_scale, const int8_t* k_zp,
                    const int8_t* v_zp, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                    const int32_t* query_start_loc, int32_t num_seqs,
                    int32_t num_q_tokens, int32_t max_q_len,
                    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t block_size, int32_t num_blocks, float scale,
                    int32_t max_context_len, int32_t partition_size,
                    void* workspace, size_t workspace_bytes, void* stream);

/* pa_decode without caller-provided workspace: the split-KV scratch is a
 * built-in 40 MiB device array inside this library. The pages have no
 * counterpart to this call; it exists for callers that cannot allocate
 * device memory themselves -- for example code embedded in a host
 * application whose own allocator owns all device memory (a stray
 * cudaMalloc would escape its accounting or fail under its memory cap), or
 * a latency-critical decode loop that must not call cudaMalloc/cudaFree,
 * which can synchronise the device.
 *   - Arguments and results are exactly those of pa_decode, minus
 *     workspace/workspace_bytes. The caller still passes (and owns) every
 *     input and output buffer.
 *   - If pa_decode_workspace_size() for these arguments exceeds 40 MiB
 *     (41943040 bytes) the call returns PA_ERR_UNSUPPORTED and launches
 *     nothing. 40 MiB covers every call with at most 16 query rows per KV
 *     head (q heads per KV head x max_q_len), at any batch size; calls with
 *     more rows may need a larger partition_size, or pa_decode.
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating
 *     library routine. Every GPU that loads the library holds the 40 MiB
 *     array until the process exits.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture. The cached address is not
 *     valid after cudaDeviceReset: do not use this call across a reset.
 *   - Every call first clears the array's arrival counters with a
 *     cudaMemsetAsync on `stream` (no allocation), so a call that gave up
 *     (non-zero device error word) leaves no stale count for the next one.
 *   - All calls share the one array and it keeps the last call's contents;
 *     calls whose work overlaps on the GPU (different streams, or different
 *     host threads) race on it and must be serialised. */
pa_status pa_decode_no_alloc(void* out, pa_dtype out_dtype, const void* q,
                             pa_dtype q_dtype, const void* k_cache,
                             const void* v_cache, pa_dtype kv_dtype,
                             const float* k_scale, const float* v_scale,
                             const int8_t* k_zp, const int8_t* v_zp,
                             const int32_t* block_tables,
                             int32_t max_blocks_per_seq,
                             const int32_t* context_lens,
                             const int32_t* query_start_loc, int32_t num_seqs,
                             int32_t num_q_tokens, int32_t max_q_len,
                             int32_t num_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size,
                             int32_t num_blocks, float scale,
                             int32_t max_context_len, int32_t partition_size,
                             void* stream);

/* Workspace bytes of pa_decode_shared_prefix for these sizes (0 for invalid
 * sizes). */
size_t pa_decode_shared_prefix_workspace_size(
    int32_t num_seqs, int32_t num_q_tokens, int32_t num_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t max_q_len,
    int32_t max_context_len, int32_t num_groups, int32_t max_group_q_len,
    int32_t max_prefix_len, int32_t max_blocks_per_seq);

/* Decode attention with read-once shared prefixes (copy-on-write forks,
 * [p2] §2.1). The result is that of pa_decode with partition_size 0 on the
 * same arguments (16-bit caches only); the difference is that the blocks a
 * group of forks shares are read once per group and KV head instead of once
 * per fork:
 *   1. each group's first prefix_len[g] tokens are attended by all of the
 *      group's query rows together (no causal mask is needed: every prefix
 *      token precedes every query of the group),
 *   2. every sequence attends its own tokens [prefix_len, L) with the usual
 *      causal offset for query runs,
 *   3. each output row merges the two results by their log-sum-exp (the
 *      rule of the split-KV reduce).
 *   group_start   device int32 [num_groups + 1]: group g is sequences
 *                 group_start[g] .. group_start[g + 1] - 1; groups cover
 *                 0 .. num_seqs in order, none empty
 *   prefix_len    device int32 [num_groups]: a multiple of 16, at most
 *                 max_prefix_len and at most L - r + 1 for every member;
 *                 every member's block table holds the same physical ids
 *                 for the first prefix_len / 16 blocks (pa_pool_prefix_groups
 *                 computes both arrays). 0 means no shared prefix.
 *   max_group_q_len host: the largest number of query tokens in one group
 *   max_prefix_len  host: the largest prefix_len
 *   workspace     pa_decode_shared_prefix_workspace_size() bytes, 256-byte
 *                 aligned. Its first 24576 bytes are arrival counters with
 *                 pa_decode's rule: zero before the first call, left zero
 *                 by every call; the rest needs no initialisation.
 * Other arguments as pa_decode. Under PA_VALIDATE=1 the group arrays are
 * also checked against the block tables (PA_ERR_VALIDATION). INT8 caches
 * return PA_ERR_UNSUPPORTED. */
pa_status pa_decode_shared_prefix(
    void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype,
    const void* k_cache, const void* v_cache, pa_dtype kv_dtype,
    const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, const int32_t* query_start_loc,
    int32_t num_seqs, int32_t num_q_tokens, int32_t max_q_len,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int32_t num_blocks, float scale,
    int32_t max_context_len, const int32_t* group_start,
    const int32_t* prefix_len, int32_t num_groups, int32_t max_group_q_len,
    int32_t max_prefix_len, void* workspace, size_t workspace_bytes,
    void* stream);

/* Device error word bits. */
#define PA_DEVERR_WAIT_FULL  (1u << 0) /* a consumer gave up waiting for a staged tile */
#define PA_DEVERR_WAIT_EMPTY (1u << 1) /* a producer gave up waiting for a free stage */
#define PA_DEVERR_WAIT_DRAIN (1u << 2) /* the exit drain gave up on an in-flight copy */
#define PA_DEVERR_BAD_BLOCK  (1u << 3) /* a block-table entry outside the pool */
#define PA_DEVERR_BAD_SLOT   (1u << 4) /* a slot_mapping entry outside the pool */
#define PA_DEVERR_BAD_GROUP  (1u << 5) /* a shared-prefix group range or prefix length */
#define PA_DEVERR_WORKSPACE  (1u << 6) /* a workspace arrival counter was not zero */

/* Read and clear the device error word that kernels set instead of
 * trapping (a bounded wait that gave up, an index a kernel refused).
 * Synchronises `stream`. *code = 0 when no error was recorded; returns
 * PA_ERR_DEVICE when *code != 0. */
pa_status pa_device_error(void* stream, uint32_t* code);

#ifdef __cplusplus
}
#endif
#endif /* PA_H_ */
