/*
 * ra.h -- C ABI of the GB300 (sm_103a) RadixAttention hot path.
 *
 * RadixAttention keeps the KV cache of every token in a token-granular pool;
 * requests that share a prefix (a path of the radix tree) share the pool
 * slots of that prefix, so a new request only computes KV for its unmatched
 * suffix and attention reads the shared prefix from the pool (SGLang paper
 * summary, §3 "Efficient KV Cache Reuse with RadixAttention"; yaopepe.com
 * explainer of the same paper, §04, "reference the shared KV, prefill only the
 * unmatched suffix").  A request's slots are one row of the `req_to_token`
 * table, selected by `req_pool_indices`; each step's new tokens are written to
 * the slots in `out_cache_loc`; decode reads `seq_lens` (anrans handbook,
 * "v0.2：不到四千行的调度核心跑出 3.1 倍", 来源一: the CUDA-graph decode inputs).
 *
 * Common conventions
 *  - All pointers are DEVICE pointers on the current CUDA device unless noted.
 *  - Pools: K and V are bf16 arrays [num_slots, num_kv_heads, head_dim],
 *    row-major; one slot = one token.  head_dim must be 64 or 128.
 *  - GQA: q head h reads kv head h / (num_q_heads / num_kv_heads).
 *  - Index arrays are int32.  req_to_token is [table_rows, table_stride]
 *    row-major; entry (r, j) is the slot of position j of the request stored
 *    in row r.
 *  - Buffer alignment: pools, q, o, k_new, v_new and workspace must be
 *    16-byte aligned; index arrays 4-byte aligned.
 *  - Ownership: the caller owns every buffer.  The library never allocates,
 *    frees or synchronises; every call only enqueues kernels on `stream`, so
 *    calls can be captured in a CUDA graph.  Grids are sized from the host-side
 *    bounds (max_*), and kernels read the actual lengths from device memory.
 *  - Errors: host-side validation returns a status and never launches on
 *    failure; ra_last_error_message() gives a thread-local description.
 *    Device-side checks never trap: an out-of-range slot, table row or length
 *    is replaced by a safe value, the access is skipped, and, if
 *    `device_error` is non-NULL, the matching RA_DEVERR_* bit is OR-ed into
 *    that word (the caller zeroes it and reads it back when it wants).
 *  - Ordering: on one stream, call ra_kv_store for the step's new tokens and
 *    write their slots into req_to_token BEFORE the attention calls that read
 *    them.  Attention reads every key, cached prefix and new suffix alike,
 *    from the pool.
 */
#ifndef RA_H_
#define RA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* ra_stream_t;

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, misaligned buffer, Hq % Hkv != 0 ... */
  RA_ERR_UNSUPPORTED = 2,      /* a shape the kernels are not built for (head_dim, GQA group) */
  RA_ERR_WORKSPACE = 3,        /* workspace smaller than the matching *_workspace_bytes() */
  RA_ERR_CUDA = 4              /* a CUDA runtime call or kernel launch failed */
} ra_status;

/* Bits OR-ed into *device_error by the kernels. */
#define RA_DEVERR_SLOT 0x1u    /* a slot id outside [0, num_slots) was met (read as slot 0 / skipped) */
#define RA_DEVERR_TABLE 0x2u   /* a req_pool_indices entry outside [0, table_rows) */
#define RA_DEVERR_LENGTH 0x4u  /* a length outside its host-side bound, or a seq_len < 1 */
#define RA_DEVERR_TIMEOUT 0x8u /* a bounded wait inside a kernel gave up (the kernel returned early) */

/*
 * ra_kv_store -- write this step's new K/V rows into their pool slots.
 *   pool[out_cache_loc[i], :, :] = new[i, :, :] for K and V, i < num_tokens.
 * Source: anrans handbook "v0.2：不到四千行的调度核心跑出 3.1 倍", 来源一 (each
 * step's tokens get `out_cache_loc` slots; padded graph requests write the
 * dummy slot 0); the low-latency-mode page (aihot.news, "SGLang 发布
 * Low-Latency Mode", AMD 低延迟内核) lists the KV-cache write as a step of the
 * decoder layer.
 *   k_pool, v_pool: bf16 [num_slots, num_kv_heads, head_dim], written in place.
 *   k_new, v_new:   bf16 [num_tokens, num_kv_heads, head_dim].
 *   out_cache_loc:  int32 [num_tokens]; entries must be distinct except the
 *                   dummy slot 0 (whose final contents are then unspecified).
 * A bit copy: the result is bit-identical to the inputs.  num_tokens == 0 is a
 * no-op.  Out-of-range slots are skipped and flagged (RA_DEVERR_SLOT).
 */
ra_status ra_kv_store(void* k_pool, void* v_pool, int64_t num_slots, int32_t num_kv_heads, int32_t head_dim,
                      const void* k_new, const void* v_new, const int32_t* out_cache_loc, int64_t num_tokens,
                      uint32_t* device_error, ra_stream_t stream);

/*
 * ra_extend_attention -- prefill of new suffix tokens over a cached prefix.
 * For request b (row req_pool_indices[b] of the table), suffix token i <
 * extend_lens[b] is at position p = prefix_lens[b] + i and attends to the
 * keys at positions 0..p (the cached prefix and its own suffix up to itself):
 *   o[t, h, :] = sum_j softmax_j(sm_scale * <q[t, h], K[slot_j, h / G]>) V[slot_j, h / G]
 * with t = qo_indptr[b] + i and slot_j = req_to_token[req_pool_indices[b], j].
 * Source: SGLang paper summary, §3 (KV of a prefix depends only on its tokens,
 * so the cached prefix is reused); yaopepe.com explainer, §04 (longest prefix
 * match, the matched KV is referenced and only the unmatched suffix is
 * prefilled).
 *   q, o:            bf16 [total_q, num_q_heads, head_dim]; o must not alias q or the pools.
 *   qo_indptr:       int32 [batch + 1], qo_indptr[0] = 0, qo_indptr[batch] = total_q.
 *   prefix_lens, extend_lens: int32 [batch]; extend_lens[b] = qo_indptr[b+1] - qo_indptr[b].
 *   max_extend_len, max_prefix_len: host-side upper bounds of those arrays
 *                    (grid sizing); a device value above its bound is flagged
 *                    RA_DEVERR_LENGTH and the rows above the bound are skipped.
 *   workspace:       device scratch of at least ra_extend_workspace_bytes(batch,
 *                    total_q, num_q_heads, num_kv_heads) bytes, 16-byte aligned
 *                    (may be NULL when batch or total_q is 0); it holds the
 *                    work list of (request, query tile) pairs, ordered longest
 *                    key range first, that a one-CTA pass builds on the stream
 *                    before the attention kernel runs.  Smaller: RA_ERR_WORKSPACE.
 *                    The contents are scratch; calls that overlap on the GPU
 *                    need separate workspaces.
 * The suffix keys must already be stored (ra_kv_store) and listed in the table.
 * Rows with extend_lens[b] == 0 write nothing; prefix_lens[b] == 0 is plain
 * causal attention.  batch == 0 or total_q == 0 is a no-op.  A request with
 * prefix_lens[b] + extend_lens[b] > table_stride is flagged RA_DEVERR_LENGTH and
 * skipped, and so is a request whose rows qo_indptr[b] .. qo_indptr[b] +
 * extend_lens[b] - 1 do not lie inside [0, total_q): no row outside o is ever
 * written.  The sum of extend_lens must not exceed total_q (excess tiles are
 * flagged RA_DEVERR_LENGTH and skipped).
 * Runs on tcgen05 tensor cores with TMEM accumulators; K/V rows are gathered
 * from the pool into 128B-swizzled shared-memory tiles, the query tile comes
 * in by one TMA tile load.
 */
ra_status ra_extend_attention(const void* k_pool, const void* v_pool, int64_t num_slots, int32_t num_kv_heads,
                              int32_t head_dim, const void* q, void* o, int32_t num_q_heads, float sm_scale,
                              const int32_t* req_to_token, int64_t table_stride, int64_t table_rows,
                              const int32_t* req_pool_indices, const int32_t* prefix_lens,
                              const int32_t* extend_lens, const int32_t* qo_indptr, int32_t batch, int64_t total_q,
                              int32_t max_extend_len, int32_t max_prefix_len, void* workspace,
                              size_t workspace_bytes, uint32_t* device_error, ra_stream_t stream);

/* Workspace bytes ra_extend_attention needs (0 for invalid head counts). */
size_t ra_extend_workspace_bytes(int32_t batch, int64_t total_q, int32_t num_q_heads, int32_t num_kv_heads);

/*
 * ra_decode_attention -- one new query token per request over its context.
 * Request b (table row req_pool_indices[b]) has seq_lens[b] >= 1 tokens, the
 * new one included (its K/V already stored); its query attends to positions
 * 0..seq_lens[b]-1:
 *   o[b, h, :] = sum_j softmax_j(sm_scale * <q[b, h], K[slot_j, h / G]>) V[slot_j, h / G]
 * Source: anrans handbook "v0.2：不到四千行的调度核心跑出 3.1 倍", 来源一 (decode
 * step inputs req_pool_indices / seq_lens / out_cache_loc); SGLang paper
 * summary, §3 (shared prefixes are read from the shared cache).
 *   q, o:     bf16 [batch, num_q_heads, head_dim]; o must not alias q or the pools.
 *   seq_lens: int32 [batch]; max_seq_len is its host-side upper bound.
 * Key ranges are split across CTAs (split-KV) and merged with a log-sum-exp
 * combine pass; the partial results live in `workspace`.  The split is planned
 * on the device from the actual lengths: at most 456 equal items (>= 128 keys)
 * plus one shorter item per request, so the workspace is bounded by
 * (456 + batch) partial rows per q head whatever max_seq_len is.
 *
 * Optional prefix-grouped (cascade) read, num_groups > 0: group g lists
 * decode requests group_reqs[group_indptr[g] .. group_indptr[g+1]) whose table
 * entries at positions group_prefix_start[g] .. group_prefix_len[g]-1 are the
 * same slots (a node of the radix tree they all pass through).  Those keys are
 * read from HBM once per group and kv head for all members (the yaopepe.com
 * explainer, §04 figure: the shared prefix's KV is stored once and referenced
 * by every branch); each member then reads only its own positions from the
 * largest group_prefix_len of its groups to seq_lens[b]-1, and all partial
 * results are merged exactly.  The result equals the non-grouped call up to
 * floating-point rounding.
 *   Multi-level: a request may be in up to max_group_levels groups, one per
 *   level, group_level[g] in [0, max_group_levels); its groups' ranges must be
 *   disjoint and together cover positions 0 .. (largest group_prefix_len)-1
 *   (the nested nodes of one path from the root of the tree).
 *   group_prefix_start may be NULL (all 0) and group_level NULL (all 0: one
 *   group per request at most).
 *   Preconditions: 0 <= group_prefix_start[g] < group_prefix_len[g] <=
 *   seq_lens[b] for each member; the members' table rows agree on the range
 *   (it is read through the first member's row).  max_group_prefix_len (bound
 *   of group_prefix_len), max_group_size and max_group_levels are host-side
 *   bounds; a device value outside them is flagged and its group skipped.
 *   With num_groups == 0 the group pointers may be NULL.
 */
ra_status ra_decode_attention(const void* k_pool, const void* v_pool, int64_t num_slots, int32_t num_kv_heads,
                              int32_t head_dim, const void* q, void* o, int32_t num_q_heads, float sm_scale,
                              const int32_t* req_to_token, int64_t table_stride, int64_t table_rows,
                              const int32_t* req_pool_indices, const int32_t* seq_lens, int32_t batch,
                              int32_t max_seq_len, int32_t num_groups, const int32_t* group_indptr,
                              const int32_t* group_reqs, const int32_t* group_prefix_start,
                              const int32_t* group_prefix_len, const int32_t* group_level,
                              int32_t max_group_prefix_len, int32_t max_group_size, int32_t max_group_levels,
                              void* workspace,
                              size_t workspace_bytes, uint32_t* device_error, ra_stream_t stream);

/* Bytes of workspace ra_decode_attention needs for these host-side bounds
 * (same arguments as the call).  Depends on nothing else. */
size_t ra_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t max_seq_len, int32_t num_groups, int32_t max_group_prefix_len,
                                 int32_t max_group_size, int32_t max_group_levels);

/*
 * ra_decode_attention_store -- ra_kv_store of the decode step's new tokens and
 * ra_decode_attention in one call, the store fused into the call's first
 * kernel (one launch fewer per step).  A decode step writes one new token per
 * request at out_cache_loc and then attends over the context that includes it
 * (anrans handbook "v0.2：不到四千行的调度核心跑出 3.1 倍", 来源一: the decode
 * inputs req_pool_indices, seq_lens and out_cache_loc).
 *   k_new, v_new: bf16 [batch, num_kv_heads, head_dim], row b = request b's
 *     new token; out_cache_loc: int32 [batch], its slot.  The pool is written
 *     as by ra_kv_store(k_pool, v_pool, ..., k_new, v_new, out_cache_loc,
 *     batch, ...) (bit copy; a slot outside the pool is skipped and flagged
 *     RA_DEVERR_SLOT), before any key is read; the caller has already listed
 *     out_cache_loc[b] in req_to_token at position seq_lens[b] - 1 (or wherever
 *     its table says), exactly as for ra_kv_store followed by
 *     ra_decode_attention.
 *   Every other argument, the workspace size and the result are those of
 *   ra_decode_attention.  k_new / v_new 16-byte aligned, out_cache_loc 4-byte
 *   aligned; all three non-null.
 */
ra_status ra_decode_attention_store(void* k_pool, void* v_pool, int64_t num_slots, int32_t num_kv_heads,
                                    int32_t head_dim, const void* k_new, const void* v_new,
                                    const int32_t* out_cache_loc, const void* q, void* o, int32_t num_q_heads,
                                    float sm_scale, const int32_t* req_to_token, int64_t table_stride,
                                    int64_t table_rows, const int32_t* req_pool_indices, const int32_t* seq_lens,
                                    int32_t batch, int32_t max_seq_len, int32_t num_groups,
                                    const int32_t* group_indptr, const int32_t* group_reqs,
                                    const int32_t* group_prefix_start, const int32_t* group_prefix_len,
                                    const int32_t* group_level, int32_t max_group_prefix_len, int32_t max_group_size,
                                    int32_t max_group_levels, void* workspace, size_t workspace_bytes,
                                    uint32_t* device_error, ra_stream_t stream);

/*
 * ra_decode_attention_static -- ra_decode_attention for callers that cannot
 * allocate device memory.  The paper has no counterpart: this is an interface
 * addition for callers such as a plugin that runs under a host framework's
 * fixed memory plan and may not call cudaMalloc, or a runtime that has no
 * device allocator of its own.
 *   Same arguments and results as ra_decode_attention, without the workspace:
 *   the split-KV scratch lives in one file-scope device array of
 *   RA_DECODE_STATIC_SCRATCH_BYTES that every GPU loading this library holds
 *   until the process exits.  Nothing is allocated or freed by the call.
 *   A call whose ra_decode_workspace_bytes(...) exceeds that size returns
 *   RA_ERR_WORKSPACE with a message and launches nothing.
 *   The first call on a device (with that device current) looks up the array's
 *   device address; the address is kept for that device's current CUDA context
 *   and looked up again in a new context (after cudaDeviceReset, for
 *   instance).  Make the first call in each context outside any stream capture.
 *   All calls share the array and it keeps the last call's contents: calls
 *   that overlap on the GPU (other streams, unordered threads) race on it.
 */
#define RA_DECODE_STATIC_SCRATCH_BYTES (32u << 20)
ra_status ra_decode_attention_static(const void* k_pool, const void* v_pool, int64_t num_slots,
                                     int32_t num_kv_heads, int32_t head_dim, const void* q, void* o,
                                     int32_t num_q_heads, float sm_scale, const int32_t* req_to_token,
                                     int64_t table_stride, int64_t table_rows, const int32_t* req_pool_indices,
                                     const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                     int32_t num_groups, const int32_t* group_indptr, const int32_t* group_reqs,
                                     const int32_t* group_prefix_start, const int32_t* group_prefix_len,
                                     const int32_t* group_level, int32_t max_group_prefix_len,
                                     int32_t max_group_size, int32_t max_group_levels, uint32_t* device_error,
                                     ra_stream_t stream);

/*
 * ra_selftest_bounded_wait -- check, on the current device, that a wait inside a kernel that runs out
 * returns instead of hanging.  The pages have no counterpart: every wait in this library's kernels (on
 * an mbarrier or on a counter another CTA raises) is bounded by a clock deadline, after which the kernel
 * flags RA_DEVERR_TIMEOUT and leaves; this call runs one CTA that waits, with a deadline of
 * deadline_cycles SM clock cycles (1 .. 2^32), on an mbarrier no thread arrives at and on a counter no
 * thread raises.  Both waits run out: the kernel OR-s RA_DEVERR_TIMEOUT into *device_error (a device
 * word, 4-byte aligned, that the caller zeroes and reads back) and returns.  Enqueues one kernel on
 * `stream`; nothing else is touched.
 */
ra_status ra_selftest_bounded_wait(int64_t deadline_cycles, uint32_t* device_error, ra_stream_t stream);

/* Static description of a status code. */
const char* ra_status_string(ra_status status);

/* Thread-local description of the last failure of a call on this thread ("" if none). */
const char* ra_last_error_message(void);

/* ABI revision of this header (bumped on any signature change). */
int32_t ra_abi_version(void);

#define RA_ABI_VERSION 5

#ifdef __cplusplus
}
#endif

#endif /* RA_H_ */
