/*
 * pkv.h — C ABI of the paged GQA decode-attention library (sm_103a, GB300).
 *
 * The problem these calls solve is stated in "Agent-Infer: 纯 Rust 编写的高性能 LLM
 * 推理引擎", section "分页 KV 缓存" (paged KV cache): the KV cache is a token pool
 * with page size 1 (SGLang's TokenToKVPool), one decode step is batched across all
 * requests, the attention work plan is built once per step rather than once per
 * layer, and its buffers are preallocated (same page, section "优化历程", stages 2
 * and 3). Grouped-query attention with 32 query heads on 8 KV heads at head_dim
 * 128, and head_dim 256 for the hybrid model's full-attention layers, come from
 * "Pegainfer: 纯Rust+CUDA构建的LLM推理引擎", sections "1. 注意力机制优化" and
 * "2. Qwen3.5的混合架构支持".
 *
 * Conventions for every call:
 *  - Pointers are plain device addresses unless a parameter name ends in _host.
 *    The caller owns every buffer it passes; no call keeps a pointer after it
 *    returns, except that the device work (kernels, copies) it enqueued on
 *    `stream` reads and writes them until that work completes.
 *  - bf16 means IEEE bfloat16 bit patterns (2 bytes, little endian).
 *  - Layouts are dense row-major:
 *      pool  (K or V): [pool_slots, n_kv_heads, head_dim] bf16 — one pool row per
 *                      token slot; one (slot, head) row is head_dim*2 bytes
 *      q, out        : [batch, n_qo_heads, head_dim] bf16
 *      lse           : [batch, n_qo_heads] fp32
 *      kv_indptr     : [batch + 1] int32, kv_indptr[0] = 0, non-decreasing
 *      kv_indices    : [kv_indptr[batch]] int32 pool slots; request b attends over
 *                      kv_indices[kv_indptr[b] .. kv_indptr[b+1]) in that order
 *    Query head h reads KV head h / (n_qo_heads / n_kv_heads).
 *  - Device pointers to q, pools, new rows and out must be 16-byte aligned.
 *  - Every call returns PKV_OK (0) or a negative PKV_ERR_* code, and checks its
 *    arguments on the host before anything is enqueued; on an error nothing is
 *    enqueued. pkv_last_error() then describes the failure (per thread).
 *  - No call synchronises the stream or allocates device memory, except
 *    paged_decode_plan_create / _destroy and the optional debug checks
 *    (pkv_set_debug_checks), which copy index arrays to the host synchronously.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *  - Supported shapes: head_dim 128 or 256; n_qo_heads a multiple of n_kv_heads
 *    with group size G = n_qo_heads / n_kv_heads in {1, 2, 4, 8};
 *    1 <= n_kv_heads <= 8.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pkv_stream_t; /* same type as cudaStream_t */
typedef struct pkv_plan pkv_plan;          /* opaque, owned by the library */

enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1, /* null pointer, negative size, misalignment, bad CSR */
    PKV_ERR_UNSUPPORTED = -2, /* head_dim / group size / head count not supported */
    PKV_ERR_PLAN = -3,        /* plan missing, too small, or built for other shapes */
    PKV_ERR_CUDA = -4,        /* a CUDA runtime call or kernel launch failed */
    PKV_ERR_INDEX = -5        /* debug checks: slot id out of range / indptr mismatch */
};

/*
 * kvpool_append — write this step's new K/V rows into their pool slots.
 *   k_pool[slot_ids[i], :, :] = k_new[i, :, :]  and  v_pool[...] = v_new[i, :, :]
 * for i < n. This is the scatter that fills the page-size-1 token pool each decode
 * step ("Agent-Infer", section "分页 KV 缓存"; the step's scatter is named in
 * section "优化历程", stage 7).
 *   k_pool, v_pool : [pool_slots, n_kv_heads, head_dim] bf16, written in place
 *   slot_ids       : [n] int32 device array; ids must be distinct and in
 *                    [0, pool_slots) — duplicates leave the row undefined; an
 *                    out-of-range id is reported (PKV_ERR_INDEX) only when debug
 *                    checks are on
 *   k_new, v_new   : [n, n_kv_heads, head_dim] bf16
 *   n              : number of rows (0 is a no-op)
 * The copy is bit-exact. Enqueued on `stream`; returns without waiting.
 */
int kvpool_append(void* k_pool, void* v_pool, const int32_t* slot_ids, const void* k_new,
                  const void* v_new, int64_t n, int n_kv_heads, int head_dim,
                  int64_t pool_slots, pkv_stream_t stream);

/*
 * kvpool_offload / kvpool_prefetch — the host KV tier: move pool rows between HBM
 * and pinned host memory. When HBM is full, older KV rows move to CPU memory and are
 * prefetched back when a request needs them again ("Agent-Infer", section "CPU 卸载").
 *   offload : k_host[host_slots[i]] = k_pool[dev_slots[i]]   (and V), i < n
 *   prefetch: k_pool[dev_slots[i]]  = k_host[host_slots[i]]  (and V)
 *   k_pool, v_pool : [pool_slots, n_kv_heads, head_dim] bf16 device pools
 *   k_host, v_host : [host_slots_cap, n_kv_heads, head_dim] bf16 in PINNED host memory
 *                    (cudaHostAlloc / a pinned torch tensor), read and written by the
 *                    GPU directly (NVLink-C2C on GB300); pageable memory is rejected
 *                    with PKV_ERR_INVALID_ARG before any launch
 *   dev_slots, host_slots : [n] int32 device arrays; destinations must be distinct
 *                    (checked, with ranges, only when debug checks are on)
 * Bit-exact copies; enqueued on `stream` (a side stream lets them overlap attention of
 * other layers). The caller points the requests' kv_indices at the prefetched slots.
 */
int kvpool_offload(const void* k_pool, const void* v_pool, const int32_t* dev_slots, void* k_host,
                   void* v_host, const int32_t* host_slots, int64_t n, int n_kv_heads,
                   int head_dim, int64_t pool_slots, int64_t host_slots_cap, pkv_stream_t stream);
int kvpool_prefetch(void* k_pool, void* v_pool, const int32_t* dev_slots, const void* k_host,
                    const void* v_host, const int32_t* host_slots, int64_t n, int n_kv_heads,
                    int head_dim, int64_t pool_slots, int64_t host_slots_cap, pkv_stream_t stream);

/*
 * paged_decode_plan_create — allocate a reusable plan for one model shape.
 * Sizes every buffer once (pinned host staging, device work list, split
 * workspace) so that no decode step allocates ("Agent-Infer", section "优化历程",
 * stage 2: preallocated buffers).
 *   *plan      : receives the new plan
 *   max_batch  : largest batch any step will use (>= 1)
 *   max_tokens : largest kv_indptr[batch] any step will use (>= 0)
 *   n_qo_heads, n_kv_heads, head_dim : the attention shape the plan serves
 * Uses the current CUDA device; the plan must be used on that device: every call that
 * takes the plan returns PKV_ERR_INVALID_ARG when another device is current.
 * Synchronous. Returns PKV_ERR_UNSUPPORTED for shapes outside the supported set.
 *
 * Small plans (max_batch x KV-head groups within the thread-block clusters the
 * device holds at once, and max_tokens at most 16 x 8 pipeline stages, 2048 tokens
 * at head_dim 128 with 8 KV heads; or, where only clusters of 8 (4) all fit, at most
 * 8 (4) x 8 stages) run their steps in single-launch mode, the
 * latency-bound decode of one or a few requests: paged_decode_plan uploads
 * nothing, and each attention call is one launch of a cluster kernel in which 16
 * (or 8, or 4) CTAs split each (request, head group), read kv_indptr on the device,
 * and merge their parts through distributed shared memory. In this mode each attention
 * launch carries the step's batch: a CUDA graph of attention calls is valid only
 * for steps with the batch it was captured with (PKV_PLAN_PERSISTENT keeps the
 * persistent grid, whose graphs serve any batch). paged_decode_plan_mode reports
 * the mode.
 */
int paged_decode_plan_create(pkv_plan** plan, int max_batch, int64_t max_tokens,
                             int n_qo_heads, int n_kv_heads, int head_dim);

/*
 * paged_decode_plan — build this step's work partition, once per decode step.
 * ("Agent-Infer", section "分页 KV 缓存": the plan runs once per step, not once per
 * layer; section "优化历程", stage 3.) Splits long contexts into chunks so that
 * skewed batches fill every SM, and records which requests need a log-sum-exp
 * merge. The persistent CTAs get contiguous ranges of the step's (request, head
 * group) runs, balanced in the kernel's pipeline stages plus a fixed cost per
 * piece: the smallest budget that the greedy fill fits into the grid, so the
 * slowest CTA is as short as that cost model allows. The result is copied to the device asynchronously on `stream` from the
 * plan's pinned staging; every paged_decode_attn call of the step with this
 * batch reuses it.
 *   kv_indptr_host : [batch + 1] int32 HOST array, the same values as the device
 *                    kv_indptr later passed to paged_decode_attn
 *   batch          : 0 <= batch <= max_batch; kv_indptr_host[batch] <= max_tokens
 * The plan has two pinned staging buffers and fills them in turn, so before
 * filling one the call waits (host side) only for the upload of the step before
 * the previous one: the host may run up to two steps ahead of the GPU without
 * blocking here. Use the same stream (or order the streams) for the plan and the
 * attention calls of a step.
 */
int paged_decode_plan(pkv_plan* plan, const int32_t* kv_indptr_host, int batch,
                      pkv_stream_t stream);

/*
 * paged_decode_plan_shared — paged_decode_plan for a step in which runs of
 * consecutive requests list the same first slots (a shared prompt prefix, as the
 * prefix cache of "Agent-Infer", section "前缀缓存", produces). Requests
 * [shared_indptr_host[s], shared_indptr_host[s+1]) all list the same
 * shared_len_host[s] slot ids first, s < n_shared; the runs are disjoint and in
 * batch order, and every member lists more slots than its shared prefix (its
 * newest token is private). The attention kernel then reads each shared slot once
 * for up to 16 / G requests at a time (16 query rows per KV head) instead
 * of once per request, and merges each member's prefix and suffix parts by
 * log-sum-exp.
 * PRECONDITION: the members of a run list identical slot ids in their first
 * shared_len_host[s] entries of kv_indices. The kernel reads the shared slots from
 * the first member's list on behalf of all members, so a description that is not
 * true of kv_indices gives wrong results for the other members. With debug checks
 * on (pkv_set_debug_checks), the attention calls that use the plan verify it on
 * the host and return PKV_ERR_INDEX, launching nothing, when it does not hold.
 * When it holds, results are those of paged_decode_plan (up to fp32 rounding).
 * For shapes without a shared-prefix kernel (only head_dim 128 with 4 KV heads
 * per group has one) the description is not used. Otherwise as paged_decode_plan.
 */
int paged_decode_plan_shared(pkv_plan* plan, const int32_t* kv_indptr_host, int batch,
                             const int32_t* shared_indptr_host, int n_shared,
                             const int32_t* shared_len_host, pkv_stream_t stream);

/*
 * paged_decode_attn — batched decode attention over the token pool, once per layer.
 * For every request b and query head h, with g = h / (n_qo_heads / n_kv_heads) and
 * idx = kv_indices[kv_indptr[b] .. kv_indptr[b+1]):
 *   s_j      = sm_scale * dot(q[b,h,:], K[idx_j, g, :])
 *   lse[b,h] = ln sum_j exp(s_j)                      (natural log, scale included)
 *   out[b,h] = sum_j exp(s_j - lse[b,h]) * V[idx_j, g, :]
 * computed with fp32 accumulation and an online softmax; long contexts are split
 * into chunks whose partial results are merged by log-sum-exp. An empty context
 * gives out = 0 and lse = -inf.
 *   q          : [batch, n_qo_heads, head_dim] bf16
 *   k_pool, v_pool : [pool_slots, n_kv_heads, head_dim] bf16 (read only)
 *   kv_indptr  : [batch + 1] int32 device array (must equal the plan's host copy)
 *   kv_indices : int32 device array of pool slots (must be valid slots)
 *   sm_scale   : the softmax scale (e.g. 1/sqrt(head_dim)), finite
 *   out        : [batch, n_qo_heads, head_dim] bf16, written (round to nearest even)
 *   lse        : [batch, n_qo_heads] fp32, written; may be NULL
 *   plan       : built by paged_decode_plan for this step with the same batch and
 *                created for the same (n_qo_heads, n_kv_heads, head_dim)
 * Launches the split-KV kernel and then the LSE-merge kernel (the latter exits at
 * once when no context was split); a plan in single-launch mode (small plans, see
 * paged_decode_plan_create) launches one cluster kernel instead. A plan serves one
 * stream at a time.
 */
int paged_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* kv_indptr, const int32_t* kv_indices, int batch,
                      int n_qo_heads, int n_kv_heads, int head_dim, float sm_scale,
                      void* out, float* lse, const pkv_plan* plan, pkv_stream_t stream);

/*
 * paged_decode_attn_tiered — paged_decode_attn over a slot list whose older rows may
 * sit in the host KV tier. When HBM is full, old KV rows move to CPU memory
 * ("Agent-Infer", section "CPU 卸载"); kvpool_prefetch brings them back before a
 * step, while this call reads them where they are: a slot id s >= 0 names row s of
 * k_pool / v_pool, and s < 0 names row -1 - s of k_host / v_host, which the kernel
 * reads over NVLink-C2C (16-byte copies into the same shared-memory stages as the
 * device rows). Results are those of paged_decode_attn over the same rows.
 *   pool_slots   : rows of k_pool / v_pool
 *   k_host, v_host : [host_slots, n_kv_heads, head_dim] bf16 in PINNED host memory
 *                  mapped for the GPU (cudaHostAlloc, a pinned torch tensor); pageable
 *                  memory is rejected with PKV_ERR_INVALID_ARG before any launch
 *   host_slots   : rows of each host pool (> 0)
 *   kv_indices   : entries in [-host_slots, pool_slots) (checked, with debug checks
 *                  on, as PKV_ERR_INDEX)
 * Other arguments as for paged_decode_attn. Host rows move at the link's rate (about
 * 200 GB/s on GB300), some thirty times slower than HBM, so a step spends time in
 * proportion to its host rows; the plan, built from kv_indptr alone, balances the
 * CTAs as if every row were in HBM.
 */
int paged_decode_attn_tiered(const void* q, const void* k_pool, const void* v_pool,
                             int64_t pool_slots, const void* k_host, const void* v_host,
                             int64_t host_slots, const int32_t* kv_indptr,
                             const int32_t* kv_indices, int batch, int n_qo_heads,
                             int n_kv_heads, int head_dim, float sm_scale, void* out,
                             float* lse, const pkv_plan* plan, pkv_stream_t stream);

/*
 * paged_decode_append_attn — kvpool_append followed by paged_decode_attn, in one
 * launch (plus the merge kernel): each request's newest K/V row is read straight
 * from k_new / v_new by the attention kernel, which also writes it to its pool
 * slot, so the step needs no separate append kernel. The pages' decode step writes
 * the token's K/V into its pool slot and then attends over the request's slots
 * ("Agent-Infer", section "分页 KV 缓存"); this call does both.
 *   slot_ids   : [batch] int32 device array; slot_ids[b] must be request b's LAST
 *                listed slot, kv_indices[kv_indptr[b+1] - 1], and appear in no
 *                other request's list (a newly appended token is private)
 *   k_new, v_new : [batch, n_kv_heads, head_dim] bf16, one new row per request
 *   pool_slots : rows of each pool (used by the debug checks)
 *   every request must have a non-empty context (its newest token); other
 *   arguments as for paged_decode_attn. After the call, k_pool/v_pool hold the new
 *   rows at slot_ids, bit-exact, and out/lse equal those of append-then-attend.
 * With debug checks on, the precondition on slot_ids is verified on the host.
 */
int paged_decode_append_attn(const void* q, void* k_pool, void* v_pool, const int32_t* kv_indptr,
                             const int32_t* kv_indices, const int32_t* slot_ids, const void* k_new,
                             const void* v_new, int batch, int n_qo_heads, int n_kv_heads,
                             int head_dim, int64_t pool_slots, float sm_scale, void* out,
                             float* lse, const pkv_plan* plan, pkv_stream_t stream);

/*
 * paged_decode_attn_static — the same attention as paged_decode_attn, for callers
 * that cannot allocate device memory: an engine that has given all free HBM to
 * its KV pool, a runtime whose allocator must own every device buffer, or a path
 * that must not hit cudaMalloc's implicit synchronisation. The paper has no
 * counterpart; it is an addition of this library.
 *   Arguments as for paged_decode_attn, plus kv_indptr_host ([batch + 1] int32
 *   HOST copy of kv_indptr, read during the call only); there is no plan: every
 *   call plans the step on the host.
 *   Scratch: the work list, a status word, a zero row and the split workspace live
 *   in one file-scope __device__ array of 32 MiB that every GPU loading the library
 *   holds until exit; nothing is allocated. The CUDA driver places the array on a
 *   device when it loads the library's code there (with lazy module loading, at
 *   the first call). The first call on a device (with that device current) looks
 *   the array up with cudaGetSymbolAddress and zeroes its status word and zero row
 *   on `stream`, waiting for that. A call on a stream that is being captured returns
 *   PKV_ERR_UNSUPPORTED without enqueuing anything: its work list is staged in one
 *   shared host array, which a graph would read again at every replay. Steps needing
 *   more than 32 MiB of scratch (or more than 1024 CTAs, 4096 (request, head
 *   group) pairs or 8192 work units) return PKV_ERR_PLAN with the size in the
 *   message.
 *   All calls share the array and leave its contents behind: calls whose kernels
 *   overlap on the GPU race. Calls queued one after another on one stream are
 *   ordered. Calls from several host threads are serialised on the host.
 *   The work list is copied from pageable host memory with cudaMemcpyAsync; the
 *   CUDA runtime may block the host during that copy until it has staged the
 *   bytes.
 *   A bounded pipeline wait that runs out (1 s) sets the array's status word,
 *   which stays set until paged_decode_attn_static_status reads it.
 */
int paged_decode_attn_static(const void* q, const void* k_pool, const void* v_pool,
                             const int32_t* kv_indptr_host, const int32_t* kv_indptr,
                             const int32_t* kv_indices, int batch, int n_qo_heads,
                             int n_kv_heads, int head_dim, float sm_scale, void* out,
                             float* lse, pkv_stream_t stream);

/*
 * paged_decode_attn_static_status — wait for `stream` and the device, then read
 * and clear the status word of paged_decode_attn_static's array on the current
 * device (this library's own; the paper has no counterpart). *status = 0: every
 * static call since the last read completed its pipeline waits (or none ran on
 * this device); nonzero: some wait exceeded its bound and that call's outputs are
 * invalid. Allocates nothing.
 */
int paged_decode_attn_static_status(pkv_stream_t stream, int* status);

/* paged_decode_plan_destroy — free a plan (waits for its pending copy). NULL is a no-op. */
void paged_decode_plan_destroy(pkv_plan* plan);

/*
 * paged_decode_plan_host — the planner alone, on the host, with no CUDA call.
 * Computes the work list paged_decode_plan / paged_decode_plan_shared would upload,
 * for inspection and tests. The work of one layer is a list of items, each a run of
 * slots of one KV-head group (heads_per_cta consecutive KV heads) attended by one
 * request, or, for a shared prefix, by up to requests_per_unit requests of a
 * sharing group; the items are laid end to end and cut into `ctas` ranges of equal
 * token count (fewer for a small step); a run is split only where a range boundary
 * falls inside it.
 *   kv_indptr_host : [batch + 1] int32
 *   n_kv_heads, head_dim : the attention shape
 *   heads_per_cta  : KV heads per group: 1, 2 or 4, at most 512 / head_dim and
 *                    dividing n_kv_heads; 0 = the largest allowed
 *   ctas           : persistent CTAs (SMs x resident CTAs per SM on the device)
 *   shared_indptr_host, n_shared, shared_len_host, requests_per_unit : sharing
 *                    groups as for paged_decode_plan_shared (n_shared = 0: none)
 *   units_out      : [max_units * 8] int32 — per unit {request b, head group,
 *                    first token, end token (exclusive), first partial slot or -1
 *                    when the unit writes out/lse directly, requests served,
 *                    kv_indptr[b] + first token, context length of b, or for a
 *                    shared prefix -2 when other units of its sharing group read
 *                    the same slots and -1 when none does}, listed CTA by CTA
 *   cta_begin_out  : [ctas + 1] int32 — CTA c runs units [cta_begin[c], cta_begin[c+1]);
 *                    every CTA of the grid has an entry (possibly an empty range)
 *   merges_out     : [max_merges * 4] int32 — per (request, head group) with partial
 *                    results {request, head group, first entry in the part list,
 *                    number of parts}
 *   part_list_out  : [max_partials] int32 — partial slots named by the merges
 *   counts_out     : [5] int32 — {units, CTAs with work, merge records, partial
 *                    slots, tokens per CTA range}
 * Returns PKV_ERR_PLAN if an output array is too small.
 */
int paged_decode_plan_host(const int32_t* kv_indptr_host, int batch, int n_kv_heads,
                           int head_dim, int heads_per_cta, int ctas,
                           const int32_t* shared_indptr_host, int n_shared,
                           const int32_t* shared_len_host, int requests_per_unit,
                           int32_t* units_out, int max_units, int32_t* cta_begin_out,
                           int32_t* merges_out, int max_merges, int32_t* part_list_out,
                           int max_partials, int32_t* counts_out);

/* paged_decode_plan_info — counts of the plan's current step (any out pointer may be NULL). */
int paged_decode_plan_info(const pkv_plan* plan, int* batch, int* n_units, int* n_merges,
                           int* chunk_tokens, int* n_ctas);

/*
 * ---------------------------------------------------------------------------
 * Chunked prefill over the same pool
 * ---------------------------------------------------------------------------
 * "Agent-Infer", section "连续批处理" (continuous batching): long prefills are cut
 * into chunks (512 tokens by default, 64 while decodes are running) so that decode
 * steps run between them. A chunk is a request's newest C tokens. Their K/V rows
 * are already in the pool (kvpool_append) and their slots are the last C entries of
 * the request's slot list of L >= C entries. Query c of the chunk (c < C) sits at
 * list position p = L - C + c and attends causally to entries 0 .. p:
 *   s_j      = sm_scale * dot(q[i,h,:], K[idx_j, g, :]),   j <= p
 *   lse[i,h] = ln sum_{j<=p} exp(s_j)
 *   out[i,h] = sum_{j<=p} exp(s_j - lse[i,h]) * V[idx_j, g, :]
 * with i = qo_indptr[b] + c and g = h / (n_qo_heads / n_kv_heads).
 */
typedef struct pkv_prefill_plan pkv_prefill_plan; /* opaque, library-owned */

/*
 * paged_prefill_plan_create — allocate a reusable prefill plan for one shape.
 *   max_batch    : largest batch of any step (>= 1)
 *   max_q_tokens : largest qo_indptr[batch] of any step (>= 0)
 *   n_qo_heads, n_kv_heads, head_dim : head_dim 128 or 256; group size
 *                  n_qo_heads / n_kv_heads in {1, 2, 4, 8}
 * Uses the current device, which must be current for every call that takes the plan
 * (PKV_ERR_INVALID_ARG otherwise). Synchronous. PKV_ERR_UNSUPPORTED for other shapes.
 */
int paged_prefill_plan_create(pkv_prefill_plan** plan, int max_batch, int64_t max_q_tokens,
                              int n_qo_heads, int n_kv_heads, int head_dim);

/*
 * paged_prefill_plan — the step's work list, once per prefill step (reused by every
 * layer). Cuts every chunk into tiles of 128 / G query tokens per KV head and orders
 * the tiles longest causal range first. Uploaded asynchronously on `stream` from
 * pinned staging; waits on the host for the previous step's upload first.
 *   qo_indptr_host : [batch + 1] int32 HOST copy of the chunk offsets (qo_indptr[0] = 0,
 *                    non-decreasing, qo_indptr[batch] <= max_q_tokens)
 *   kv_indptr_host : [batch + 1] int32 HOST copy of the slot-list offsets; every
 *                    request lists at least as many slots as its chunk has tokens
 * Returns PKV_ERR_INVALID_ARG for bad offsets, PKV_ERR_PLAN if batch > max_batch.
 */
int paged_prefill_plan(pkv_prefill_plan* plan, const int32_t* qo_indptr_host,
                       const int32_t* kv_indptr_host, int batch, pkv_stream_t stream);

/*
 * paged_prefill_attn — causal attention of the planned chunks, once per layer.
 *   q          : [qo_indptr[batch], n_qo_heads, head_dim] bf16
 *   k_pool, v_pool, kv_indices : as for paged_decode_attn (the chunk's rows appended)
 *   qo_indptr, kv_indptr : [batch + 1] int32 device arrays equal to the plan's host
 *                copies (checked against them when debug checks are on)
 *   out        : [qo_indptr[batch], n_qo_heads, head_dim] bf16, written
 *   lse        : [qo_indptr[batch], n_qo_heads] fp32 natural-log lse, or NULL
 *   plan       : built by paged_prefill_plan for this step, same shape
 * One kernel launch on the fifth-generation tensor cores (tcgen05, accumulators in
 * tensor memory; 230 KB of shared memory per CTA, one CTA per SM), plus a merge
 * kernel when the plan split long ranges; none when the step has no query tokens.
 * bf16 inputs, fp32 accumulation, probabilities rounded to bf16 for P V, an online
 * softmax; q, pools and out must be 16-byte aligned. Every pipeline wait is bounded
 * (1 s); an expired one is reported by paged_prefill_plan_status.
 */
int paged_prefill_attn(const void* q, const void* k_pool, const void* v_pool,
                       const int32_t* qo_indptr, const int32_t* kv_indptr,
                       const int32_t* kv_indices, int batch, int n_qo_heads, int n_kv_heads,
                       int head_dim, float sm_scale, void* out, float* lse,
                       const pkv_prefill_plan* plan, pkv_stream_t stream);

/*
 * paged_prefill_plan_host — the prefill planner alone, on the host, with no CUDA call
 * (for inspection and tests). Same offset checks as paged_prefill_plan.
 *   split_target : a step with fewer tile units than this has its long ranges split
 *                  (paged_prefill_plan uses two waves of the device's grid, three at
 *                  head_dim 256); 0 = never
 *   units_out    : [max_units * 8] int32 — per unit {workspace block or -1, KV head,
 *                  first query row, query rows, kv_indptr[b], list position of the
 *                  first query, first list entry, end list entry (exclusive)}
 *   merges_out   : [max_merges * 8] int32 — per split unit {first query row, query rows,
 *                  KV head, first workspace block, blocks, 0, 0, 0}
 *   counts_out   : [3] int32 — {units, merge records, workspace blocks}
 * Returns PKV_ERR_PLAN if an output array is too small.
 */
int paged_prefill_plan_host(const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                            int batch, int n_qo_heads, int n_kv_heads, int head_dim,
                            int split_target, int32_t* units_out, int max_units,
                            int32_t* merges_out, int max_merges, int32_t* counts_out);

/*
 * paged_prefill_plan_status — read and clear the prefill plan's device status word
 * (synchronous). 0: every prefill kernel that used the plan completed its pipeline
 * waits; nonzero: some wait exceeded its bound (1 s) and that launch's outputs are
 * invalid.
 */
int paged_prefill_plan_status(pkv_prefill_plan* plan, int* status);

/* paged_prefill_plan_destroy — free a prefill plan (waits for its pending upload). NULL is a no-op. */
void paged_prefill_plan_destroy(pkv_prefill_plan* plan);

/*
 * paged_decode_plan_host_times — host time spent by the plan's successful
 * paged_decode_plan / paged_decode_plan_shared calls since the last reset (this
 * library's own; the pages have no counterpart): in the partition itself
 * (*compute_us) and waiting for a staging buffer to be free (*wait_us), summed
 * over *calls calls, in microseconds. reset != 0 zeroes the counters after they
 * are read. Any out pointer may be NULL. No CUDA call.
 */
int paged_decode_plan_host_times(pkv_plan* plan, double* compute_us, double* wait_us,
                                 int64_t* calls, int reset);

/* Flags for paged_decode_plan_set_flags. */
#define PKV_PLAN_EARLY_GATHER 1u
#define PKV_PLAN_PERSISTENT 2u
#define PKV_PLAN_SINGLE_LAUNCH 4u

/*
 * paged_decode_plan_set_flags — options for the attention calls that use `plan`
 * (this library's own; the pages have no counterpart). Replaces the plan's flags.
 *   PKV_PLAN_EARLY_GATHER: the caller promises that kv_indptr, kv_indices and every
 *     K/V pool row that the step's attention calls read were written by work enqueued on
 *     the stream before this step's paged_decode_plan / paged_decode_plan_shared
 *     call, and that nothing writes them between that call and the step's last
 *     attention call. Exempt are the newest rows that paged_decode_append_attn
 *     takes from k_new / v_new and writes itself. The attention kernel then starts
 *     loading those rows as soon as it is scheduled, while the kernel before it on
 *     the stream may still run (programmatic dependent launch); the work after the
 *     plan's host-to-device copy has all started after the writes completed. q,
 *     k_new, v_new and the newest rows are still read only after the previous
 *     kernel has completed. This fits a step whose pool was filled by earlier
 *     steps and whose new token is appended by paged_decode_append_attn. It does
 *     not fit a step that calls kvpool_append or kvpool_prefetch after the plan.
 *     Off by default; a broken promise gives stale rows, not an error.
 *   PKV_PLAN_PERSISTENT: a small plan's steps run on the persistent grid with an
 *     uploaded work list instead of in single-launch mode (paged_decode_plan_create);
 *     takes effect from the next paged_decode_plan call.
 *   PKV_PLAN_SINGLE_LAUNCH: every step runs in single-launch mode (as a small plan's
 *     do) whatever max_tokens, for callers whose requests are short: the mode splits
 *     each request 16 ways on its own cluster (8 or 4 ways on clusters of 8 or 4 when
 *     larger clusters for max_batch x KV-head groups do not all fit the device at
 *     once), so a step of requests of a few hundred to a few thousand tokens takes one
 *     launch with no upload and no merge kernel, while a step with one long context
 *     streams it on only 2-8 SMs and is slower than on the persistent grid. Results
 *     are the same either way. Returns PKV_ERR_UNSUPPORTED when max_batch x KV-head
 *     groups exceed even the clusters of 4 the device holds at once, and
 *     PKV_ERR_INVALID_ARG together with PKV_PLAN_PERSISTENT. Takes effect from the
 *     next paged_decode_plan call; graphs then follow the single-launch rule above.
 *   flags : a bitwise OR of PKV_PLAN_* values (0 = none)
 * Returns PKV_ERR_PLAN for a NULL plan and PKV_ERR_INVALID_ARG for unknown bits (the
 * plan's flags are then unchanged).
 * Takes effect for attention calls enqueued after it returns.
 */
int paged_decode_plan_set_flags(pkv_plan* plan, unsigned flags);

/*
 * paged_decode_plan_mode — *single_launch = 1 when the plan's steps run in the
 * single-launch small-step mode (see paged_decode_plan_create), 0 when they run on
 * the persistent grid with an uploaded work list. No CUDA call.
 */
int paged_decode_plan_mode(const pkv_plan* plan, int* single_launch);

/*
 * paged_decode_plan_status — read and clear the plan's device status word
 * (synchronous). 0: every attention kernel that used the plan completed its
 * pipeline waits; nonzero: some wait exceeded its bound (1 s) and that launch's
 * outputs are invalid.
 */
int paged_decode_plan_status(pkv_plan* plan, int* status);

/*
 * pkv_set_debug_checks — when on (nonzero), kvpool_append, the decode attention
 * calls and paged_prefill_attn also check, before launching, that each device array
 * is device (or managed) memory of the right device (PKV_ERR_INVALID_ARG naming the
 * array; a host pointer would fault the kernel instead), and copy slot ids / indptr /
 * indices to the host and check them (range, and agreement with the plan,
 * PKV_ERR_INDEX); this synchronises the stream. Off by default. Process-wide.
 */
void pkv_set_debug_checks(int on);

/*
 * pkv_inject_stall — failure injection for tests of the bounded waits (this
 * library's own; the pages have no counterpart). The next n_launches attention
 * launches (paged_decode_attn / paged_decode_append_attn / paged_prefill_attn, any
 * thread) run with producers that issue no copies. Every pipeline wait of such a
 * launch expires after its bound (1 s), the launch ends without a fault or a hang
 * (the prefill kernel frees its tensor memory on that path too), and the plan's
 * status word reads nonzero (paged_decode_plan_status / paged_prefill_plan_status);
 * its outputs are invalid. Later launches are unaffected. 0 cancels. Process-wide.
 */
void pkv_inject_stall(int n_launches);

/* pkv_last_error — message of the last failed call on this thread ("" if none). */
const char* pkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
