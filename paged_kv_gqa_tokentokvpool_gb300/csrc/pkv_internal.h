// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <initializer_list>
#include <vector>

#include "pkv.h"

namespace pkv {

// ---- tracing ------------------------------------------------------------
// Every C entry point that enqueues GPU work runs inside an NVTX range of its name
// (NVTX v3, header only), so profiler timelines show the library's calls and their
// kernels, and ncu can select kernels by call (--nvtx --nvtx-include "name/"). With
// no profiling tool attached a range costs a check of a function pointer.
struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

// ---- launches -----------------------------------------------------------
// Kernels are launched with programmatic stream serialisation (PDL) unless the
// environment variable PKV_PDL is "0" (a diagnostic switch: results do not depend
// on it, only how soon a kernel starts): a kernel may then be scheduled while its
// predecessor on the stream is still running, and does only plan reads and
// barrier set-up before its griddepcontrol.wait.
bool pdl_enabled();
// Whether the plan's steps run in single-launch mode (see paged_decode_plan_set_flags).
bool single_launch_mode(const pkv_plan* p);
// PKV_OK when the current device is plan_device, else PKV_ERR_INVALID_ARG (message set).
int check_plan_device(const char* who, int plan_device);
// Debug checks: every named array (NULL ones skipped) is device or managed memory of
// `device`, else PKV_ERR_INVALID_ARG naming it (a host or foreign pointer would fault
// the kernel instead).
struct NamedPtr {
    const char* name;
    const void* ptr;
};
int check_on_device(const char* who, int device, std::initializer_list<NamedPtr> arrays);

// ---- errors -------------------------------------------------------------
int fail(int code, const char* fmt, ...);  // records the message, returns code
void clear_error();
bool debug_checks();
// One injected stall (pkv_inject_stall) for the attention launch being prepared:
// true if this launch is to withhold its copies (and the count is taken down).
bool take_injected_stall();

// ---- shapes ----------------------------------------------------------------
// A CTA of the decode kernel serves one KV-head group of 1, 2 or 4 consecutive
// KV heads, at most kHeadGroupElems / head_dim of them, so that one token's K (or
// V) row of a group is at most kHeadGroupElems bf16 = 1 KB, one bulk copy.
// heads_per_group() is the largest group the shape allows, the group every plan
// uses (the host-only planner entry also accepts smaller ones).
constexpr int kHeadGroupElems = 512;
inline int heads_per_group(int n_kv_heads, int head_dim) {
    const int cap = kHeadGroupElems / head_dim;
    return n_kv_heads < cap ? n_kv_heads : cap;
}

// ---- plan ----------------------------------------------------------------
// One work unit of the decode kernel: tokens [tok_begin, tok_end) of the slot list
// of request b, KV-head group hg, attended for the nreq requests b .. b+nreq-1
// (nreq > 1 only for a prefix those requests share); idx_begin = kv_indptr[b] +
// tok_begin is where the unit's slot ids start in kv_indices, and len is request
// b's context length, which tells the fused append which token is the newest (for
// a shared prefix: -2 if other units of the sharing group read the same slots, so
// their rows should stay in L2, else -1). partial < 0: the unit covers a whole context and writes
// out/lse; otherwise request b+r writes partial slot partial + r of the workspace.
struct Unit {
    int32_t b, hg, tok_begin, tok_end, partial, nreq, idx_begin, len;
};
// One (request, head group) whose result is merged from partial results: the
// slots part_list[first .. first + count).
struct Merge {
    int32_t b, hg, first, count;
};
static_assert(sizeof(Unit) == 32 && sizeof(Merge) == 16, "plan record sizes");

// No piece of a context split across CTAs is planned shorter than this.
constexpr int kMinChunkTokens = 64;
// Tokens of K/V that one decode pipeline stage holds for a head group of hpc heads
// of head_dim: a stage carries kStageRows rows of kHeadGroupElems bf16 of K and as
// many of V, so a smaller group takes proportionally more tokens per stage.
constexpr int kStageRows = 16;
inline int decode_stage_tokens(int hpc, int head_dim) {
    return kStageRows * (kHeadGroupElems / (hpc * head_dim));
}

struct PlanLimits {
    int max_units;
    int max_merges;
    int max_partials;
};
struct PlanCounts {
    int n_units, n_ctas, n_merges, n_partials, chunk_tokens;
};
// Runs of consecutive requests that list the same first len[s] slots: requests
// [indptr[s], indptr[s+1]) share len[s] slots; prefix units serve up to
// requests_per_unit of them at once.
struct PlanSharing {
    const int32_t* indptr;
    const int32_t* len;
    int n;
    int requests_per_unit;
};

int plan_max_units(int ctas, int max_batch, int n_groups);
// Pure host planner. units[max_units], cta_begin[ctas + 1] (every CTA of the grid
// gets an entry; unused ones an empty range), merges[max_merges],
// part_list[max_partials]. stage_tokens: decode_stage_tokens() of the plan's head
// group (the planner's cost model). sharing may be NULL.
// Returns PKV_OK, PKV_ERR_PLAN (capacity) or PKV_ERR_INVALID_ARG (bad indptr).
int plan_compute(const int32_t* indptr, int batch, int n_groups, int ctas, int stage_tokens,
                 const PlanLimits& lim,
                 const PlanSharing* sharing, Unit* units, int* cta_begin, Merge* merges,
                 int32_t* part_list, PlanCounts* out);

// ---- kernels -------------------------------------------------------------
struct DecodeArgs {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* kv_indices;
    const Unit* units;
    const int32_t* cta_begin;
    const Merge* merges;
    const int32_t* part_list;  // partial slots of the merge records
    int n_ctas;           // grid size: every CTA of the plan (some may have no units)
    bool shared;          // the shared-prefix kernel (prefix units of several requests)
    bool early;           // slot ids and old pool rows may be loaded before the
                          // previous kernel completes (PKV_PLAN_EARLY_GATHER)
    bool withhold;        // injected stall (pkv_inject_stall): the producer issues no
                          // copies, so every pipeline wait of the launch expires
    int heads_per_cta;    // KV heads of one group
    int n_qo_heads;
    int n_kv_heads;
    int head_dim;
    float sm_scale;
    void* out;
    float* lse;
    float* ws_o;          // [max partials, group q heads, head_dim] fp32 partial outputs
    float* ws_lse;        // [max partials, group q heads] fp32 partial lse (base 2)
    const int32_t* meta_header;  // device copy of {merge records, partial slots, 0, 0}
    int merge_ctas;       // grid of the merge kernel (fixed per plan)
    int* status;          // device status word (nonzero: a wait timed out)
    const void* zero_row; // kHeadGroupElems bf16 zeros (tile padding)
    // Fused append (all three set, or all NULL): request b's last listed token is
    // read from row b of k_new / v_new, and that row is written to pool slot
    // slot_ids[b] (k_pool / v_pool are then written, despite the const).
    const void* k_new;
    const void* v_new;
    const int32_t* slot_ids;
    // Host KV tier (both set, or both NULL; never with the fused append): GPU-visible
    // addresses of pinned host pools; a negative slot id -1 - h names host row h.
    const void* k_host;
    const void* v_host;
    // Single-launch small steps (small != 0: the cluster size, 16 or 8): no work list;
    // the kernel reads the step's kv_indptr ([batch + 1], on the device) and merges
    // split parts in each cluster.
    int small;
    int batch;
    const int32_t* kv_indptr;
};

bool decode_shape_supported(int n_qo_heads, int n_kv_heads, int head_dim);
// Resident CTAs per SM of the decode kernel (plain or shared-prefix instance)
// for this shape (0 on error or when no such instance exists).
int decode_ctas_per_sm(int n_qo_heads, int n_kv_heads, int head_dim, int heads_per_cta,
                       bool shared);
// Query rows per KV head that one unit of the shared-prefix kernel serves (so
// rows / G requests of a sharing group), or 0 when this shape has no such kernel.
int decode_shared_rows(int n_qo_heads, int n_kv_heads, int head_dim, int heads_per_cta);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// ---- small steps in one launch ----------------------------------------------
// CTAs of one thread-block cluster of the single-launch kernel (a non-portable
// cluster size): each (request, head group) of a small step is split 16 ways.
constexpr int kSmallCluster = 16;
// The smaller clusters (portable sizes) the mode falls back to when a plan's clusters of
// 16 do not all fit the device at once: each request split 8, then 4 ways.
constexpr int kSmallClusterSizes[3] = {16, 8, 4};
// A small-step plan's longest context gives each CTA at most this many stages.
constexpr int kSmallMaxStages = 8;
// Clusters of that kernel resident at once for this shape (0: it cannot run here).
int decode_small_clusters(int n_qo_heads, int n_kv_heads, int head_dim, int cluster_size);

// Row scatter between two pools (either may be pinned host memory mapped for the GPU):
// dst[dst_slots[i]] = src[src_slots[i]] for K and V, i < n.
cudaError_t launch_tier_copy(const void* k_src, const void* v_src, const int32_t* src_slots,
                             void* k_dst, void* v_dst, const int32_t* dst_slots, int64_t n,
                             int row_bytes, cudaStream_t stream);

cudaError_t launch_append(void* k_pool, void* v_pool, const int32_t* slot_ids,
                          const void* k_new, const void* v_new, int64_t n, int row_bytes,
                          cudaStream_t stream);

}  // namespace pkv

struct pkv_plan {
    int device = 0;
    // persistent CTAs of the plain and of the shared-prefix kernel (the staging is
    // sized for the larger grid)
    int num_sms = 0, ctas_per_sm = 0, ctas = 0, ctas_shared = 0, ctas_max = 0;
    int max_batch = 0;
    int64_t max_tokens = 0;
    int n_qo_heads = 0, n_kv_heads = 0, head_dim = 0, n_groups = 0, heads_per_cta = 0;
    pkv::PlanLimits lim{};
    size_t meta_bytes = 0;
    // Two pinned staging buffers (header, cta_begin, merges, part list, units), used
    // in turn: a step's plan call waits only for the upload of the step before the
    // previous one, so the host may run two steps ahead of the GPU.
    void* host_staging[2] = {nullptr, nullptr};
    cudaEvent_t copy_done[2] = {nullptr, nullptr};
    bool copy_pending[2] = {false, false};
    int next_staging = 0;          // the buffer the next plan call fills
    void* dev_meta = nullptr;      // device copy of the same (used prefix uploaded per step)
    float* ws_o = nullptr;
    float* ws_lse = nullptr;
    int* dev_state = nullptr;      // status word, padding
    void* zero_row = nullptr;
    // host time of the plan calls since the last reset (paged_decode_plan_host_times)
    double compute_ns = 0, wait_ns = 0;
    int64_t timed_calls = 0;
    // the current step
    bool planned = false;
    int batch = 0;
    pkv::PlanCounts counts{};
    size_t off_cta = 0, off_merge = 0, off_list = 0, off_units = 0;  // offsets in the staging
    int share_rows = 0;  // requests per shared-prefix unit (0: this shape has no such kernel)
    int merge_ctas = 0;  // grid of the merge kernel
    unsigned flags = 0;  // PKV_PLAN_* options
    bool shared = false; // the current step runs the shared-prefix kernel
    int launch_ctas = 0; // grid of the current step's decode kernel
    // Small-step mode (fixed at creation): every step runs as one launch of the
    // cluster kernel, which reads kv_indptr on the device; nothing is uploaded.
    bool small = false;
    // every step of the plan could run in that mode: max_batch x groups clusters fit the
    // device at once (PKV_PLAN_SINGLE_LAUNCH selects the mode whatever max_tokens)
    bool small_fits = false;
    // the cluster size of the mode: the largest of 16, 8, 4 whose clusters all fit
    int small_cs = 0;
    bool step_small = false;  // the current step runs in that mode
    std::vector<int32_t> indptr_host;
    // the current step's sharing description (checked against kv_indices when
    // debug checks are on and the shared-prefix kernel runs)
    std::vector<int32_t> shared_indptr_host, shared_len_host;
};
