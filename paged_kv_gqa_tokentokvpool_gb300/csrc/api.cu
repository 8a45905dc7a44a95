// The C ABI (include/pkv.h): argument checks, plan lifetime, launches.
//
// Every entry point validates its arguments on the host and returns an error code
// before enqueuing anything, so a bad call never reaches the GPU. The plan owns
// the only memory the library allocates, sized once at creation.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "pkv_internal.h"

namespace pkv {
namespace {

thread_local std::string g_last_error;
int g_debug_checks = 0;
std::atomic<int> g_stalls_to_inject{0};  // pkv_inject_stall

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_fail(cudaError_t e, const char* what) {
    return fail(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

}  // namespace

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

void clear_error() { g_last_error.clear(); }
bool debug_checks() { return g_debug_checks != 0; }

bool take_injected_stall() {
    int stalls = g_stalls_to_inject.load();
    while (stalls > 0 && !g_stalls_to_inject.compare_exchange_weak(stalls, stalls - 1)) {
    }
    return stalls > 0;
}

// A plan's buffers live on the device it was created on: calls that use it must run
// with that device current, or its kernels would address another GPU's memory.
int check_plan_device(const char* who, int plan_device) {
    int dev = -1;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "%s: cudaGetDevice: %s", who, cudaGetErrorString(e));
    if (dev != plan_device)
        return fail(PKV_ERR_INVALID_ARG, "%s: the plan belongs to device %d but device %d is current",
                    who, plan_device, dev);
    return PKV_OK;
}

int check_on_device(const char* who, int device, std::initializer_list<NamedPtr> arrays) {
    for (const NamedPtr& a : arrays) {
        if (a.ptr == nullptr) continue;
        cudaPointerAttributes attr{};
        const cudaError_t e = cudaPointerGetAttributes(&attr, a.ptr);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(PKV_ERR_INVALID_ARG, "%s: %s is not memory CUDA knows (%s)", who, a.name,
                        cudaGetErrorString(e));
        }
        if (attr.type == cudaMemoryTypeManaged) continue;
        if (attr.type != cudaMemoryTypeDevice || attr.device != device)
            return fail(PKV_ERR_INVALID_ARG, "%s: %s is not device memory of device %d", who, a.name,
                        device);
    }
    return PKV_OK;
}

// The plan's steps run as single launches of the cluster kernel: small plans unless
// PKV_PLAN_PERSISTENT, and any plan whose clusters fit with PKV_PLAN_SINGLE_LAUNCH.
bool single_launch_mode(const pkv_plan* p) {
    if (p->flags & PKV_PLAN_PERSISTENT) return false;
    return p->small || ((p->flags & PKV_PLAN_SINGLE_LAUNCH) && p->small_fits);
}

bool pdl_enabled() {
    static const bool on = [] {
        const char* env = std::getenv("PKV_PDL");
        return !(env && env[0] == '0');
    }();
    return on;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_last_error(void) { return g_last_error.c_str(); }

void pkv_set_debug_checks(int on) { g_debug_checks = on ? 1 : 0; }

void pkv_inject_stall(int n_launches) { g_stalls_to_inject.store(n_launches > 0 ? n_launches : 0); }

int kvpool_append(void* k_pool, void* v_pool, const int32_t* slot_ids, const void* k_new,
                  const void* v_new, int64_t n, int n_kv_heads, int head_dim,
                  int64_t pool_slots, pkv_stream_t stream) {
    TraceRange trace("kvpool_append");
    clear_error();
    if (n < 0) return fail(PKV_ERR_INVALID_ARG, "kvpool_append: n = %lld < 0", (long long)n);
    if (n_kv_heads <= 0 || head_dim <= 0 || pool_slots <= 0)
        return fail(PKV_ERR_INVALID_ARG, "kvpool_append: n_kv_heads, head_dim, pool_slots must be > 0");
    const int64_t row_bytes = int64_t(n_kv_heads) * head_dim * 2;
    if (row_bytes % 16 != 0)
        return fail(PKV_ERR_UNSUPPORTED, "kvpool_append: row of %lld bytes is not a multiple of 16",
                    (long long)row_bytes);
    if (n > pool_slots)
        return fail(PKV_ERR_INVALID_ARG, "kvpool_append: n = %lld rows exceed pool_slots = %lld",
                    (long long)n, (long long)pool_slots);
    if (n == 0) return PKV_OK;
    if (!k_pool || !v_pool || !slot_ids || !k_new || !v_new)
        return fail(PKV_ERR_INVALID_ARG, "kvpool_append: NULL pointer argument");
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new))
        return fail(PKV_ERR_INVALID_ARG, "kvpool_append: pools and new rows must be 16-byte aligned");
    if (debug_checks()) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (int rc = check_on_device("kvpool_append", dev,
                                     {{"k_pool", k_pool}, {"v_pool", v_pool}, {"slot_ids", slot_ids},
                                      {"k_new", k_new}, {"v_new", v_new}});
            rc != PKV_OK)
            return rc;
        std::vector<int32_t> ids(n);
        cudaError_t e = cudaMemcpyAsync(ids.data(), slot_ids, n * sizeof(int32_t),
                                        cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return cuda_fail(e, "kvpool_append: debug copy of slot_ids");
        std::vector<int32_t> sorted(ids);
        std::sort(sorted.begin(), sorted.end());
        for (int64_t i = 0; i < n; ++i) {
            if (ids[i] < 0 || ids[i] >= pool_slots)
                return fail(PKV_ERR_INDEX, "kvpool_append: slot_ids[%lld] = %d outside [0, %lld)",
                            (long long)i, ids[i], (long long)pool_slots);
            if (i > 0 && sorted[i] == sorted[i - 1])
                return fail(PKV_ERR_INDEX, "kvpool_append: slot id %d appears twice", sorted[i]);
        }
    }
    cudaError_t e = launch_append(k_pool, v_pool, slot_ids, k_new, v_new, n,
                                  static_cast<int>(row_bytes), stream);
    if (e != cudaSuccess) return cuda_fail(e, "kvpool_append: launch");
    return PKV_OK;
}

namespace {

// GPU-visible address of a pool argument: device memory (want_host = false) or
// pinned host memory mapped into the GPU's address space (want_host = true).
// Pageable or unknown memory is rejected here, so it never reaches a kernel.
int gpu_address(const char* who, const char* name, const void* p, bool want_host, void** out) {
    cudaPointerAttributes attr{};
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PKV_ERR_INVALID_ARG, "%s: %s is not memory CUDA knows (%s)", who, name,
                    cudaGetErrorString(e));
    }
    if (want_host) {
        if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr)
            return fail(PKV_ERR_INVALID_ARG,
                        "%s: %s must be pinned host memory mapped for the GPU (cudaHostAlloc, "
                        "or a pinned torch tensor)", who, name);
        *out = attr.devicePointer;
    } else {
        if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
            return fail(PKV_ERR_INVALID_ARG, "%s: %s must be device memory", who, name);
        *out = const_cast<void*>(p);
    }
    return PKV_OK;
}

int check_slots(const char* who, const char* name, const int32_t* slots, int64_t n, int64_t cap,
                bool distinct, cudaStream_t stream) {
    std::vector<int32_t> ids(n);
    cudaError_t e = cudaMemcpyAsync(ids.data(), slots, n * sizeof(int32_t), cudaMemcpyDeviceToHost,
                                    stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "debug copy of slot ids");
    for (int64_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= cap)
            return fail(PKV_ERR_INDEX, "%s: %s[%lld] = %d outside [0, %lld)", who, name, (long long)i,
                        ids[i], (long long)cap);
    if (distinct) {
        std::sort(ids.begin(), ids.end());
        for (int64_t i = 1; i < n; ++i)
            if (ids[i] == ids[i - 1])
                return fail(PKV_ERR_INDEX, "%s: %s repeats slot %d", who, name, ids[i]);
    }
    return PKV_OK;
}

// Shared by kvpool_offload and kvpool_prefetch: dst[dst_slots] = src[src_slots].
int tier_copy(const char* who, bool to_host, const void* k_dev, const void* v_dev,
              const int32_t* dev_slots, const void* k_host, const void* v_host,
              const int32_t* host_slots, int64_t n, int n_kv_heads, int head_dim,
              int64_t pool_slots, int64_t host_slots_cap, pkv_stream_t stream) {
    if (n < 0) return fail(PKV_ERR_INVALID_ARG, "%s: n = %lld < 0", who, (long long)n);
    if (n_kv_heads <= 0 || head_dim <= 0 || pool_slots <= 0 || host_slots_cap <= 0)
        return fail(PKV_ERR_INVALID_ARG,
                    "%s: n_kv_heads, head_dim, pool_slots, host_slots_cap must be > 0", who);
    const int64_t row_bytes = int64_t(n_kv_heads) * head_dim * 2;
    if (row_bytes % 16 != 0)
        return fail(PKV_ERR_UNSUPPORTED, "%s: row of %lld bytes is not a multiple of 16", who,
                    (long long)row_bytes);
    if (n == 0) return PKV_OK;
    if (!k_dev || !v_dev || !dev_slots || !k_host || !v_host || !host_slots)
        return fail(PKV_ERR_INVALID_ARG, "%s: NULL pointer argument", who);
    if (!aligned16(k_dev) || !aligned16(v_dev) || !aligned16(k_host) || !aligned16(v_host))
        return fail(PKV_ERR_INVALID_ARG, "%s: pools must be 16-byte aligned", who);
    void *kd = nullptr, *vd = nullptr, *kh = nullptr, *vh = nullptr;
    int rc = gpu_address(who, "k_pool", k_dev, false, &kd);
    if (rc == PKV_OK) rc = gpu_address(who, "v_pool", v_dev, false, &vd);
    if (rc == PKV_OK) rc = gpu_address(who, "k_host", k_host, true, &kh);
    if (rc == PKV_OK) rc = gpu_address(who, "v_host", v_host, true, &vh);
    if (rc != PKV_OK) return rc;
    if (!aligned16(kh) || !aligned16(vh))
        return fail(PKV_ERR_INVALID_ARG, "%s: host pools must be 16-byte aligned", who);
    if (debug_checks()) {
        rc = check_slots(who, "dev_slots", dev_slots, n, pool_slots, !to_host, stream);
        if (rc == PKV_OK)
            rc = check_slots(who, "host_slots", host_slots, n, host_slots_cap, to_host, stream);
        if (rc != PKV_OK) return rc;
    }
    cudaError_t e = to_host
                        ? launch_tier_copy(kd, vd, dev_slots, kh, vh, host_slots, n,
                                           static_cast<int>(row_bytes), stream)
                        : launch_tier_copy(kh, vh, host_slots, kd, vd, dev_slots, n,
                                           static_cast<int>(row_bytes), stream);
    if (e != cudaSuccess) return cuda_fail(e, "launch");
    return PKV_OK;
}

}  // namespace

int kvpool_offload(const void* k_pool, const void* v_pool, const int32_t* dev_slots, void* k_host,
                   void* v_host, const int32_t* host_slots, int64_t n, int n_kv_heads,
                   int head_dim, int64_t pool_slots, int64_t host_slots_cap, pkv_stream_t stream) {
    TraceRange trace("kvpool_offload");
    clear_error();
    return tier_copy("kvpool_offload", true, k_pool, v_pool, dev_slots, k_host, v_host,
                     host_slots, n, n_kv_heads, head_dim, pool_slots, host_slots_cap, stream);
}

int kvpool_prefetch(void* k_pool, void* v_pool, const int32_t* dev_slots, const void* k_host,
                    const void* v_host, const int32_t* host_slots, int64_t n, int n_kv_heads,
                    int head_dim, int64_t pool_slots, int64_t host_slots_cap, pkv_stream_t stream) {
    TraceRange trace("kvpool_prefetch");
    clear_error();
    return tier_copy("kvpool_prefetch", false, k_pool, v_pool, dev_slots, k_host, v_host,
                     host_slots, n, n_kv_heads, head_dim, pool_slots, host_slots_cap, stream);
}

namespace {

// Checks a sharing description against the step's contexts: runs of consecutive
// requests, each member listing at least len + 1 slots (its newest token stays
// private). Returns PKV_OK or an error code with the message set.
int check_sharing(const char* who, const int32_t* kv_indptr_host, int batch,
                  const int32_t* shared_indptr_host, int n_shared, const int32_t* shared_len_host) {
    if (n_shared < 0) return fail(PKV_ERR_INVALID_ARG, "%s: n_shared %d < 0", who, n_shared);
    if (n_shared == 0) return PKV_OK;
    if (!shared_indptr_host || !shared_len_host)
        return fail(PKV_ERR_INVALID_ARG, "%s: NULL sharing arrays", who);
    for (int s = 0; s < n_shared; ++s) {
        const int m0 = shared_indptr_host[s], m1 = shared_indptr_host[s + 1];
        if (m0 < 0 || m1 < m0 || m1 > batch)
            return fail(PKV_ERR_INVALID_ARG, "%s: shared_indptr is not a non-decreasing run in [0, %d]",
                        who, batch);
        if (shared_len_host[s] < 0)
            return fail(PKV_ERR_INVALID_ARG, "%s: shared_len[%d] < 0", who, s);
        for (int b = m0; b < m1; ++b)
            if (kv_indptr_host[b + 1] - kv_indptr_host[b] <= shared_len_host[s])
                return fail(PKV_ERR_INVALID_ARG,
                            "%s: request %d lists %d slots, not more than its shared prefix of %d",
                            who, b, kv_indptr_host[b + 1] - kv_indptr_host[b], shared_len_host[s]);
    }
    return PKV_OK;
}

}  // namespace

int paged_decode_plan_host(const int32_t* kv_indptr_host, int batch, int n_kv_heads,
                           int head_dim, int heads_per_cta, int ctas,
                           const int32_t* shared_indptr_host, int n_shared,
                           const int32_t* shared_len_host, int requests_per_unit,
                           int32_t* units_out, int max_units, int32_t* cta_begin_out,
                           int32_t* merges_out, int max_merges, int32_t* part_list_out,
                           int max_partials, int32_t* counts_out) {
    clear_error();
    if (!counts_out || (max_units > 0 && !units_out) || !cta_begin_out ||
        (max_merges > 0 && !merges_out) || (max_partials > 0 && !part_list_out))
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_plan_host: NULL output");
    if (ctas <= 0 || n_kv_heads <= 0 || head_dim <= 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_plan_host: ctas, n_kv_heads, head_dim must be > 0");
    const int hpg = heads_per_cta > 0 ? heads_per_cta : heads_per_group(n_kv_heads, head_dim);
    if (hpg < 1 || hpg > heads_per_group(n_kv_heads, head_dim) || n_kv_heads % hpg != 0)
        return fail(PKV_ERR_UNSUPPORTED,
                    "paged_decode_plan_host: %d KV heads per group do not fit %d heads of dim %d",
                    hpg, n_kv_heads, head_dim);
    if (batch > 0 && !kv_indptr_host)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_plan_host: kv_indptr_host is NULL");
    int rc = check_sharing("paged_decode_plan_host", kv_indptr_host, batch, shared_indptr_host,
                           n_shared, shared_len_host);
    if (rc != PKV_OK) return rc;
    const PlanSharing sh{shared_indptr_host, shared_len_host, n_shared,
                         requests_per_unit > 0 ? requests_per_unit : 1};
    PlanCounts c{};
    rc = plan_compute(kv_indptr_host, batch, n_kv_heads / hpg, ctas,
                      decode_stage_tokens(hpg, head_dim),
                      PlanLimits{max_units, max_merges, max_partials}, n_shared > 0 ? &sh : nullptr,
                      reinterpret_cast<Unit*>(units_out), cta_begin_out,
                      reinterpret_cast<Merge*>(merges_out), part_list_out, &c);
    if (rc != PKV_OK) return rc;
    counts_out[0] = c.n_units;
    counts_out[1] = c.n_ctas;
    counts_out[2] = c.n_merges;
    counts_out[3] = c.n_partials;
    counts_out[4] = c.chunk_tokens;
    return PKV_OK;
}

void paged_decode_plan_destroy(pkv_plan* p) {
    if (p == nullptr) return;
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(p->device);
    for (int i = 0; i < 2; ++i) {
        if (p->copy_done[i]) {
            cudaEventSynchronize(p->copy_done[i]);
            cudaEventDestroy(p->copy_done[i]);
        }
        if (p->host_staging[i]) cudaFreeHost(p->host_staging[i]);
    }
    if (p->dev_meta) cudaFree(p->dev_meta);
    if (p->ws_o) cudaFree(p->ws_o);
    if (p->ws_lse) cudaFree(p->ws_lse);
    if (p->dev_state) cudaFree(p->dev_state);
    if (p->zero_row) cudaFree(p->zero_row);
    if (prev >= 0) cudaSetDevice(prev);
    delete p;
}

namespace {
size_t round16(size_t x) { return (x + 15) & ~size_t(15); }
}  // namespace

int paged_decode_plan_create(pkv_plan** out_plan, int max_batch, int64_t max_tokens,
                             int n_qo_heads, int n_kv_heads, int head_dim) {
    clear_error();
    if (!out_plan) return fail(PKV_ERR_INVALID_ARG, "paged_decode_plan_create: plan is NULL");
    *out_plan = nullptr;
    if (max_batch < 1 || max_tokens < 0 || max_tokens >= (int64_t(1) << 31))
        return fail(PKV_ERR_INVALID_ARG,
                    "paged_decode_plan_create: need max_batch >= 1 and 0 <= max_tokens < 2^31");
    if (!decode_shape_supported(n_qo_heads, n_kv_heads, head_dim))
        return fail(PKV_ERR_UNSUPPORTED,
                    "paged_decode_plan_create: unsupported shape (n_qo_heads=%d, n_kv_heads=%d, "
                    "head_dim=%d); need head_dim 128/256, group 1/2/4/8, n_kv_heads 1/2/4/8",
                    n_qo_heads, n_kv_heads, head_dim);
    pkv_plan* p = new (std::nothrow) pkv_plan();
    if (!p) return fail(PKV_ERR_INVALID_ARG, "paged_decode_plan_create: out of host memory");
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) {
        delete p;
        return cuda_fail(e, "paged_decode_plan_create: device query");
    }
    const int hpg = heads_per_group(n_kv_heads, head_dim);
    p->heads_per_cta = hpg;
    p->ctas_per_sm = decode_ctas_per_sm(n_qo_heads, n_kv_heads, head_dim, hpg, false);
    // Shared-prefix units serve 16 / G requests where a kernel for them exists; it
    // runs on its own fixed grid.
    const int shared_per_sm = decode_ctas_per_sm(n_qo_heads, n_kv_heads, head_dim, hpg, true);
    p->share_rows = shared_per_sm > 0
                        ? decode_shared_rows(n_qo_heads, n_kv_heads, head_dim, hpg) /
                              (n_qo_heads / n_kv_heads)
                        : 0;
    if (p->ctas_per_sm <= 0) {
        delete p;
        return fail(PKV_ERR_CUDA, "paged_decode_plan_create: occupancy query failed");
    }
    p->ctas = p->num_sms * p->ctas_per_sm;
    p->ctas_shared = p->share_rows > 0 ? p->num_sms * shared_per_sm : 0;
    // A plan whose every step is small runs its steps as single launches of the
    // cluster kernel: all (request, head group) clusters resident at once (clusters of
    // 16, else of 8), and a CTA's share of the longest context the plan allows at most
    // kSmallMaxStages stages.
    {
        const int64_t items = int64_t(max_batch) * (n_kv_heads / hpg);
        const int64_t max_share = int64_t(kSmallCluster) * kSmallMaxStages * decode_stage_tokens(hpg, head_dim);
        p->small_cs = 0;
        for (int cs : kSmallClusterSizes)
            if (items <= decode_small_clusters(n_qo_heads, n_kv_heads, head_dim, cs)) {
                p->small_cs = cs;
                break;
            }
        p->small_fits = p->small_cs > 0;
        // automatic: no CTA's share of any request can exceed kSmallMaxStages stages
        p->small = p->small_fits && max_tokens <= max_share / kSmallCluster * p->small_cs;
    }
    p->ctas_max = std::max(p->ctas, p->ctas_shared);
    p->max_batch = max_batch;
    p->max_tokens = max_tokens;
    p->n_qo_heads = n_qo_heads;
    p->n_kv_heads = n_kv_heads;
    p->head_dim = head_dim;
    p->n_groups = n_kv_heads / hpg;
    p->lim.max_units = plan_max_units(p->ctas_max, max_batch, p->n_groups);
    p->lim.max_merges = max_batch * p->n_groups;
    p->lim.max_partials = p->lim.max_units * std::max(1, p->share_rows);
    p->indptr_host.reserve(max_batch + 1);
    // staging layout: header[4] | cta_begin[ctas + 1] | merges[max_merges] |
    //                 part_list[max_partials] | units[max_units]
    p->off_cta = 16;
    p->off_merge = round16(p->off_cta + sizeof(int32_t) * (p->ctas_max + 1));
    p->off_list = round16(p->off_merge + sizeof(Merge) * p->lim.max_merges);
    p->off_units = round16(p->off_list + sizeof(int32_t) * p->lim.max_partials);
    p->meta_bytes = p->off_units + sizeof(Unit) * p->lim.max_units;
    const int group_q_heads = hpg * (n_qo_heads / n_kv_heads);
    // The merge kernel runs one warp per (merged context, query head of its group),
    // four warps a CTA: enough CTAs for the largest step to need one pass, up to
    // four per SM.
    const int64_t merge_warps = int64_t(p->lim.max_merges) * group_q_heads;
    p->merge_ctas = static_cast<int>(
        std::max<int64_t>(1, std::min<int64_t>((merge_warps + 3) / 4, int64_t(p->num_sms) * 4)));
    const size_t ws_o_bytes = sizeof(float) * size_t(p->lim.max_partials) * group_q_heads * head_dim;
    const size_t ws_lse_bytes = sizeof(float) * size_t(p->lim.max_partials) * group_q_heads;
    const size_t state_bytes = sizeof(int) * 32;
    e = cudaMallocHost(&p->host_staging[0], p->meta_bytes);
    if (e == cudaSuccess) e = cudaMallocHost(&p->host_staging[1], p->meta_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&p->dev_meta, p->meta_bytes);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&p->ws_o), ws_o_bytes);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&p->ws_lse), ws_lse_bytes);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&p->dev_state), state_bytes);
    if (e == cudaSuccess) e = cudaMemset(p->dev_state, 0, state_bytes);
    if (e == cudaSuccess) e = cudaMalloc(&p->zero_row, sizeof(uint16_t) * kHeadGroupElems);
    if (e == cudaSuccess) e = cudaMemset(p->zero_row, 0, sizeof(uint16_t) * kHeadGroupElems);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i)
        e = cudaEventCreateWithFlags(&p->copy_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        paged_decode_plan_destroy(p);
        return cuda_fail(e, "paged_decode_plan_create: allocation");
    }
    *out_plan = p;
    return PKV_OK;
}

namespace {

int plan_impl(const char* who, pkv_plan* p, const int32_t* kv_indptr_host, int batch,
              const int32_t* shared_indptr_host, int n_shared, const int32_t* shared_len_host,
              pkv_stream_t stream) {
    if (!p) return fail(PKV_ERR_PLAN, "%s: plan is NULL", who);
    p->planned = false;
    if (int rc = check_plan_device(who, p->device); rc != PKV_OK) return rc;
    if (batch < 0 || batch > p->max_batch)
        return fail(PKV_ERR_PLAN, "%s: batch %d outside [0, %d]", who, batch, p->max_batch);
    if (!kv_indptr_host) return fail(PKV_ERR_INVALID_ARG, "%s: kv_indptr_host is NULL", who);
    if (int64_t(kv_indptr_host[batch]) > p->max_tokens)
        return fail(PKV_ERR_PLAN, "%s: %d tokens exceed the plan's max_tokens %lld", who,
                    kv_indptr_host[batch], (long long)p->max_tokens);
    if (kv_indptr_host[0] != 0)
        return fail(PKV_ERR_INVALID_ARG, "%s: kv_indptr[0] = %d, expected 0", who, kv_indptr_host[0]);
    for (int b = 0; b < batch; ++b)
        if (kv_indptr_host[b + 1] < kv_indptr_host[b])
            return fail(PKV_ERR_INVALID_ARG, "%s: kv_indptr decreases at %d", who, b);
    int rc = check_sharing(who, kv_indptr_host, batch, shared_indptr_host, n_shared,
                           shared_len_host);
    if (rc != PKV_OK) return rc;
    const bool small = single_launch_mode(p);
    bool share = false;
    if (p->share_rows > 0 && !small)
        for (int s = 0; s < n_shared; ++s)
            share |= shared_len_host[s] > 0 && shared_indptr_host[s + 1] > shared_indptr_host[s];
    const PlanSharing sh{shared_indptr_host, shared_len_host, n_shared, p->share_rows};
    p->step_small = small;
    if (small) {
        // nothing to upload: the cluster kernel reads kv_indptr itself
        const int items = batch * p->n_groups;
        const int st = decode_stage_tokens(p->n_kv_heads / p->n_groups, p->head_dim);
        int longest = 0;
        for (int b = 0; b < batch; ++b)
            longest = std::max(longest, kv_indptr_host[b + 1] - kv_indptr_host[b]);
        const int cs = p->small_cs;
        p->counts = PlanCounts{items * cs, items * cs, items, items * cs,
                               ((longest + cs - 1) / cs + st - 1) / st * st};
        p->batch = batch;
        p->shared = false;
        p->launch_ctas = items * cs;
        p->shared_indptr_host.clear();
        p->shared_len_host.clear();
        p->indptr_host.assign(kv_indptr_host, kv_indptr_host + batch + 1);
        ++p->timed_calls;
        p->planned = true;
        return PKV_OK;
    }
    // The staging buffer this call fills may still feed the upload of the step
    // before the previous one (the buffers are used in turn).
    const int sb = p->next_staging;
    const auto t0 = std::chrono::steady_clock::now();
    if (p->copy_pending[sb]) {
        cudaError_t e = cudaEventSynchronize(p->copy_done[sb]);
        if (e != cudaSuccess) return cuda_fail(e, "waiting for an earlier plan copy");
        p->copy_pending[sb] = false;
    }
    const auto t1 = std::chrono::steady_clock::now();
    char* st = static_cast<char*>(p->host_staging[sb]);
    PlanCounts c{};
    const int ctas = share ? p->ctas_shared : p->ctas;
    rc = plan_compute(kv_indptr_host, batch, p->n_groups, ctas,
                      decode_stage_tokens(p->n_kv_heads / p->n_groups, p->head_dim), p->lim,
                      share ? &sh : nullptr,
                      reinterpret_cast<Unit*>(st + p->off_units),
                      reinterpret_cast<int32_t*>(st + p->off_cta),
                      reinterpret_cast<Merge*>(st + p->off_merge),
                      reinterpret_cast<int32_t*>(st + p->off_list), &c);
    if (rc != PKV_OK) return rc;
    const auto t2 = std::chrono::steady_clock::now();
    int32_t* header = reinterpret_cast<int32_t*>(st);
    header[0] = c.n_merges;
    header[1] = c.n_partials;
    header[2] = header[3] = 0;
    const size_t bytes = p->off_units + sizeof(Unit) * c.n_units;
    cudaError_t e = cudaMemcpyAsync(p->dev_meta, st, bytes, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaEventRecord(p->copy_done[sb], stream);
    if (e != cudaSuccess) return cuda_fail(e, "plan upload");
    p->copy_pending[sb] = true;
    p->next_staging = sb ^ 1;
    p->wait_ns += std::chrono::duration<double, std::nano>(t1 - t0).count();
    p->compute_ns += std::chrono::duration<double, std::nano>(t2 - t1).count();
    ++p->timed_calls;
    if (share) {
        p->shared_indptr_host.assign(shared_indptr_host, shared_indptr_host + n_shared + 1);
        p->shared_len_host.assign(shared_len_host, shared_len_host + n_shared);
    } else {
        p->shared_indptr_host.clear();
        p->shared_len_host.clear();
    }
    p->batch = batch;
    p->counts = c;
    p->shared = share;
    p->launch_ctas = ctas;
    p->indptr_host.assign(kv_indptr_host, kv_indptr_host + batch + 1);
    p->planned = true;
    return PKV_OK;
}

}  // namespace

int paged_decode_plan(pkv_plan* p, const int32_t* kv_indptr_host, int batch, pkv_stream_t stream) {
    TraceRange trace("paged_decode_plan");
    clear_error();
    return plan_impl("paged_decode_plan", p, kv_indptr_host, batch, nullptr, 0, nullptr, stream);
}

int paged_decode_plan_shared(pkv_plan* p, const int32_t* kv_indptr_host, int batch,
                             const int32_t* shared_indptr_host, int n_shared,
                             const int32_t* shared_len_host, pkv_stream_t stream) {
    TraceRange trace("paged_decode_plan_shared");
    clear_error();
    return plan_impl("paged_decode_plan_shared", p, kv_indptr_host, batch, shared_indptr_host,
                     n_shared, shared_len_host, stream);
}

int paged_decode_plan_info(const pkv_plan* p, int* batch, int* n_units, int* n_merges,
                           int* chunk_tokens, int* n_ctas) {
    clear_error();
    if (!p) return fail(PKV_ERR_PLAN, "paged_decode_plan_info: plan is NULL");
    if (batch) *batch = p->batch;
    if (n_units) *n_units = p->counts.n_units;
    if (n_merges) *n_merges = p->counts.n_merges;
    if (chunk_tokens) *chunk_tokens = p->counts.chunk_tokens;
    if (n_ctas) *n_ctas = p->counts.n_ctas;
    return PKV_OK;
}

int paged_decode_plan_host_times(pkv_plan* p, double* compute_us, double* wait_us,
                                 int64_t* calls, int reset) {
    clear_error();
    if (!p) return fail(PKV_ERR_PLAN, "paged_decode_plan_host_times: plan is NULL");
    if (compute_us) *compute_us = p->compute_ns * 1e-3;
    if (wait_us) *wait_us = p->wait_ns * 1e-3;
    if (calls) *calls = p->timed_calls;
    if (reset) {
        p->compute_ns = p->wait_ns = 0;
        p->timed_calls = 0;
    }
    return PKV_OK;
}

int paged_decode_plan_set_flags(pkv_plan* p, unsigned flags) {
    clear_error();
    if (!p) return fail(PKV_ERR_PLAN, "paged_decode_plan_set_flags: plan is NULL");
    constexpr unsigned kKnown = PKV_PLAN_EARLY_GATHER | PKV_PLAN_PERSISTENT | PKV_PLAN_SINGLE_LAUNCH;
    if (flags & ~kKnown)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_plan_set_flags: unknown flags 0x%x",
                    flags & ~kKnown);
    if ((flags & PKV_PLAN_PERSISTENT) && (flags & PKV_PLAN_SINGLE_LAUNCH))
        return fail(PKV_ERR_INVALID_ARG,
                    "paged_decode_plan_set_flags: PKV_PLAN_PERSISTENT and PKV_PLAN_SINGLE_LAUNCH "
                    "exclude each other");
    if ((flags & PKV_PLAN_SINGLE_LAUNCH) && !p->small_fits)
        return fail(PKV_ERR_UNSUPPORTED,
                    "paged_decode_plan_set_flags: max_batch x KV-head groups (%d) exceed the "
                    "thread-block clusters the device holds at once",
                    p->max_batch * p->n_groups);
    p->flags = flags;
    return PKV_OK;
}

int paged_decode_plan_mode(const pkv_plan* p, int* single_launch) {
    clear_error();
    if (!p || !single_launch) return fail(PKV_ERR_INVALID_ARG, "paged_decode_plan_mode: NULL argument");
    *single_launch = single_launch_mode(p) ? 1 : 0;
    return PKV_OK;
}

int paged_decode_plan_status(pkv_plan* p, int* status) {
    clear_error();
    if (!p || !status) return fail(PKV_ERR_INVALID_ARG, "paged_decode_plan_status: NULL argument");
    int* word = p->dev_state;
    int v = 0;
    cudaError_t e = cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && v != 0) e = cudaMemset(word, 0, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e, "paged_decode_plan_status: read");
    *status = v;
    return PKV_OK;
}

namespace {

// Shared by paged_decode_attn and paged_decode_append_attn: checks against the plan,
// optional debug checks, then the decode (+ merge) launch.
int attn_impl(const char* who, const void* q, const void* k_pool, const void* v_pool,
              const int32_t* kv_indptr, const int32_t* kv_indices, int batch, int n_qo_heads,
              int n_kv_heads, int head_dim, float sm_scale, void* out, float* lse,
              const pkv_plan* p, pkv_stream_t stream, const int32_t* slot_ids, const void* k_new,
              const void* v_new, int64_t pool_slots, const void* k_host = nullptr,
              const void* v_host = nullptr, int64_t host_slots = 0) {
    if (!p) return fail(PKV_ERR_PLAN, "%s: plan is NULL", who);
    if (!p->planned) return fail(PKV_ERR_PLAN, "%s: paged_decode_plan was not run", who);
    if (int rc = check_plan_device(who, p->device); rc != PKV_OK) return rc;
    if (n_qo_heads != p->n_qo_heads || n_kv_heads != p->n_kv_heads || head_dim != p->head_dim)
        return fail(PKV_ERR_PLAN, "%s: shape (%d, %d, %d) differs from the plan's (%d, %d, %d)", who,
                    n_qo_heads, n_kv_heads, head_dim, p->n_qo_heads, p->n_kv_heads, p->head_dim);
    if (batch != p->batch)
        return fail(PKV_ERR_PLAN, "%s: batch %d differs from the planned batch %d", who, batch,
                    p->batch);
    if (!std::isfinite(sm_scale)) return fail(PKV_ERR_INVALID_ARG, "%s: sm_scale not finite", who);
    if (batch == 0) return PKV_OK;
    if (!q || !k_pool || !v_pool || !kv_indptr || !out || (!kv_indices && p->indptr_host[batch] > 0))
        return fail(PKV_ERR_INVALID_ARG, "%s: NULL pointer argument", who);
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return fail(PKV_ERR_INVALID_ARG, "%s: q, pools and out must be 16-byte aligned", who);
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(PKV_ERR_INVALID_ARG, "%s: lse must be 4-byte aligned", who);
    const bool fused = slot_ids != nullptr;
    const bool tiered = k_host != nullptr;
    void *kh = nullptr, *vh = nullptr;
    if (tiered) {
        if (!v_host || host_slots <= 0)
            return fail(PKV_ERR_INVALID_ARG, "%s: host pools need v_host and host_slots > 0", who);
        if (!aligned16(k_host) || !aligned16(v_host))
            return fail(PKV_ERR_INVALID_ARG, "%s: host pools must be 16-byte aligned", who);
        int rc = gpu_address(who, "k_host", k_host, true, &kh);
        if (rc == PKV_OK) rc = gpu_address(who, "v_host", v_host, true, &vh);
        if (rc != PKV_OK) return rc;
        if (!aligned16(kh) || !aligned16(vh))
            return fail(PKV_ERR_INVALID_ARG, "%s: host pools must be 16-byte aligned", who);
    }
    if (fused) {
        if (!k_new || !v_new) return fail(PKV_ERR_INVALID_ARG, "%s: NULL new rows", who);
        if (!aligned16(k_new) || !aligned16(v_new))
            return fail(PKV_ERR_INVALID_ARG, "%s: new rows must be 16-byte aligned", who);
        for (int b = 0; b < batch; ++b)
            if (p->indptr_host[b + 1] == p->indptr_host[b])
                return fail(PKV_ERR_INVALID_ARG,
                            "%s: request %d has an empty context, so it has no newest token", who, b);
    }
    if (debug_checks()) {
        if (int rc = check_on_device(who, p->device,
                                     {{"q", q}, {"k_pool", k_pool}, {"v_pool", v_pool},
                                      {"kv_indptr", kv_indptr}, {"kv_indices", kv_indices},
                                      {"out", out}, {"lse", lse}, {"slot_ids", slot_ids},
                                      {"k_new", k_new}, {"v_new", v_new}});
            rc != PKV_OK)
            return rc;
        std::vector<int32_t> ip(batch + 1);
        cudaError_t e = cudaMemcpyAsync(ip.data(), kv_indptr, ip.size() * sizeof(int32_t),
                                        cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return cuda_fail(e, "debug copy of kv_indptr");
        for (int b = 0; b <= batch; ++b)
            if (ip[b] != p->indptr_host[b])
                return fail(PKV_ERR_INDEX, "%s: kv_indptr[%d] = %d but the plan has %d", who, b, ip[b],
                            p->indptr_host[b]);
        const int32_t n = ip[batch];
        std::vector<int32_t> idx(n > 0 ? n : 0);
        if (n > 0) {
            e = cudaMemcpyAsync(idx.data(), kv_indices, idx.size() * sizeof(int32_t),
                                cudaMemcpyDeviceToHost, stream);
            if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return cuda_fail(e, "debug copy of kv_indices");
            for (int32_t i = 0; i < n; ++i)
                if (idx[i] < (tiered ? -host_slots : 0) || (pool_slots > 0 && idx[i] >= pool_slots))
                    return fail(PKV_ERR_INDEX, "%s: kv_indices[%d] = %d is not a %s slot", who, i,
                                idx[i], tiered ? "pool or host-pool" : "pool");
        }
        if (p->shared) {
            // the shared-prefix kernel reads each shared slot once, from the first
            // member's list, for every member: the members must list the same ids
            const std::vector<int32_t>& sp = p->shared_indptr_host;
            const std::vector<int32_t>& sl = p->shared_len_host;
            for (size_t s = 0; s + 1 < sp.size(); ++s)
                for (int m = sp[s] + 1; m < sp[s + 1]; ++m)
                    for (int32_t j = 0; j < sl[s]; ++j)
                        if (idx[ip[m] + j] != idx[ip[sp[s]] + j])
                            return fail(PKV_ERR_INDEX,
                                        "%s: request %d lists slot %d at position %d of its shared "
                                        "prefix, but request %d (the first of its sharing group) "
                                        "lists %d there", who, m, idx[ip[m] + j], j, sp[s],
                                        idx[ip[sp[s]] + j]);
        }
        if (fused) {
            std::vector<int32_t> ids(batch);
            e = cudaMemcpyAsync(ids.data(), slot_ids, ids.size() * sizeof(int32_t),
                                cudaMemcpyDeviceToHost, stream);
            if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return cuda_fail(e, "debug copy of slot_ids");
            for (int b = 0; b < batch; ++b)
                if (ids[b] != idx[ip[b + 1] - 1])
                    return fail(PKV_ERR_INDEX,
                                "%s: slot_ids[%d] = %d is not request %d's last listed slot (%d)",
                                who, b, ids[b], b, idx[ip[b + 1] - 1]);
        }
    }
    const char* meta = static_cast<const char*>(p->dev_meta);
    DecodeArgs a{};
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.kv_indices = kv_indices;
    a.meta_header = reinterpret_cast<const int32_t*>(meta);
    a.cta_begin = reinterpret_cast<const int32_t*>(meta + p->off_cta);
    a.merges = reinterpret_cast<const Merge*>(meta + p->off_merge);
    a.part_list = reinterpret_cast<const int32_t*>(meta + p->off_list);
    a.units = reinterpret_cast<const Unit*>(meta + p->off_units);
    a.n_ctas = p->launch_ctas;
    a.shared = p->shared;
    a.early = (p->flags & PKV_PLAN_EARLY_GATHER) != 0;
    a.withhold = take_injected_stall();
    a.heads_per_cta = p->heads_per_cta;
    a.n_qo_heads = n_qo_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.sm_scale = sm_scale;
    a.out = out;
    a.lse = lse;
    a.ws_o = p->ws_o;
    a.ws_lse = p->ws_lse;
    a.merge_ctas = p->merge_ctas;
    a.status = p->dev_state;
    a.zero_row = p->zero_row;
    a.k_new = fused ? k_new : nullptr;
    a.v_new = fused ? v_new : nullptr;
    a.slot_ids = fused ? slot_ids : nullptr;
    a.k_host = tiered ? kh : nullptr;
    a.v_host = tiered ? vh : nullptr;
    a.small = p->step_small ? p->small_cs : 0;
    a.batch = batch;
    a.kv_indptr = kv_indptr;
    cudaError_t e = launch_decode(a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launch");
    return PKV_OK;
}

}  // namespace

int paged_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* kv_indptr, const int32_t* kv_indices, int batch,
                      int n_qo_heads, int n_kv_heads, int head_dim, float sm_scale, void* out,
                      float* lse, const pkv_plan* p, pkv_stream_t stream) {
    TraceRange trace("paged_decode_attn");
    clear_error();
    return attn_impl("paged_decode_attn", q, k_pool, v_pool, kv_indptr, kv_indices, batch,
                     n_qo_heads, n_kv_heads, head_dim, sm_scale, out, lse, p, stream, nullptr,
                     nullptr, nullptr, 0);
}

int paged_decode_attn_tiered(const void* q, const void* k_pool, const void* v_pool,
                             int64_t pool_slots, const void* k_host, const void* v_host,
                             int64_t host_slots, const int32_t* kv_indptr,
                             const int32_t* kv_indices, int batch, int n_qo_heads, int n_kv_heads,
                             int head_dim, float sm_scale, void* out, float* lse,
                             const pkv_plan* p, pkv_stream_t stream) {
    TraceRange trace("paged_decode_attn_tiered");
    clear_error();
    if (!k_host || !v_host)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attn_tiered: k_host and v_host are required");
    if (pool_slots <= 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attn_tiered: pool_slots must be > 0");
    return attn_impl("paged_decode_attn_tiered", q, k_pool, v_pool, kv_indptr, kv_indices, batch,
                     n_qo_heads, n_kv_heads, head_dim, sm_scale, out, lse, p, stream, nullptr,
                     nullptr, nullptr, pool_slots, k_host, v_host, host_slots);
}

int paged_decode_append_attn(const void* q, void* k_pool, void* v_pool, const int32_t* kv_indptr,
                             const int32_t* kv_indices, const int32_t* slot_ids, const void* k_new,
                             const void* v_new, int batch, int n_qo_heads, int n_kv_heads,
                             int head_dim, int64_t pool_slots, float sm_scale, void* out,
                             float* lse, const pkv_plan* p, pkv_stream_t stream) {
    TraceRange trace("paged_decode_append_attn");
    clear_error();
    if (!slot_ids) return fail(PKV_ERR_INVALID_ARG, "paged_decode_append_attn: slot_ids is NULL");
    if (pool_slots <= 0)
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_append_attn: pool_slots must be > 0");
    return attn_impl("paged_decode_append_attn", q, k_pool, v_pool, kv_indptr, kv_indices, batch,
                     n_qo_heads, n_kv_heads, head_dim, sm_scale, out, lse, p, stream, slot_ids,
                     k_new, v_new, pool_slots);
}

}  // extern "C"
