// paged_decode_attn_static: decode attention without any device allocation.
//
// paged_decode_attn needs a plan object, and creating a plan allocates device
// memory (its work list and the split workspace). Some callers cannot do that:
// an engine that has handed all free HBM to its KV pool up front, a runtime whose
// own allocator must own every device buffer, or a latency-critical path that must
// not hit cudaMalloc's implicit synchronisation. This entry point serves them. It
// plans the step on the host on every call and keeps everything the kernels need
// besides the caller's inputs and outputs — the work list, the status word, a row
// of zeros and the split-context workspace — in one file-scope __device__ array of
// kStaticScratchBytes, which every GPU that loads the library holds until the
// process exits.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress, keeps it for later calls, and
// zeroes the status word and the zero row on the call's stream, waiting for that
// (the only synchronisation the entry point does); make that first call before any
// stream capture. Every call shares the one array and leaves its contents behind,
// so calls whose kernels overlap on the GPU (two streams, or two host threads
// without ordering) race on it; the host side holds a mutex for the duration of
// each call. The status word is set by a kernel whose bounded pipeline wait ran
// out and stays set until paged_decode_attn_static_status reads and clears it.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB per GPU
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Host-side limits of the work list (the step's plan), and its staging buffer.
constexpr int kMaxCtas = 1024;
constexpr int kMaxMerges = 4096;
constexpr int kMaxUnits = 8192;
constexpr size_t kOffCta = 16;
constexpr size_t kOffMerge = (kOffCta + sizeof(int32_t) * (kMaxCtas + 1) + 255) / 256 * 256;
constexpr size_t kOffList = kOffMerge + sizeof(Merge) * kMaxMerges;
constexpr size_t kOffUnits = kOffList + sizeof(int32_t) * kMaxUnits;
constexpr size_t kMetaBytes = (kOffUnits + sizeof(Unit) * kMaxUnits + 255) / 256 * 256;
// Device layout of the array: work list | status word | zero row | partial lse | partial out
constexpr size_t kOffStatus = kMetaBytes;
constexpr size_t kOffZero = kOffStatus + 256;
constexpr size_t kOffWork = kOffZero + 256 * ((sizeof(uint16_t) * kHeadGroupElems + 255) / 256);

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_mutex;
alignas(256) unsigned char g_stage[kMetaBytes];  // host staging of the work list

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int paged_decode_attn_static(const void* q, const void* k_pool, const void* v_pool,
                                        const int32_t* kv_indptr_host, const int32_t* kv_indptr,
                                        const int32_t* kv_indices, int batch, int n_qo_heads,
                                        int n_kv_heads, int head_dim, float sm_scale, void* out,
                                        float* lse, pkv_stream_t stream) {
    TraceRange trace("paged_decode_attn_static");
    clear_error();
    if (!decode_shape_supported(n_qo_heads, n_kv_heads, head_dim))
        return fail(PKV_ERR_UNSUPPORTED,
                    "paged_decode_attn_static: unsupported shape (n_qo_heads=%d, n_kv_heads=%d, "
                    "head_dim=%d)", n_qo_heads, n_kv_heads, head_dim);
    if (batch < 0) return fail(PKV_ERR_INVALID_ARG, "paged_decode_attn_static: batch %d < 0", batch);
    if (!std::isfinite(sm_scale))
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attn_static: sm_scale not finite");
    if (batch == 0) return PKV_OK;
    if (!kv_indptr_host || !q || !k_pool || !v_pool || !kv_indptr || !out ||
        (!kv_indices && kv_indptr_host[batch] > 0))
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attn_static: NULL pointer argument");
    const auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return fail(PKV_ERR_INVALID_ARG,
                    "paged_decode_attn_static: q, pools and out must be 16-byte aligned");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(PKV_ERR_INVALID_ARG, "paged_decode_attn_static: lse must be 4-byte aligned");

    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &capturing);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "paged_decode_attn_static: stream query: %s", cudaGetErrorString(e));
    if (capturing != cudaStreamCaptureStatusNone)
        return fail(PKV_ERR_UNSUPPORTED,
                    "paged_decode_attn_static: the stream is being captured (the work list is "
                    "staged in one shared host array, which a graph would replay)");

    std::lock_guard<std::mutex> lock(g_mutex);
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "paged_decode_attn_static: device query: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PKV_ERR_UNSUPPORTED, "paged_decode_attn_static: device %d beyond %d", dev, kMaxDevices);
    if (g_scratch_addr[dev] == nullptr) {  // once per device, with that device current
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return fail(PKV_ERR_CUDA, "paged_decode_attn_static: cudaGetSymbolAddress: %s",
                        cudaGetErrorString(e));
        // the status word and the zero row start at zero; no kernel writes the
        // zero row, and only paged_decode_attn_static_status clears the status
        e = cudaMemsetAsync(static_cast<unsigned char*>(ptr) + kOffStatus, 0,
                            kOffWork - kOffStatus, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess)
            return fail(PKV_ERR_CUDA, "paged_decode_attn_static: set-up: %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = ptr;
    }
    unsigned char* scratch = static_cast<unsigned char*>(g_scratch_addr[dev]);

    const int hpc = heads_per_group(n_kv_heads, head_dim);
    const int per_sm = decode_ctas_per_sm(n_qo_heads, n_kv_heads, head_dim, hpc, false);
    if (per_sm <= 0) return fail(PKV_ERR_CUDA, "paged_decode_attn_static: occupancy query failed");
    const int ctas = sms * per_sm;
    if (ctas > kMaxCtas)
        return fail(PKV_ERR_PLAN, "paged_decode_attn_static: %d CTAs exceed the static maximum %d",
                    ctas, kMaxCtas);
    const int n_groups = n_kv_heads / hpc;
    if (int64_t(batch) * n_groups > kMaxMerges)
        return fail(PKV_ERR_PLAN,
                    "paged_decode_attn_static: batch %d x %d head groups exceeds the static maximum "
                    "of %d (request, head group) pairs", batch, n_groups, kMaxMerges);
    PlanCounts c{};
    const int max_units = std::min(kMaxUnits, plan_max_units(ctas, batch, n_groups));
    int rc = plan_compute(kv_indptr_host, batch, n_groups, ctas, decode_stage_tokens(hpc, head_dim),
                          PlanLimits{max_units, kMaxMerges, max_units}, nullptr,
                          reinterpret_cast<Unit*>(g_stage + kOffUnits),
                          reinterpret_cast<int32_t*>(g_stage + kOffCta),
                          reinterpret_cast<Merge*>(g_stage + kOffMerge),
                          reinterpret_cast<int32_t*>(g_stage + kOffList), &c);
    if (rc != PKV_OK) return rc;
    const int qheads = hpc * (n_qo_heads / n_kv_heads);
    const size_t lse_bytes = round256(sizeof(float) * size_t(c.n_partials) * qheads);
    const size_t o_bytes = sizeof(float) * size_t(c.n_partials) * qheads * head_dim;
    if (kOffWork + lse_bytes + o_bytes > kStaticScratchBytes)
        return fail(PKV_ERR_PLAN,
                    "paged_decode_attn_static: this step needs %zu bytes of scratch; the static "
                    "maximum is %zu (32 MiB)", kOffWork + lse_bytes + o_bytes, kStaticScratchBytes);
    int32_t* header = reinterpret_cast<int32_t*>(g_stage);
    header[0] = c.n_merges;
    header[1] = c.n_partials;
    header[2] = header[3] = 0;

    // Upload the work list from the (pageable) staging: the copy has read the
    // staging when cudaMemcpyAsync returns, so the next call may overwrite it. The
    // kernels that follow on the stream start only after this copy has completed,
    // which orders them after the previous call's kernels on the same stream.
    e = cudaMemcpyAsync(scratch, g_stage, kOffUnits + sizeof(Unit) * c.n_units,
                        cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "paged_decode_attn_static: upload: %s", cudaGetErrorString(e));

    DecodeArgs a{};
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.kv_indices = kv_indices;
    a.meta_header = reinterpret_cast<const int32_t*>(scratch);
    a.cta_begin = reinterpret_cast<const int32_t*>(scratch + kOffCta);
    a.merges = reinterpret_cast<const Merge*>(scratch + kOffMerge);
    a.part_list = reinterpret_cast<const int32_t*>(scratch + kOffList);
    a.shared = false;
    a.early = false;
    a.withhold = take_injected_stall();
    a.units = reinterpret_cast<const Unit*>(scratch + kOffUnits);
    a.n_ctas = ctas;
    a.heads_per_cta = hpc;
    a.n_qo_heads = n_qo_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.sm_scale = sm_scale;
    a.out = out;
    a.lse = lse;
    a.ws_lse = reinterpret_cast<float*>(scratch + kOffWork);
    a.ws_o = reinterpret_cast<float*>(scratch + kOffWork + lse_bytes);
    a.merge_ctas = sms;
    a.status = reinterpret_cast<int*>(scratch + kOffStatus);
    a.zero_row = scratch + kOffZero;
    a.k_host = a.v_host = nullptr;
    a.small = 0;
    e = launch_decode(a, stream);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "paged_decode_attn_static: launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

extern "C" int paged_decode_attn_static_status(pkv_stream_t stream, int* status) {
    clear_error();
    if (!status) return fail(PKV_ERR_INVALID_ARG, "paged_decode_attn_static_status: status is NULL");
    std::lock_guard<std::mutex> lock(g_mutex);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(PKV_ERR_CUDA, "paged_decode_attn_static_status: device query failed");
    *status = 0;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "paged_decode_attn_static_status: %s", cudaGetErrorString(e));
    if (g_scratch_addr[dev] == nullptr) return PKV_OK;  // no call has run on this device
    int* word = reinterpret_cast<int*>(static_cast<unsigned char*>(g_scratch_addr[dev]) + kOffStatus);
    int v = 0;
    e = cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && v != 0) e = cudaMemset(word, 0, sizeof v);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return fail(PKV_ERR_CUDA, "paged_decode_attn_static_status: %s", cudaGetErrorString(e));
    *status = v;
    return PKV_OK;
}
