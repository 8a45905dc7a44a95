// KV append: scatter this step's new K/V rows into their token-pool slots.
//
// The pool has page size 1 ("Agent-Infer: 纯 Rust 编写的高性能 LLM 推理引擎", section
// "分页 KV 缓存"), so a decode step writes exactly one pool row per request and
// layer: row `slot_ids[i]` of K and of V receives new row i. A row holds all KV
// heads of one token (n_kv_heads * head_dim bf16, 2 KB for 8 x 128), contiguous in
// both the source and the pool, so the copy is 16-byte vectors: consecutive
// threads move consecutive vectors of one row (fully coalesced 2 KB reads and
// writes), and one grid-stride loop covers K and V, each thread loading four
// vectors before it stores them (a prefill chunk appends thousands of rows, and
// the loads in flight set the rate). Pure HBM traffic: 2 * n * row bytes read and
// written, plus 4 bytes of slot id per row.
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256)
kvpool_append_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                     const int32_t* __restrict__ slot_ids, const uint4* __restrict__ k_new,
                     const uint4* __restrict__ v_new, int64_t n, int row_vecs) {
    // Launched with programmatic stream serialisation: let the next kernel be
    // scheduled now, but touch nothing until the previous kernel has finished
    // (its readers of the pool, or its producers of the new rows).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int kUnroll = 4;
    const int64_t per_pool = n * row_vecs;
    const int64_t total = 2 * per_pool;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i0 = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i0 < total;
         i0 += kUnroll * stride) {
        uint4 val[kUnroll];
        int64_t off[kUnroll];  // vector index in its pool; -1: past the end
        bool to_v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            to_v[u] = i >= per_pool;
            off[u] = -1;
            if (i < total) {
                const int64_t j = to_v[u] ? i - per_pool : i;
                const int64_t row = j / row_vecs;
                val[u] = to_v[u] ? __ldg(v_new + j) : __ldg(k_new + j);
                off[u] = int64_t(__ldg(slot_ids + row)) * row_vecs + (j - row * row_vecs);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (off[u] >= 0) (to_v[u] ? v_pool : k_pool)[off[u]] = val[u];
    }
}

}  // namespace

cudaError_t launch_append(void* k_pool, void* v_pool, const int32_t* slot_ids,
                          const void* k_new, const void* v_new, int64_t n, int row_bytes,
                          cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const int row_vecs = row_bytes / 16;
    const int64_t total = 2 * n * row_vecs;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    // At most four CTAs per SM: with PDL they can all be resident (and waiting)
    // next to the previous kernel's CTAs; the loop covers the rest.
    static int sms_of[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (sms_of[dev] == 0 &&
        cudaDeviceGetAttribute(&sms_of[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms_of[dev] = 152;
    blocks = (blocks + 3) / 4;  // four vectors per thread and pass
    blocks = blocks < 4 * sms_of[dev] ? blocks : 4 * sms_of[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kvpool_append_kernel, static_cast<uint4*>(k_pool),
                              static_cast<uint4*>(v_pool), slot_ids,
                              static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                              n, row_vecs);
}

}  // namespace pkv
