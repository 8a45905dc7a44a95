// Host KV tier: move pool rows between HBM and pinned host memory.
//
// "Agent-Infer: 纯 Rust 编写的高性能 LLM 推理引擎", section "CPU 卸载": when HBM is full,
// older KV blocks move to CPU memory and are prefetched back to the GPU when a request
// needs them again, so a context can outgrow device memory. With page size 1 a "block"
// is a set of token rows, so the tier is two row scatters between a device pool
// [pool_slots, n_kv_heads, head_dim] and a host pool of the same row size:
//   offload : host[host_slots[i]] = dev[dev_slots[i]]
//   prefetch: dev[dev_slots[i]]   = host[host_slots[i]]
// for K and V. On GB300 the host pool is Grace memory reached over NVLink-C2C; the
// kernel reads and writes it directly (the pinned buffer is mapped into the GPU's
// address space), 16 bytes per thread, several vectors in flight per thread so the
// link sees enough outstanding requests. Each row is 2 x n_kv_heads x head_dim bytes
// of K, the same of V, contiguous on both sides.
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kTierThreads = 256;
constexpr int kTierUnroll = 4;

__global__ void __launch_bounds__(kTierThreads)
kv_tier_copy_kernel(const uint4* __restrict__ k_src, const uint4* __restrict__ v_src,
                    const int32_t* __restrict__ src_slots, uint4* __restrict__ k_dst,
                    uint4* __restrict__ v_dst, const int32_t* __restrict__ dst_slots, int64_t n,
                    int row_vecs) {
    const int64_t per_pool = n * row_vecs;
    const int64_t total = 2 * per_pool;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t base = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; base < total;
         base += stride * kTierUnroll) {
        uint4 val[kTierUnroll];
        int64_t dst_index[kTierUnroll];  // -1: nothing to store
        bool dst_v[kTierUnroll];
#pragma unroll
        for (int u = 0; u < kTierUnroll; ++u) {  // all loads first
            const int64_t i = base + u * stride;
            dst_index[u] = -1;
            dst_v[u] = false;
            if (i < total) {
                const bool is_v = i >= per_pool;
                const int64_t j = is_v ? i - per_pool : i;
                const int64_t row = j / row_vecs, col = j - row * row_vecs;
                const int64_t s = __ldg(src_slots + row), d = __ldg(dst_slots + row);
                val[u] = (is_v ? v_src : k_src)[s * row_vecs + col];
                dst_index[u] = d * row_vecs + col;
                dst_v[u] = is_v;
            }
        }
#pragma unroll
        for (int u = 0; u < kTierUnroll; ++u)
            if (dst_index[u] >= 0) (dst_v[u] ? v_dst : k_dst)[dst_index[u]] = val[u];
    }
}

}  // namespace

cudaError_t launch_tier_copy(const void* k_src, const void* v_src, const int32_t* src_slots,
                             void* k_dst, void* v_dst, const int32_t* dst_slots, int64_t n,
                             int row_bytes, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int row_vecs = row_bytes / 16;
    const int64_t total = 2 * n * row_vecs;
    int64_t blocks = (total + int64_t(kTierThreads) * kTierUnroll - 1) / (int64_t(kTierThreads) * kTierUnroll);
    const int64_t cap = int64_t(sms) * 8;
    blocks = blocks < cap ? blocks : cap;
    kv_tier_copy_kernel<<<static_cast<unsigned>(blocks), kTierThreads, 0, stream>>>(
        static_cast<const uint4*>(k_src), static_cast<const uint4*>(v_src), src_slots,
        static_cast<uint4*>(k_dst), static_cast<uint4*>(v_dst), dst_slots, n, row_vecs);
    return cudaGetLastError();
}

}  // namespace pkv
