// Split-KV paged decode attention with grouped-query heads, and its LSE merge.
//
// What is computed ("Agent-Infer: 纯 Rust 编写的高性能 LLM 推理引擎", section
// "分页 KV 缓存": batched decode over a page-size-1 token pool; "Pegainfer:
// 纯Rust+CUDA构建的LLM推理引擎", section "1. 注意力机制优化": 32 query heads share 8
// KV heads, head_dim 128; section "2. Qwen3.5的混合架构支持": head_dim 256):
// for request b and query head h (KV head g = h / G),
//     out[b,h] = softmax_j(sm_scale * q[b,h] . K[idx_j, g]) . V[idx_j, g]
//     lse[b,h] = ln sum_j exp(sm_scale * q[b,h] . K[idx_j, g]).
//
// Work decomposition: one CTA per work unit of the step's plan (a request and a
// token range of its slot list), one warp per KV head inside the CTA. A warp keeps
// the G query heads of its group in registers, so each K/V row it loads serves all
// G heads; lane i owns head_dim/32 consecutive dimensions, so one (slot, head) row
// of 256 or 512 bytes is one coalesced 8- or 16-byte-per-lane load. Slot ids are
// fetched 32 at a time (one per lane) and broadcast with shuffles; rows are loaded
// U tokens ahead of their use. Scores are reduced across the warp with xor
// shuffles, then an online softmax in base 2 (scores pre-multiplied by
// sm_scale * log2 e) rescales the fp32 accumulators. A unit that covers a whole
// context writes bf16 out and lse; a unit that covers part of one writes its
// normalised fp32 output and base-2 lse to the plan's workspace, and the merge
// kernel combines the parts: lse = log2 sum_c 2^lse_c, out = sum_c 2^(lse_c - lse)
// out_c (the log-sum-exp identity for attention over disjoint parts of a context).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// 2^x with the hardware's approximate exponential unit (ex2.approx, PTX ISA).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int VD>
struct RowVec;
template <>
struct RowVec<4> {
    using T = uint2;
};
template <>
struct RowVec<8> {
    using T = uint4;
};

// bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 bits.
template <int VD>
__device__ __forceinline__ void unpack(const typename RowVec<VD>::T& raw, float (&f)[VD]) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(&raw);
#pragma unroll
    for (int i = 0; i < VD / 2; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <int VD>
__device__ __forceinline__ typename RowVec<VD>::T pack_bf16(const float (&f)[VD]) {
    typename RowVec<VD>::T raw;
    uint32_t* w = reinterpret_cast<uint32_t*>(&raw);
#pragma unroll
    for (int i = 0; i < VD / 2; ++i) {
        __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&p);
    }
    return raw;
}

template <int D, int G, int U>
__global__ void __launch_bounds__(256)
split_kv_decode_kernel(const __nv_bfloat16* __restrict__ q,
                       const __nv_bfloat16* __restrict__ k_pool,
                       const __nv_bfloat16* __restrict__ v_pool,
                       const int32_t* __restrict__ kv_indptr,
                       const int32_t* __restrict__ kv_indices, const Unit* __restrict__ units,
                       int n_kv_heads, float scale_log2, __nv_bfloat16* __restrict__ out,
                       float* __restrict__ lse, float* __restrict__ ws_o,
                       float* __restrict__ ws_lse) {
    constexpr int VD = D / 32;
    using Vec = typename RowVec<VD>::T;
    const Unit u = units[blockIdx.x];
    const int kvh = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int hq = n_kv_heads * G;
    const int64_t row_elems = int64_t(n_kv_heads) * D;
    const int64_t ctx0 = kv_indptr[u.b];

    float qf[G][VD];
    const __nv_bfloat16* qp = q + (int64_t(u.b) * hq + kvh * G) * D + lane * VD;
#pragma unroll
    for (int g = 0; g < G; ++g) unpack<VD>(*reinterpret_cast<const Vec*>(qp + g * D), qf[g]);

    float m[G], l[G], o[G][VD];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = neg_inf();
        l[g] = 0.f;
#pragma unroll
        for (int i = 0; i < VD; ++i) o[g][i] = 0.f;
    }

    const __nv_bfloat16* kp = k_pool + kvh * D + lane * VD;
    const __nv_bfloat16* vp = v_pool + kvh * D + lane * VD;
    for (int t0 = u.tok_begin; t0 < u.tok_end; t0 += 32) {
        const int n = min(32, u.tok_end - t0);
        const int my_slot = lane < n ? __ldg(kv_indices + ctx0 + t0 + lane) : 0;
        for (int j = 0; j < n; j += U) {
            Vec kr[U], vr[U];
#pragma unroll
            for (int uu = 0; uu < U; ++uu) {
                const int64_t slot = __shfl_sync(kFull, my_slot, j + uu);
                if (j + uu < n) {
                    kr[uu] = __ldg(reinterpret_cast<const Vec*>(kp + slot * row_elems));
                    vr[uu] = __ldg(reinterpret_cast<const Vec*>(vp + slot * row_elems));
                } else {
                    kr[uu] = Vec{};
                    vr[uu] = Vec{};
                }
            }
            float s[U][G];
#pragma unroll
            for (int uu = 0; uu < U; ++uu) {
                float kf[VD];
                unpack<VD>(kr[uu], kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < VD; ++i) acc = fmaf(qf[g][i], kf[i], acc);
                    s[uu][g] = acc;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int uu = 0; uu < U; ++uu)
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        s[uu][g] += __shfl_xor_sync(kFull, s[uu][g], off);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float mx = m[g];
#pragma unroll
                for (int uu = 0; uu < U; ++uu) {
                    s[uu][g] = (j + uu < n) ? s[uu][g] * scale_log2 : neg_inf();
                    mx = fmaxf(mx, s[uu][g]);
                }
                const float alpha = ex2(m[g] - mx);
                m[g] = mx;
                l[g] *= alpha;
#pragma unroll
                for (int i = 0; i < VD; ++i) o[g][i] *= alpha;
#pragma unroll
                for (int uu = 0; uu < U; ++uu) {
                    s[uu][g] = ex2(s[uu][g] - mx);
                    l[g] += s[uu][g];
                }
            }
#pragma unroll
            for (int uu = 0; uu < U; ++uu) {
                float vf[VD];
                unpack<VD>(vr[uu], vf);
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int i = 0; i < VD; ++i) o[g][i] = fmaf(s[uu][g], vf[i], o[g][i]);
            }
        }
    }

#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int h = kvh * G + g;
        const bool empty = (l[g] == 0.f);
        const float inv = empty ? 0.f : 1.f / l[g];
        const float lse2 = empty ? neg_inf() : m[g] + __log2f(l[g]);
        float r[VD];
#pragma unroll
        for (int i = 0; i < VD; ++i) r[i] = o[g][i] * inv;
        if (u.partial < 0) {
            const int64_t oh = int64_t(u.b) * hq + h;
            *reinterpret_cast<Vec*>(out + oh * D + lane * VD) = pack_bf16<VD>(r);
            if (lse != nullptr && lane == 0) lse[oh] = lse2 * kLn2;
        } else {
            const int64_t ph = int64_t(u.partial) * hq + h;
            float* dst = ws_o + ph * D + lane * VD;
#pragma unroll
            for (int i = 0; i < VD; i += 4)
                *reinterpret_cast<float4*>(dst + i) = make_float4(r[i], r[i + 1], r[i + 2], r[i + 3]);
            if (lane == 0) ws_lse[ph] = lse2;
        }
    }
}

// One CTA per split request; warp w merges query heads w, w + 4, ...
template <int D>
__global__ void __launch_bounds__(128)
lse_merge_kernel(const Merge* __restrict__ merges, int hq, const float* __restrict__ ws_o,
                 const float* __restrict__ ws_lse, __nv_bfloat16* __restrict__ out,
                 float* __restrict__ lse) {
    constexpr int VD = D / 32;
    using Vec = typename RowVec<VD>::T;
    const Merge mg = merges[blockIdx.x];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int h = warp; h < hq; h += blockDim.x / 32) {
        float mx = neg_inf();
        for (int c = 0; c < mg.count; ++c) mx = fmaxf(mx, ws_lse[int64_t(mg.first + c) * hq + h]);
        float sum = 0.f;
        for (int c = 0; c < mg.count; ++c) sum += ex2(ws_lse[int64_t(mg.first + c) * hq + h] - mx);
        const float total = mx + __log2f(sum);
        float acc[VD];
#pragma unroll
        for (int i = 0; i < VD; ++i) acc[i] = 0.f;
        for (int c = 0; c < mg.count; ++c) {
            const int64_t ph = int64_t(mg.first + c) * hq + h;
            const float w = ex2(ws_lse[ph] - total);
            const float* src = ws_o + ph * D + lane * VD;
#pragma unroll
            for (int i = 0; i < VD; i += 4) {
                const float4 x = *reinterpret_cast<const float4*>(src + i);
                acc[i] = fmaf(w, x.x, acc[i]);
                acc[i + 1] = fmaf(w, x.y, acc[i + 1]);
                acc[i + 2] = fmaf(w, x.z, acc[i + 2]);
                acc[i + 3] = fmaf(w, x.w, acc[i + 3]);
            }
        }
        const int64_t oh = int64_t(mg.b) * hq + h;
        *reinterpret_cast<Vec*>(out + oh * D + lane * VD) = pack_bf16<VD>(acc);
        if (lse != nullptr && lane == 0) lse[oh] = total * kLn2;
    }
}

template <int D, int G>
cudaError_t launch_shape(const DecodeArgs& a, cudaStream_t stream) {
    constexpr int U = 4;
    if (a.n_units > 0) {
        split_kv_decode_kernel<D, G, U><<<a.n_units, 32 * a.n_kv_heads, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k_pool),
            static_cast<const __nv_bfloat16*>(a.v_pool), a.kv_indptr, a.kv_indices, a.units,
            a.n_kv_heads, a.sm_scale * kLog2e, static_cast<__nv_bfloat16*>(a.out), a.lse,
            a.ws_o, a.ws_lse);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (a.n_merges > 0) {
        lse_merge_kernel<D><<<a.n_merges, 128, 0, stream>>>(
            a.merges, a.n_qo_heads, a.ws_o, a.ws_lse, static_cast<__nv_bfloat16*>(a.out), a.lse);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

template <int D, int G>
int occupancy_shape(int n_kv_heads) {
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, split_kv_decode_kernel<D, G, 4>,
                                                      32 * n_kv_heads, 0) != cudaSuccess)
        return 0;
    return blocks;
}

#define PKV_DISPATCH(D_, FN, ...)                         \
    switch (G) {                                          \
        case 1: return FN<D_, 1>(__VA_ARGS__);            \
        case 2: return FN<D_, 2>(__VA_ARGS__);            \
        case 4: return FN<D_, 4>(__VA_ARGS__);            \
        case 8: return FN<D_, 8>(__VA_ARGS__);            \
        default: break;                                   \
    }

}  // namespace

bool decode_shape_supported(int n_qo_heads, int n_kv_heads, int head_dim) {
    if (n_kv_heads <= 0 || n_qo_heads <= 0 || n_qo_heads % n_kv_heads != 0) return false;
    const int G = n_qo_heads / n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return false;
    if (head_dim != 128 && head_dim != 256) return false;
    return n_kv_heads <= 8;
}

int decode_ctas_per_sm(int n_qo_heads, int n_kv_heads, int head_dim) {
    if (!decode_shape_supported(n_qo_heads, n_kv_heads, head_dim)) return 0;
    const int G = n_qo_heads / n_kv_heads;
    if (head_dim == 128) {
        PKV_DISPATCH(128, occupancy_shape, n_kv_heads)
    } else {
        PKV_DISPATCH(256, occupancy_shape, n_kv_heads)
    }
    return 0;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    const int G = a.n_qo_heads / a.n_kv_heads;
    if (a.head_dim == 128) {
        PKV_DISPATCH(128, launch_shape, a, stream)
    } else {
        PKV_DISPATCH(256, launch_shape, a, stream)
    }
    return cudaErrorInvalidValue;
}

}  // namespace pkv
