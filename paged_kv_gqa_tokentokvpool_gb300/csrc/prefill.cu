// Chunked-prefill attention over the page-size-1 token pool.
//
// What is computed ("Agent-Infer: 纯 Rust 编写的高性能 LLM 推理引擎", section
// "连续批处理": long prefills run in chunks of 512 tokens, 64 while decodes are
// running, between decode steps; the pool is the same TokenToKVPool as for decode,
// section "分页 KV 缓存"): a chunk is a request's newest C tokens, already appended,
// so they are the last C of its L listed slots. Query c of the chunk sits at list
// position p = L - C + c and attends causally to entries 0 .. p:
//     out[i,h] = softmax_{j<=p}(sm_scale * q[i,h] . K[idx_j, g]) . V[idx_j, g]
//     lse[i,h] = ln sum_{j<=p} exp(sm_scale * q[i,h] . K[idx_j, g])
// with g = h / G (grouped-query attention, "Pegainfer: 纯Rust+CUDA构建的LLM推理引擎",
// section "1. 注意力机制优化").
//
// Design for sm_103a. Unlike decode, every K/V row here serves the 64 / G query
// tokens of a tile times G heads, so the work is a dense contraction per KV head:
//  * One CTA per work unit (request, KV head, tile of 64 / G chunk tokens): its 64
//    query rows (token, head) are four 16-row warp tiles. The plan orders units
//    longest causal range first, so the grid drains evenly.
//  * The unit's q rows are staged once in shared memory and then held as mma
//    fragments in registers for the whole unit; the request's slot rows
//    of that KV head stream through a ring of 32-token K/V tiles gathered with
//    16-byte cp.async (each thread copies whole 16-byte pieces of scattered pool
//    rows; a stage's slot ids are loaded one iteration ahead of its copies).
//  * Tensor cores, FlashAttention-2 orientation: per warp and tile
//      S[16 x 32] = Q[16 x D] K^T    and    O[16 x D] += P[16 x 32] V[32 x D]
//    with mma.sync m16n8k16 (bf16, fp32 accumulate). K fragments come by
//    ldmatrix, V by ldmatrix.trans, and the probabilities pass from the S
//    accumulators to the A operand of P V in registers.
//  * Online softmax in base 2 with fp32 state per row; the causal mask compares
//    each token's list position with the row's query position, and the ring
//    stops at the unit's last query position.
//  * No spin-waits: the ring is cp.async groups and CTA barriers.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <new>
#include <vector>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

using namespace ptx;

constexpr int kPfWarps = 4;
constexpr int kPfThreads = 32 * kPfWarps;
constexpr int kPfRows = 16 * kPfWarps;  // query rows (token, head) per CTA
constexpr int kPfKvTile = 32;           // KV tokens per ring stage
constexpr int kPfPad = 8;               // bf16 padding per shared row: conflict-free ldmatrix
constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// One work unit: query tokens q_row0 .. q_row0 + n_q - 1 (rows of q/out) of one
// request, KV head g, over list entries kv_lo .. kv_hi - 1 of the request's slot
// list (which starts at kv_begin in kv_indices). The unit's first query sits at list
// position pos0. part < 0: the unit covers every entry its queries see and writes
// out/lse; otherwise it is one piece of a split range, kv_lo <= pos0 and kv_lo a
// multiple of the ring tile, and writes its 64 rows' normalised fp32 output and
// base-2 lse to workspace block `part`.
struct PfUnit {
    int32_t part, g, q_row0, n_q, kv_begin, pos0, kv_lo, kv_hi;
};
static_assert(sizeof(PfUnit) == 32, "unit record");

// The pieces of one split unit: workspace blocks first .. first + count - 1, for
// query tokens q_row0 .. q_row0 + n_q - 1 and KV head g.
struct PfMerge {
    int32_t q_row0, n_q, g, first, count, pad0, pad1, pad2;
};
static_assert(sizeof(PfMerge) == 32, "merge record");

struct PfArgs {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* kv_indices;
    const PfUnit* units;
    int n_qo_heads;
    int n_kv_heads;
    float scale_log2;  // sm_scale * log2(e)
    void* out;
    float* lse;
    float* ws_o;       // [blocks, 64, head_dim] partial outputs of split units
    float* ws_lse;     // [blocks, 64] their base-2 lse
    const PfMerge* merges;
    int n_merges;
};

template <int D, int G>
struct PfCfg {
    static constexpr int kStages = D == 128 ? 3 : 2;   // 2 CTAs per SM at D = 256
    static constexpr int kPitch = D + kPfPad;          // shared row pitch (bf16)
    static constexpr int kQBytes = kPfRows * kPitch * 2;
    static constexpr int kKvBytes = kPfKvTile * kPitch * 2;  // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kKvBytes;
    static constexpr int kSmem = kQBytes + kStages * kStageBytes;
    static constexpr int kChunks = D / 8;                  // 16-byte pieces per row
    static constexpr int kPieces = kPfKvTile * kChunks / kPfThreads;  // per thread, K (or V)
    static constexpr int kKSteps = D / 16;
    static constexpr int kNT = kPfKvTile / 8;              // 8-token column tiles of S
    static constexpr int kDT = D / 8;                      // 8-dim column tiles of O
    static_assert(kPieces * kPfThreads == kPfKvTile * kChunks, "ring pieces");
};

// ---------------------------------------------------------------------------
// kernel
// ---------------------------------------------------------------------------

// Slot ids of the pieces this thread copies for KV tile `tile` (-1 past the range).
template <int D, int G>
__device__ __forceinline__ void load_tile_slots(const PfArgs& a, const PfUnit& un, int tile,
                                                int (&slot)[PfCfg<D, G>::kPieces]) {
    using C = PfCfg<D, G>;
#pragma unroll
    for (int i = 0; i < C::kPieces; ++i) {
        const int tok = (threadIdx.x + i * kPfThreads) / C::kChunks;
        const int j = tile * kPfKvTile + tok;
        slot[i] = j < un.kv_hi ? __ldg(a.kv_indices + un.kv_begin + j) : -1;
    }
}

// Issue the cp.async copies of KV tile pieces into ring stage `st` (tokens past the
// unit's range are zero-filled).
template <int D, int G>
__device__ __forceinline__ void issue_tile(const PfArgs& a, const PfUnit& un, uint8_t* smem,
                                           int st, const int (&slot)[PfCfg<D, G>::kPieces]) {
    using C = PfCfg<D, G>;
    const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_pool);
    const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_pool);
    uint8_t* sk = smem + C::kQBytes + st * C::kStageBytes;
    uint8_t* sv = sk + C::kKvBytes;
#pragma unroll
    for (int i = 0; i < C::kPieces; ++i) {
        const int c = threadIdx.x + i * kPfThreads;
        const int tok = c / C::kChunks, part = c % C::kChunks;
        const bool valid = slot[i] >= 0;
        const int64_t off = (int64_t(valid ? slot[i] : 0) * a.n_kv_heads + un.g) * D + part * 8;
        const int soff = (tok * C::kPitch + part * 8) * 2;
        cp_async16(smem_u32(sk + soff), kp + off, valid);
        cp_async16(smem_u32(sv + soff), vp + off, valid);
    }
}

template <int D, int G>
__global__ void __launch_bounds__(kPfThreads) paged_prefill_kernel(const PfArgs a) {
    using C = PfCfg<D, G>;
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();
    const PfUnit un = a.units[blockIdx.x];  // plan data: read before the wait
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    // q, the pools and their indices may come from the previous kernel
    pdl_wait();

    // ---- the unit's q rows (row r: chunk token r / G, head r % G) -> shared memory
    {
        const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
        for (int c = tid; c < kPfRows * C::kChunks; c += kPfThreads) {
            const int r = c / C::kChunks, part = c % C::kChunks;
            const int t = r / G, h = r % G;
            const bool valid = t < un.n_q;
            const int64_t off =
                (int64_t(un.q_row0 + (valid ? t : 0)) * a.n_qo_heads + un.g * G + h) * D + part * 8;
            cp_async16(smem_u32(smem + (r * C::kPitch + part * 8) * 2), q + off, valid);
        }
    }
    // ---- ring prologue: the range's tiles 0 .. kStages - 2, and the slot ids of the
    // next one (ring index i holds list tile t0 + i)
    const int t0 = un.kv_lo / kPfKvTile;
    const int n_tiles = (un.kv_hi + kPfKvTile - 1) / kPfKvTile - t0;
    int slot[C::kPieces];
#pragma unroll
    for (int s = 0; s < C::kStages - 1; ++s) {
        if (s < n_tiles) {
            load_tile_slots<D, G>(a, un, t0 + s, slot);
            issue_tile<D, G>(a, un, smem, s, slot);
        }
        cp_async_commit();  // one group per tile (the first also holds q)
    }
    if (C::kStages - 1 < n_tiles) load_tile_slots<D, G>(a, un, t0 + C::kStages - 1, slot);

    // per lane: rows lo = 16 warp + g8 and hi = lo + 8 of the unit's 64
    const int r_lo = 16 * warp + g8, r_hi = r_lo + 8;
    const int pos_lo = un.pos0 + r_lo / G, pos_hi = un.pos0 + r_hi / G;
    float m_lo = neg_inf(), m_hi = neg_inf(), l_lo = 0.f, l_hi = 0.f;
    float o[C::kDT][4];
#pragma unroll
    for (int dt = 0; dt < C::kDT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;

    // ldmatrix lane addresses
    const uint32_t q_addr = smem_u32(smem) +
                            ((16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1)) * C::kPitch +
                             8 * (lane >> 4)) * 2;
    const int mi = lane >> 3;
    const uint32_t k_off = ((8 * (mi >> 1) + (lane & 7)) * C::kPitch + 8 * (mi & 1)) * 2;
    const uint32_t v_off = ((8 * (mi & 1) + (lane & 7)) * C::kPitch + 8 * (mi >> 1)) * 2;

    uint32_t qf[C::kKSteps][4];  // this warp's q rows as A fragments, loaded once
    bool q_loaded = false;
    for (int n = 0; n < n_tiles; ++n) {
        // copies of tile n + kStages - 1 (slot ids loaded last iteration), then the
        // slot ids of the tile after it
        const int ahead = n + C::kStages - 1;
        if (ahead < n_tiles) issue_tile<D, G>(a, un, smem, ahead % C::kStages, slot);
        cp_async_commit();
        if (ahead + 1 < n_tiles) load_tile_slots<D, G>(a, un, t0 + ahead + 1, slot);
        cp_async_wait<C::kStages - 1>();  // tile n (and q) have landed for this thread
        __syncthreads();            // ... and for every thread
        if (!q_loaded) {
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) ldsm_x4(q_addr + ks * 32, qf[ks]);
            q_loaded = true;
        }

        const int st = n % C::kStages;
        const uint32_t sk = smem_u32(smem) + C::kQBytes + st * C::kStageBytes;
        const uint32_t sv = sk + C::kKvBytes;
        // S = Q K^T for this warp's 16 rows and the tile's 32 tokens
        float s[C::kNT][4];
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
#pragma unroll
            for (int np = 0; np < C::kNT / 2; ++np) {
                uint32_t kb[4];
                ldsm_x4(sk + k_off + (16 * np * C::kPitch + 16 * ks) * 2, kb);
                mma_bf16(s[2 * np], qf[ks], kb[0], kb[1]);
                mma_bf16(s[2 * np + 1], qf[ks], kb[2], kb[3]);
            }
        }
        // causal mask and online softmax (base 2); token j of the tile is list
        // position (t0 + n) * 32 + 8 nt + 2 t4 (+1); c[0..1] are row lo, c[2..3] row hi
        const int j0 = (t0 + n) * kPfKvTile + 2 * t4;
        float mx_lo = neg_inf(), mx_hi = neg_inf();
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt) {
            const int j = j0 + 8 * nt;
            s[nt][0] = j <= pos_lo ? s[nt][0] * a.scale_log2 : neg_inf();
            s[nt][1] = j + 1 <= pos_lo ? s[nt][1] * a.scale_log2 : neg_inf();
            s[nt][2] = j <= pos_hi ? s[nt][2] * a.scale_log2 : neg_inf();
            s[nt][3] = j + 1 <= pos_hi ? s[nt][3] * a.scale_log2 : neg_inf();
            mx_lo = fmaxf(mx_lo, fmaxf(s[nt][0], s[nt][1]));
            mx_hi = fmaxf(mx_hi, fmaxf(s[nt][2], s[nt][3]));
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(kFullMask, mx_lo, off));
            mx_hi = fmaxf(mx_hi, __shfl_xor_sync(kFullMask, mx_hi, off));
        }
        // every row sees the range's first entry (kv_lo <= pos0), so the maxima are
        // finite from the range's first tile on
        const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
        const float al_lo = ex2(m_lo - mn_lo), al_hi = ex2(m_hi - mn_hi);
        m_lo = mn_lo;
        m_hi = mn_hi;
        float sum_lo = 0.f, sum_hi = 0.f;
        uint32_t pa[C::kNT / 2][4];
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt) {
            const float p0 = ex2(s[nt][0] - mn_lo), p1 = ex2(s[nt][1] - mn_lo);
            const float p2 = ex2(s[nt][2] - mn_hi), p3 = ex2(s[nt][3] - mn_hi);
            sum_lo += p0 + p1;
            sum_hi += p2 + p3;
            // S accumulators of column tiles 2k, 2k+1 form the A operand of k-step k
            pa[nt >> 1][(nt & 1) * 2] = pack_bf16x2(p0, p1);
            pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p2, p3);
        }
        l_lo = fmaf(l_lo, al_lo, sum_lo);
        l_hi = fmaf(l_hi, al_hi, sum_hi);
#pragma unroll
        for (int dt = 0; dt < C::kDT; ++dt) {
            o[dt][0] *= al_lo;
            o[dt][1] *= al_lo;
            o[dt][2] *= al_hi;
            o[dt][3] *= al_hi;
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < C::kNT / 2; ++kk) {
#pragma unroll
            for (int dp = 0; dp < C::kDT / 2; ++dp) {
                uint32_t vb[4];
                ldsm_x4_trans(sv + v_off + (16 * kk * C::kPitch + 16 * dp) * 2, vb);
                mma_bf16(o[2 * dp], pa[kk], vb[0], vb[1]);
                mma_bf16(o[2 * dp + 1], pa[kk], vb[2], vb[3]);
            }
        }
        __syncthreads();  // the stage is read before the next iteration refills it
    }
    cp_async_wait<0>();

    // ---- epilogue: rows lo / hi of this lane
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        l_lo += __shfl_xor_sync(kFullMask, l_lo, off);
        l_hi += __shfl_xor_sync(kFullMask, l_hi, off);
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = half ? r_hi : r_lo;
        const int t = r / G, h = r % G;
        if (t >= un.n_q) continue;
        const float lt = half ? l_hi : l_lo;
        const float inv = 1.f / lt;
        const float lse2 = (half ? m_hi : m_lo) + __log2f(lt);
        if (un.part >= 0) {  // a piece of a split range: fp32 partial result
            const int64_t wrow = int64_t(un.part) * kPfRows + r;
            float* dst = a.ws_o + wrow * D + 2 * t4;
#pragma unroll
            for (int dt = 0; dt < C::kDT; ++dt)
                *reinterpret_cast<float2*>(dst + 8 * dt) =
                    make_float2(o[dt][2 * half] * inv, o[dt][2 * half + 1] * inv);
            if (t4 == 0) a.ws_lse[wrow] = lse2;
            continue;
        }
        const int64_t row = int64_t(un.q_row0 + t) * a.n_qo_heads + un.g * G + h;
        __nv_bfloat16* dst = out + row * D + 2 * t4;
#pragma unroll
        for (int dt = 0; dt < C::kDT; ++dt)
            *reinterpret_cast<uint32_t*>(dst + 8 * dt) =
                pack_bf16x2(o[dt][2 * half] * inv, o[dt][2 * half + 1] * inv);
        if (a.lse != nullptr && t4 == 0) a.lse[row] = lse2 * kLn2;
    }
}

// Log-sum-exp merge of split units: one warp per (merge record, row of its 64),
// lanes over head_dim, every piece's loads issued before any is used:
//     lse = log2 sum_c 2^lse_c,   out = sum_c 2^(lse_c - lse) out_c
constexpr int kPfMergeWarps = 4;
constexpr int kPfMaxPieces = 16;  // pieces per split unit (the planner's cap)

template <int D, int G>
__global__ void __launch_bounds__(32 * kPfMergeWarps) prefill_merge_kernel(const PfArgs a) {
    pdl_launch_dependents();
    constexpr int kVD = D / 32;  // dims per lane
    const int lane = threadIdx.x & 31;
    const int w = blockIdx.x * kPfMergeWarps + (threadIdx.x >> 5);
    if (w >= a.n_merges * kPfRows) return;
    const PfMerge mg = a.merges[w / kPfRows];  // plan data
    const int r = w % kPfRows, t = r / G, h = r % G;
    if (t >= mg.n_q) return;
    pdl_wait();  // the pieces come from the kernel before
    float x[kPfMaxPieces][kVD], xl[kPfMaxPieces];
#pragma unroll
    for (int c = 0; c < kPfMaxPieces; ++c) {
        if (c < mg.count) {
            const int64_t wrow = int64_t(mg.first + c) * kPfRows + r;
            xl[c] = __ldcg(a.ws_lse + wrow);
#pragma unroll
            for (int i = 0; i < kVD; i += 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(a.ws_o + wrow * D + lane * kVD + i));
                x[c][i] = v.x;
                x[c][i + 1] = v.y;
                x[c][i + 2] = v.z;
                x[c][i + 3] = v.w;
            }
        }
    }
    float mx = neg_inf();
#pragma unroll
    for (int c = 0; c < kPfMaxPieces; ++c)
        if (c < mg.count) mx = fmaxf(mx, xl[c]);
    float sum = 0.f, acc[kVD];
#pragma unroll
    for (int i = 0; i < kVD; ++i) acc[i] = 0.f;
#pragma unroll
    for (int c = 0; c < kPfMaxPieces; ++c) {
        if (c < mg.count) {
            const float wgt = ex2(xl[c] - mx);
            sum += wgt;
#pragma unroll
            for (int i = 0; i < kVD; ++i) acc[i] = fmaf(wgt, x[c][i], acc[i]);
        }
    }
    const float inv = 1.f / sum;
    const int64_t row = int64_t(mg.q_row0 + t) * a.n_qo_heads + mg.g * G + h;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + row * D + lane * kVD;
#pragma unroll
    for (int i = 0; i < kVD; i += 2)
        *reinterpret_cast<uint32_t*>(dst + i) = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
    if (a.lse != nullptr && lane == 0) a.lse[row] = (mx + __log2f(sum)) * kLn2;
}

template <int D, int G>
cudaError_t prefill_prepare() {
    static const cudaError_t attr =
        cudaFuncSetAttribute(paged_prefill_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PfCfg<D, G>::kSmem);
    return attr;
}

// Resident CTAs per SM of the prefill kernel (0 on error).
template <int D, int G>
int prefill_occupancy() {
    if (prefill_prepare<D, G>() != cudaSuccess) return 0;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, paged_prefill_kernel<D, G>,
                                                      kPfThreads, PfCfg<D, G>::kSmem) != cudaSuccess)
        return 0;
    return blocks;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, const PfArgs& a,
                       cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    void* args[] = {const_cast<PfArgs*>(&a)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

template <int D, int G>
cudaError_t launch_prefill(const PfArgs& a, int n_units, cudaStream_t stream) {
    cudaError_t e = prefill_prepare<D, G>();
    if (e != cudaSuccess || n_units == 0) return e;
    e = launch_pdl(reinterpret_cast<const void*>(&paged_prefill_kernel<D, G>), dim3(n_units),
                   dim3(kPfThreads), PfCfg<D, G>::kSmem, a, stream);
    if (e != cudaSuccess || a.n_merges == 0) return e;
    const int warps = a.n_merges * kPfRows;
    return launch_pdl(reinterpret_cast<const void*>(&prefill_merge_kernel<D, G>),
                      dim3((warps + kPfMergeWarps - 1) / kPfMergeWarps), dim3(32 * kPfMergeWarps),
                      0, a, stream);
}

// Calls FN<D, G>::run(args...) for the runtime shape.
template <template <int, int> class FN, typename... Args>
auto prefill_dispatch(int head_dim, int group, Args&&... args) -> decltype(FN<128, 1>::run(args...)) {
#define PKV_PF(D_)                                          \
    switch (group) {                                        \
        case 1: return FN<D_, 1>::run(args...);             \
        case 2: return FN<D_, 2>::run(args...);             \
        case 4: return FN<D_, 4>::run(args...);             \
        case 8: return FN<D_, 8>::run(args...);             \
        default: break;                                     \
    }
    if (head_dim == 128) { PKV_PF(128) }
    if (head_dim == 256) { PKV_PF(256) }
#undef PKV_PF
    return FN<128, 1>::unsupported();
}

template <int D, int G>
struct PfLaunchFn {
    static cudaError_t run(const PfArgs& a, int n_units, cudaStream_t s) {
        return launch_prefill<D, G>(a, n_units, s);
    }
    static cudaError_t unsupported() { return cudaErrorInvalidValue; }
};
template <int D, int G>
struct PfOccupancyFn {
    static int run() { return prefill_occupancy<D, G>(); }
    static int unsupported() { return 0; }
};

bool prefill_shape_supported(int n_qo_heads, int n_kv_heads, int head_dim) {
    if (n_kv_heads <= 0 || n_qo_heads <= 0 || n_qo_heads % n_kv_heads != 0) return false;
    const int G = n_qo_heads / n_kv_heads;
    return (G == 1 || G == 2 || G == 4 || G == 8) && (head_dim == 128 || head_dim == 256);
}

int pf_cuda_fail(cudaError_t e, const char* what) {
    return fail(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct PfPlanCounts {
    int n_units, n_merges, n_blocks;
};

// The prefill planner (host only, no CUDA call): checks the offsets and fills
// units[0 .. n_units) and merges[0 .. n_merges).
//  1. one unit per (request, tile of tile_tokens chunk tokens, KV head), over every
//     list entry its queries see;
//  2. with fewer such units than split_target, each long range is cut at ring-tile
//     boundaries at or below its first query's position (every query then sees
//     every entry of every piece but the last) into at most kPfMaxPieces pieces of
//     about equal length; each piece writes workspace block `part`, and a merge
//     record names the unit's consecutive blocks;
//  3. units are listed longest range first.
int prefill_plan_compute(const char* who, const int32_t* qo, const int32_t* kv, int batch,
                         int tile_tokens, int n_kv_heads, int split_target, PfUnit* units,
                         int max_units, PfMerge* merges, int max_merges, int max_blocks,
                         PfPlanCounts* out) {
    if (batch > 0 && (qo[0] != 0 || kv[0] != 0))
        return fail(PKV_ERR_INVALID_ARG, "%s: offsets must start at 0", who);
    for (int b = 0; b < batch; ++b) {
        const int C = qo[b + 1] - qo[b];
        const int L = kv[b + 1] - kv[b];
        if (C < 0 || L < 0)
            return fail(PKV_ERR_INVALID_ARG, "%s: offsets decrease at request %d", who, b);
        if (C > L)
            return fail(PKV_ERR_INVALID_ARG,
                        "%s: request %d has a chunk of %d tokens but lists only %d slots", who, b,
                        C, L);
    }
    std::vector<PfUnit> tiles;
    int64_t total_tiles = 0;
    for (int b = 0; b < batch; ++b) {
        const int C = qo[b + 1] - qo[b];
        const int L = kv[b + 1] - kv[b];
        for (int t0 = 0; t0 < C; t0 += tile_tokens) {
            const int n_q = std::min(tile_tokens, C - t0);
            const int pos0 = L - C + t0;
            for (int g = 0; g < n_kv_heads; ++g) {
                tiles.push_back(PfUnit{-1, g, qo[b] + t0, n_q, kv[b], pos0, 0, pos0 + n_q});
                total_tiles += (pos0 + n_q + kPfKvTile - 1) / kPfKvTile;
            }
        }
    }
    int n = 0, n_blocks = 0, n_merges = 0;
    const bool split = int64_t(tiles.size()) < split_target && total_tiles > 0;
    const int64_t piece_tiles =
        split ? std::max<int64_t>(8, (total_tiles + split_target - 1) / split_target) : 1;
    for (const PfUnit& u : tiles) {
        int cuts = 0;  // split points at multiples of step * kPfKvTile, all <= pos0
        int64_t step = piece_tiles;
        if (split) {
            cuts = static_cast<int>(u.pos0 / (step * kPfKvTile));
            if (cuts > kPfMaxPieces - 1) {
                step = (u.pos0 / kPfKvTile + kPfMaxPieces - 1) / (kPfMaxPieces - 1);
                cuts = std::min(static_cast<int>(u.pos0 / (step * kPfKvTile)), kPfMaxPieces - 1);
            }
        }
        if (n + cuts + 1 > max_units || n_blocks + (cuts ? cuts + 1 : 0) > max_blocks ||
            (cuts && n_merges >= max_merges))
            return fail(PKV_ERR_PLAN, "%s: more work than the plan holds", who);
        if (cuts == 0) {
            units[n++] = u;
            continue;
        }
        merges[n_merges++] = PfMerge{u.q_row0, u.n_q, u.g, n_blocks, cuts + 1, 0, 0, 0};
        for (int c = 0; c <= cuts; ++c) {
            PfUnit piece = u;
            piece.part = n_blocks++;
            piece.kv_lo = static_cast<int32_t>(c * step * kPfKvTile);
            piece.kv_hi = c == cuts ? u.kv_hi : static_cast<int32_t>((c + 1) * step * kPfKvTile);
            units[n++] = piece;
        }
    }
    std::stable_sort(units, units + n, [](const PfUnit& x, const PfUnit& y) {
        return x.kv_hi - x.kv_lo > y.kv_hi - y.kv_lo;
    });
    out->n_units = n;
    out->n_merges = n_merges;
    out->n_blocks = n_blocks;
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

struct pkv_prefill_plan {
    int device = 0;
    int max_batch = 0;
    int64_t max_q_tokens = 0;
    int n_qo_heads = 0, n_kv_heads = 0, head_dim = 0;
    int tile_tokens = 0;  // query tokens per unit: 64 / G
    int max_units = 0;    // capacity of the unit list (tiles plus split pieces)
    int split_target = 0; // a step with fewer tile units than this splits long ranges
    int max_blocks = 0;   // workspace blocks of 64 rows (pieces of split units)
    int max_merges = 0;
    pkv::PfUnit* host_units = nullptr;  // pinned staging
    pkv::PfUnit* dev_units = nullptr;
    pkv::PfMerge* host_merges = nullptr;
    pkv::PfMerge* dev_merges = nullptr;
    float* ws_o = nullptr;
    float* ws_lse = nullptr;
    int n_merges = 0;
    cudaEvent_t copy_done = nullptr;
    bool copy_pending = false;
    bool planned = false;
    int batch = 0;
    int n_units = 0;
    std::vector<int32_t> qo_host, kv_host;  // the step's offsets (debug checks)
};

using namespace pkv;

extern "C" {

int paged_prefill_plan_create(pkv_prefill_plan** out_plan, int max_batch, int64_t max_q_tokens,
                              int n_qo_heads, int n_kv_heads, int head_dim) {
    clear_error();
    if (!out_plan) return fail(PKV_ERR_INVALID_ARG, "paged_prefill_plan_create: plan is NULL");
    *out_plan = nullptr;
    if (max_batch < 1 || max_q_tokens < 0 || max_q_tokens > INT32_MAX)
        return fail(PKV_ERR_INVALID_ARG,
                    "paged_prefill_plan_create: need max_batch >= 1 and 0 <= max_q_tokens < 2^31");
    if (!prefill_shape_supported(n_qo_heads, n_kv_heads, head_dim))
        return fail(PKV_ERR_UNSUPPORTED,
                    "paged_prefill_plan_create: unsupported shape (n_qo_heads=%d, n_kv_heads=%d, "
                    "head_dim=%d); need head_dim 128/256 and group 1/2/4/8",
                    n_qo_heads, n_kv_heads, head_dim);
    pkv_prefill_plan* p = new (std::nothrow) pkv_prefill_plan();
    if (!p) return fail(PKV_ERR_INVALID_ARG, "paged_prefill_plan_create: out of host memory");
    cudaError_t e = cudaGetDevice(&p->device);
    if (e != cudaSuccess) {
        delete p;
        return pf_cuda_fail(e, "paged_prefill_plan_create: device query");
    }
    p->max_batch = max_batch;
    p->max_q_tokens = max_q_tokens;
    p->n_qo_heads = n_qo_heads;
    p->n_kv_heads = n_kv_heads;
    p->head_dim = head_dim;
    p->tile_tokens = kPfRows / (n_qo_heads / n_kv_heads);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
    const int per_sm = prefill_dispatch<PfOccupancyFn>(head_dim, n_qo_heads / n_kv_heads);
    if (e != cudaSuccess || per_sm <= 0) {
        delete p;
        return fail(PKV_ERR_CUDA, "paged_prefill_plan_create: device or occupancy query failed");
    }
    // Steps with fewer tile units than two waves of the grid split long causal
    // ranges into pieces; a split step has at most 2 x target pieces.
    p->split_target = 2 * sms * per_sm;
    p->max_merges = p->split_target;
    p->max_blocks = 2 * p->split_target;
    const int64_t units = (max_q_tokens / p->tile_tokens + max_batch) * int64_t(n_kv_heads) +
                          p->max_blocks;
    if (units > INT32_MAX / 2) {
        delete p;
        return fail(PKV_ERR_INVALID_ARG, "paged_prefill_plan_create: too many work units");
    }
    p->max_units = static_cast<int>(units);
    const size_t rows = size_t(p->max_blocks) * kPfRows;
    e = cudaMallocHost(reinterpret_cast<void**>(&p->host_units), sizeof(PfUnit) * size_t(units));
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&p->dev_units), sizeof(PfUnit) * size_t(units));
    if (e == cudaSuccess)
        e = cudaMallocHost(reinterpret_cast<void**>(&p->host_merges), sizeof(PfMerge) * size_t(p->max_merges));
    if (e == cudaSuccess)
        e = cudaMalloc(reinterpret_cast<void**>(&p->dev_merges), sizeof(PfMerge) * size_t(p->max_merges));
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&p->ws_o), sizeof(float) * rows * head_dim);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&p->ws_lse), sizeof(float) * rows);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->copy_done, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        paged_prefill_plan_destroy(p);
        return pf_cuda_fail(e, "paged_prefill_plan_create: allocation");
    }
    *out_plan = p;
    return PKV_OK;
}

void paged_prefill_plan_destroy(pkv_prefill_plan* p) {
    if (p == nullptr) return;
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(p->device);
    if (p->copy_done) {
        cudaEventSynchronize(p->copy_done);
        cudaEventDestroy(p->copy_done);
    }
    if (p->host_units) cudaFreeHost(p->host_units);
    if (p->dev_units) cudaFree(p->dev_units);
    if (p->host_merges) cudaFreeHost(p->host_merges);
    if (p->dev_merges) cudaFree(p->dev_merges);
    if (p->ws_o) cudaFree(p->ws_o);
    if (p->ws_lse) cudaFree(p->ws_lse);
    if (prev >= 0) cudaSetDevice(prev);
    delete p;
}

int paged_prefill_plan(pkv_prefill_plan* p, const int32_t* qo_indptr_host,
                       const int32_t* kv_indptr_host, int batch, pkv_stream_t stream) {
    clear_error();
    const char* who = "paged_prefill_plan";
    if (!p) return fail(PKV_ERR_PLAN, "%s: plan is NULL", who);
    p->planned = false;
    if (batch < 0 || batch > p->max_batch)
        return fail(PKV_ERR_PLAN, "%s: batch %d outside [0, %d]", who, batch, p->max_batch);
    if (!qo_indptr_host || !kv_indptr_host)
        return fail(PKV_ERR_INVALID_ARG, "%s: NULL offsets", who);
    if (qo_indptr_host[0] == 0 && batch >= 0 &&
        int64_t(qo_indptr_host[batch]) > p->max_q_tokens)
        return fail(PKV_ERR_PLAN, "%s: %d query tokens exceed the plan's max_q_tokens %lld", who,
                    qo_indptr_host[batch], (long long)p->max_q_tokens);
    if (p->copy_pending) {  // the staging may still feed the previous step's copy
        cudaError_t e = cudaEventSynchronize(p->copy_done);
        if (e != cudaSuccess) return pf_cuda_fail(e, "waiting for the previous prefill plan copy");
        p->copy_pending = false;
    }
    PfPlanCounts c{};
    const int rc = prefill_plan_compute(who, qo_indptr_host, kv_indptr_host, batch,
                                        p->tile_tokens, p->n_kv_heads, p->split_target,
                                        p->host_units, p->max_units, p->host_merges,
                                        p->max_merges, p->max_blocks, &c);
    if (rc != PKV_OK) return rc;
    if (c.n_units > 0) {
        cudaError_t e = cudaMemcpyAsync(p->dev_units, p->host_units,
                                        sizeof(PfUnit) * size_t(c.n_units),
                                        cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess && c.n_merges > 0)
            e = cudaMemcpyAsync(p->dev_merges, p->host_merges, sizeof(PfMerge) * size_t(c.n_merges),
                                cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaEventRecord(p->copy_done, stream);
        if (e != cudaSuccess) return pf_cuda_fail(e, "prefill plan upload");
        p->copy_pending = true;
    }
    p->batch = batch;
    p->n_units = c.n_units;
    p->n_merges = c.n_merges;
    p->qo_host.assign(qo_indptr_host, qo_indptr_host + batch + 1);
    p->kv_host.assign(kv_indptr_host, kv_indptr_host + batch + 1);
    p->planned = true;
    return PKV_OK;
}

int paged_prefill_plan_host(const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                            int batch, int n_qo_heads, int n_kv_heads, int head_dim,
                            int split_target, int32_t* units_out, int max_units,
                            int32_t* merges_out, int max_merges, int32_t* counts_out) {
    clear_error();
    const char* who = "paged_prefill_plan_host";
    if (!prefill_shape_supported(n_qo_heads, n_kv_heads, head_dim))
        return fail(PKV_ERR_UNSUPPORTED, "%s: unsupported shape", who);
    if (!qo_indptr_host || !kv_indptr_host || !counts_out || (max_units > 0 && !units_out) ||
        (max_merges > 0 && !merges_out) || batch < 0 || max_units < 0 || max_merges < 0)
        return fail(PKV_ERR_INVALID_ARG, "%s: NULL or negative argument", who);
    PfPlanCounts c{};
    const int rc = prefill_plan_compute(
        who, qo_indptr_host, kv_indptr_host, batch, kPfRows / (n_qo_heads / n_kv_heads),
        n_kv_heads, split_target, reinterpret_cast<PfUnit*>(units_out), max_units,
        reinterpret_cast<PfMerge*>(merges_out), max_merges, 2 * std::max(split_target, 0), &c);
    if (rc != PKV_OK) return rc;
    counts_out[0] = c.n_units;
    counts_out[1] = c.n_merges;
    counts_out[2] = c.n_blocks;
    return PKV_OK;
}

int paged_prefill_attn(const void* q, const void* k_pool, const void* v_pool,
                       const int32_t* qo_indptr, const int32_t* kv_indptr,
                       const int32_t* kv_indices, int batch, int n_qo_heads, int n_kv_heads,
                       int head_dim, float sm_scale, void* out, float* lse,
                       const pkv_prefill_plan* p, pkv_stream_t stream) {
    clear_error();
    const char* who = "paged_prefill_attn";
    if (!p || !p->planned) return fail(PKV_ERR_PLAN, "%s: plan is NULL or not planned", who);
    if (batch != p->batch)
        return fail(PKV_ERR_PLAN, "%s: batch %d differs from the plan's %d", who, batch, p->batch);
    if (n_qo_heads != p->n_qo_heads || n_kv_heads != p->n_kv_heads || head_dim != p->head_dim)
        return fail(PKV_ERR_PLAN, "%s: shape differs from the plan's", who);
    if (!std::isfinite(sm_scale)) return fail(PKV_ERR_INVALID_ARG, "%s: sm_scale not finite", who);
    if (p->n_units == 0) return PKV_OK;
    if (!q || !k_pool || !v_pool || !qo_indptr || !kv_indptr || !kv_indices || !out)
        return fail(PKV_ERR_INVALID_ARG, "%s: NULL pointer argument", who);
    const auto aligned16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return fail(PKV_ERR_INVALID_ARG, "%s: q, pools and out must be 16-byte aligned", who);
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u))
        return fail(PKV_ERR_INVALID_ARG, "%s: lse must be 4-byte aligned", who);
    if (debug_checks()) {
        std::vector<int32_t> qo(batch + 1), kv(batch + 1);
        cudaError_t e = cudaMemcpyAsync(qo.data(), qo_indptr, qo.size() * 4, cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(kv.data(), kv_indptr, kv.size() * 4, cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return pf_cuda_fail(e, "paged_prefill_attn: debug copy of offsets");
        if (qo != p->qo_host || kv != p->kv_host)
            return fail(PKV_ERR_INDEX, "%s: device offsets differ from the plan's host copies", who);
    }
    PfArgs a{};
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.kv_indices = kv_indices;
    a.units = p->dev_units;
    a.n_qo_heads = n_qo_heads;
    a.n_kv_heads = n_kv_heads;
    a.scale_log2 = sm_scale * kLog2e;
    a.out = out;
    a.lse = lse;
    a.ws_o = p->ws_o;
    a.ws_lse = p->ws_lse;
    a.merges = p->dev_merges;
    a.n_merges = p->n_merges;
    const cudaError_t e = prefill_dispatch<PfLaunchFn>(head_dim, n_qo_heads / n_kv_heads, a,
                                                       p->n_units, stream);
    if (e != cudaSuccess) return pf_cuda_fail(e, "paged_prefill_attn: launch");
    return PKV_OK;
}

}  // extern "C"
