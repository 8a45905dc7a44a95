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
// Design for sm_103a. Unlike decode, every K/V row here serves the 128 / G query
// tokens of a unit times G heads, so the work is a dense contraction per KV head,
// run on the fifth-generation tensor cores (tcgen05) with accumulators in tensor
// memory:
//  * One CTA per work unit (request, KV head, tile of 128 / G chunk tokens): its 128
//    query rows (row r: token r / G, head r % G) are the M of every MMA. The plan
//    orders units longest causal range first, so the grid drains evenly.
//  * Two producer halves (two warps each) gather the unit's q rows once and the
//    request's slot rows of that KV head in K/V tiles of kKv tokens (128 at head_dim
//    128, 64 at 256), with 16-byte cp.async into separate K and V rings of
//    shared-memory stages. Each row is stored in the tensor core's 128-byte swizzled
//    layout (K-major for q and K; V's rows are the same bytes read as an MN-major
//    operand). Tokens past a range repeat its last row (finite rows the softmax masks),
//    so every copy is a full one from a per-unit base address. A thread's arrival on a
//    stage's barrier rides on its copies, and a relay thread fences the landed stage
//    (generic to async proxy) for the tensor core. Two more warps copy the first tokens of every K and V tile (32 of 128 at
//    head_dim 128, 16 of 64 at 256) with 4-row TMA gathers (cp.async.bulk.tensor
//    .tile::gather4) through tensor maps of the pools in that 128-byte swizzled
//    layout, their bytes counted on the same barrier: the SMs then take in the tiles
//    by both paths at once.
//  * An MMA warp issues, from one lane, S = Q K^T (128 x kKv, K = head_dim, operands
//    in shared memory) into one of three TMEM buffers, and O += P V (128 x head_dim,
//    K = kKv) with P read from TMEM as the A operand, each signalled on an mbarrier
//    by tcgen05.commit. P is written over the upper half of its own S buffer once the
//    softmax has read it, so S of tile n + 3 waits for P V of tile n to complete; S
//    runs up to two tiles ahead of the softmax, and the softmax never waits for a
//    buffer to write P into.
//  * Four softmax warps own one query row per thread: they read the row of S from
//    TMEM, apply the causal mask (list position <= the row's query position) and an
//    online softmax in base 2 with fp32 state (three-input maxima, and the exponent
//    arguments and row sums two entries to an instruction), write P as bf16 pairs over
//    the upper half of the same S buffer, and rescale O in TMEM when a row's running
//    maximum grows by more than 2^8 (between rescales the probabilities stay below
//    2^8, exact enough for bf16 P and fp32 sums). At the end they read O back, divide
//    by the row sum and store out and lse.
//  * Every wait is an mbarrier wait bounded by 1 s; on expiry the CTA records it in
//    the plan's status word, every role leaves its loop, the MMA and copies in
//    flight are drained (again bounded) and the tensor memory is freed. Barriers a
//    reader could fall behind on are split per buffer, so that no parity test can
//    alias.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <new>
#include <vector>

#include "pkv_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

using namespace ptx;

constexpr int kPfRows = 128;                // query rows (token, head) per unit: the MMA's M
constexpr int kPfKvTile = 128;              // planning granularity of KV ranges (split cuts)
constexpr int kPfSoftmaxWarps = 4;          // one thread per query row (TMEM lane)
constexpr int kPfProducerWarps = 4;
constexpr int kPfProducerThreads = 32 * kPfProducerWarps;
constexpr int kPfHalfThreads = kPfProducerThreads / 2;  // K rows by one half, V rows by the other
constexpr int kPfMmaWarp = kPfSoftmaxWarps + kPfProducerWarps;  // also owns the TMEM allocation
constexpr int kPfRelayWarp = kPfMmaWarp + 1;
constexpr int kPfTmaWarp = kPfRelayWarp + 1;  // two more warps (K rows, V rows)
constexpr uint32_t kPfTmemCols = 512;
constexpr int kPfSBufs = 3;                 // S buffers in TMEM (P over their upper halves)
constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;         // rescale O once a row maximum grows by more
constexpr unsigned long long kPfWaitNs = 1000000000ull;

// One work unit: query tokens q_row0 .. q_row0 + n_q - 1 (rows of q/out) of one
// request, KV head g, over list entries kv_lo .. kv_hi - 1 of the request's slot
// list (which starts at kv_begin in kv_indices). The unit's first query sits at list
// position pos0. part < 0: the unit covers every entry its queries see and writes
// out/lse; otherwise it is one piece of a split range, kv_lo <= pos0 and kv_lo a
// multiple of the ring tile, and writes its 128 rows' normalised fp32 output and
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

// Tensor maps of one call (cuTensorMapEncodeTiled): each pool as a 2D
// array [slots, n_kv_heads x head_dim] with 64 x 1 element boxes and the 128-byte
// swizzle, for 4-row gathers.
struct PfMaps {
    CUtensorMap k, v;
};

struct PfArgs {
    PfMaps maps;  // the pools, for the TMA gathers
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
    float* ws_o;       // [blocks, 128, head_dim] partial outputs of split units
    float* ws_lse;     // [blocks, 128] their base-2 lse
    const PfMerge* merges;
    int n_merges;
    int* status;       // nonzero: a wait of some CTA exceeded its bound
    bool withhold;     // injected stall (pkv_inject_stall): the producers issue no copies
};

// Tokens of every K and V tile copied by the tensor memory accelerator's gather form
// (two more warps), the rest by the producer threads' cp.async: measured best at 16
// of 64 at head_dim 256 and 32 of 128 at head_dim 128.
constexpr int pf_tma_tokens(int head_dim) { return head_dim == 256 ? 16 : 32; }

// Shared memory of one CTA (offsets from a 1024-byte aligned base). Every operand
// is stored as 64-element panels of 128-byte rows in the 128-byte swizzled layout:
// row n of a panel at (n / 8) * 1024 + (n % 8) * 128, its 16-byte chunk c at
// ((c ^ (n % 8)) * 16).
template <int D, int G>
struct PfCfg {
    // KV tokens per ring stage: the N of S and the K of P V. Each tcgen05.mma costs
    // its issuing thread about as much time as a 128 x 128 x 16 step takes the
    // tensor core, so the MMAs are made as large as shared memory allows.
    static constexpr int kKv = D == 128 ? 128 : 64;
    static constexpr int kKStages = D == 128 ? 3 : 2;  // K ring stages
    static constexpr int kVStages = D == 128 ? 3 : 2;  // V ring stages
    static constexpr int kRingStages = kKStages + kVStages;
    // stages of ring v (0: K, 1: V) and the index of its stage s among both rings
    __host__ __device__ static constexpr int stages(int v) { return v ? kVStages : kKStages; }
    __host__ __device__ static constexpr int ring_slot(int v, int s) { return (v ? kKStages : 0) + s; }
    // TMEM columns: S buffer b at b * kKv (fp32; P of its tile, kKv / 2 columns of
    // bf16 pairs, the A operand of P V, over its upper half), O in the last D columns
    static constexpr int kOCol = int(kPfTmemCols) - D;
    static constexpr int kPanels = D / 64;
    static constexpr int kQPanel = kPfRows * 128;           // bytes of one q panel
    static constexpr int kKvPanel = kKv * 128;              // bytes of one K (or V) panel
    static constexpr int kQBytes = kPanels * kQPanel;
    static constexpr int kKvBytes = kPanels * kKvPanel;     // K (or V) of one stage
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQBytes;
    static constexpr int kVOff = kKOff + kKStages * kKvBytes;
    static constexpr int kBarOff = kVOff + kVStages * kKvBytes;
    // mbarriers: landed / full / empty per stage of the K and V rings;
    // s_full, p_full and o_done per S buffer, drain; then the TMEM address and the
    // abort flag
    static constexpr int kNumBars = 3 * kRingStages + 3 * kPfSBufs + 1;
    static constexpr int kTmemOff = kBarOff + 8 * kNumBars;
    static constexpr int kAbortOff = kTmemOff + 4;
    static constexpr int kSmem = kAbortOff + 4 + 1024;      // + slack to align the base
    static constexpr int kChunks = D / 8;                   // 16-byte pieces per row
    // Two more warps copy the first kTmaTok tokens of every K and V tile by the
    // tensor memory accelerator's gather form, the producer threads the rest.
    static constexpr int kTmaTok = pf_tma_tokens(D);
    static constexpr int kThreads = 32 * (kPfRelayWarp + 1 + (kTmaTok > 0 ? 2 : 0));
    static constexpr int kTilePieces = (kKv - kTmaTok) * kChunks / kPfHalfThreads;  // per thread, K or V
    static constexpr int kQPieces = kPfRows * kChunks / kPfHalfThreads;   // q, by the K half
    static constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kPfRows, kKv, false, false);
    static constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kPfRows, D, false, true);
    static_assert(kTilePieces * kPfHalfThreads == (kKv - kTmaTok) * kChunks, "ring pieces");
    static_assert(kTmaTok % 4 == 0 && kTmaTok / 4 <= 32, "4-row gathers, one lane each");
    static_assert(kPfKvTile % kKv == 0, "split cuts fall on ring tiles");
    static_assert(kQPieces * kPfHalfThreads == kPfRows * kChunks, "q pieces");
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    static_assert(kPfSBufs * kKv <= kOCol, "TMEM columns");
};

// Byte offset of 16-byte chunk c of row n in a panel-major swizzled operand whose
// panels hold `rows` rows.
__device__ __forceinline__ uint32_t sw128_off(int n, int c, int rows) {
    return uint32_t((c >> 3) * rows * 128 + (n >> 3) * 1024 + (n & 7) * 128 + (((c & 7) ^ (n & 7)) << 4));
}

__device__ __forceinline__ unsigned long long pf_global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase of `bar` with the given parity; on expiry (or if
// another thread already gave up) records the failure and returns false.
__device__ __forceinline__ bool pf_wait(uint32_t bar, uint32_t parity, int* status,
                                        volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = pf_global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (pf_global_ns() - t0 > kPfWaitNs) {
            atomicOr(status, 1);
            *abort_flag = 1;
            return false;
        }
    }
}

// max(a, b, c) in one instruction (three-input max.f32, PTX ISA 8.8, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 16-byte asynchronous copy, always a full one.
__device__ __forceinline__ void cp_async16_full(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Non-blocking test of the phase of `bar` with the given parity.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// One arrival on `bar` once every cp.async this thread issued before has completed
// (the barrier's expected count includes it).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// A producer thread's pieces of a K (or V) tile: piece i is token kTmaTok + tokA +
// i * kStep (tokA = pt / kChunks < kStep), in its 16-byte column pt % kChunks.
template <int D, int G>
struct PfPieces {
    using C = PfCfg<D, G>;
    static constexpr int kStep = kPfHalfThreads / C::kChunks;
    static constexpr int kPeriod = 8 / kStep;  // pieces per 8-row swizzle atom
    static_assert(kPfHalfThreads % C::kChunks == 0 && 8 % kStep == 0, "piece layout");
};

// Slot ids of the rows this producer thread copies for KV tile `tile`. Tokens past the
// range repeat the range's last row (finite rows that the softmax masks), so every copy
// is a full one; on a tile wholly inside the range (all but a range's last) no entry
// needs that clamp and each id is one load at a fixed offset.
template <int D, int G>
__device__ __forceinline__ void load_tile_slots(const int32_t* ids, int kv_hi, int tile, int tokA,
                                                int (&slot)[PfCfg<D, G>::kTilePieces]) {
    using C = PfCfg<D, G>;
    constexpr int kStep = PfPieces<D, G>::kStep;
    const int first = tile * C::kKv + C::kTmaTok + tokA;  // this thread's first token
    const int32_t* p = ids + first;
    if ((tile + 1) * C::kKv <= kv_hi) {
#pragma unroll
        for (int i = 0; i < C::kTilePieces; ++i) slot[i] = __ldg(p + i * kStep);
    } else {
        const int last = kv_hi - 1 - first;  // the range's last entry, from the first token
#pragma unroll
        for (int i = 0; i < C::kTilePieces; ++i) slot[i] = __ldg(p + min(i * kStep, last));
    }
}

// cp.async of this thread's pieces of a K (or V) tile into the stage at shared address
// `dst`. `src` is this thread's 16 bytes of the row of slot 0 (its KV head and its
// 16-byte column, the same for every piece), `row_bytes` the pool's bytes per slot.
// lo[r] is the swizzled offset of piece r; piece r + kPeriod * q lies 1024 q bytes
// (q atoms of 8 rows) further.
template <int D, int G>
__device__ __forceinline__ void issue_tile(const char* src, uint32_t row_bytes, uint32_t dst,
                                           const uint32_t (&lo)[PfPieces<D, G>::kPeriod],
                                           const int (&slot)[PfCfg<D, G>::kTilePieces]) {
    using C = PfCfg<D, G>;
    constexpr int kPeriod = PfPieces<D, G>::kPeriod;
#pragma unroll
    for (int i = 0; i < C::kTilePieces; ++i)
        cp_async16_full(dst + lo[i % kPeriod] + uint32_t(1024 * (i / kPeriod)),
                        src + size_t(uint32_t(slot[i])) * row_bytes);
}

// Four rows of a 2D tensor map (row indices r0..r3, columns col .. col + 63) into 512
// consecutive bytes of shared memory at dst, completing their bytes on mbarrier bar
// (PTX ISA: cp.async.bulk.tensor, .tile::gather4). col * 2 bytes is a multiple of 16.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int col, int r0,
                                            int r1, int r2, int r3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
        : "memory");
}

template <int D, int G>
__global__ void __launch_bounds__(PfCfg<D, G>::kThreads, 1)
    paged_prefill_kernel(const __grid_constant__ PfArgs a) {
    using C = PfCfg<D, G>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the swizzled operands need 1024-byte aligned atoms
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t bars = base + C::kBarOff;
    // ring barriers of K (v = 0) and V (v = 1): landed (the producers' copies are in
    // shared memory), full (announced to the tensor core), empty (read by it)
    const auto landed = [&](int v, int s) { return bars + 8u * C::ring_slot(v, s); };
    const auto full = [&](int v, int s) { return bars + 8u * (C::kRingStages + C::ring_slot(v, s)); };
    const auto empty = [&](int v, int s) { return bars + 8u * (2 * C::kRingStages + C::ring_slot(v, s)); };
    const uint32_t bars2 = bars + 8u * 3 * C::kRingStages;
    // S of tile n written / P of tile n written / P V of tile n done: one barrier per
    // S buffer (tiles n, n + 3, ...; phase parity (n / 3) & 1). No role can run three
    // tiles ahead of a barrier's other side, so no parity test can alias.
    const auto s_full = [&](int n) { return bars2 + 8u * (n % kPfSBufs); };
    const auto p_full = [&](int n) { return bars2 + 8u * (kPfSBufs + n % kPfSBufs); };
    const auto o_done = [&](int n) { return bars2 + 8u * (2 * kPfSBufs + n % kPfSBufs); };
    const auto ph = [](int n) { return uint32_t((n / kPfSBufs) & 1); };
    const uint32_t drain = bars2 + 8u * 3 * kPfSBufs;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbortOff);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int v = 0; v < 2; ++v)
            for (int s = 0; s < C::stages(v); ++s) {
                // the producer threads' cp.async arrivals (and the TMA warp's byte count)
                mbar_init(landed(v, s), kPfHalfThreads + (C::kTmaTok > 0 ? 1 : 0));
                mbar_init(full(v, s), 1);
                mbar_init(empty(v, s), 1);
            }
        for (int b = 0; b < kPfSBufs; ++b) {
            mbar_init(s_full(b), 1);
            mbar_init(p_full(b), 32 * kPfSoftmaxWarps);
            mbar_init(o_done(b), 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kPfMmaWarp) {  // the whole warp: allocation is .sync.aligned
        tc::tmem_alloc(base + C::kTmemOff, kPfTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::kTmemOff);
    pdl_launch_dependents();
    const PfUnit un = a.units[blockIdx.x];  // plan data
    const int t0 = un.kv_lo / C::kKv;
    const int n_tiles = (un.kv_hi + C::kKv - 1) / C::kKv - t0;
    // q, the pools and their indices may come from the previous kernel, and out may
    // still be read by it
    pdl_wait();

    if (warp >= kPfSoftmaxWarps && warp < kPfMmaWarp) {
        // ================= producers =================
        // Two halves: one gathers K tiles (and the unit's q rows), the other V tiles.
        // K tile n goes to K stage n % kKStages once S of tile n - kKStages has read it,
        // V tile n to V stage n % kVStages once P V of tile n - kVStages has, so the
        // next K tiles are not held
        // back by the P V products. Each thread's arrival on the stage's `landed`
        // barrier is attached to its copies, so it completes the moment the rows are
        // in shared memory; the relay warp then announces the stage to the tensor core.
        const int half = (tid - 32 * kPfSoftmaxWarps) / kPfHalfThreads;  // 0: K, 1: V
        const int pt = (tid - 32 * kPfSoftmaxWarps) % kPfHalfThreads;
        // an injected stall: no copies, so every wait of the launch expires (bounded)
        const int n_copy_tiles = a.withhold ? 0 : n_tiles;
        if (half == 0 && !a.withhold) {   // the unit's q rows (row r: token r / G, head r % G), with K tile 0
            const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
#pragma unroll 4
            for (int i = 0; i < C::kQPieces; ++i) {
                const int c = pt + i * kPfHalfThreads;
                const int r = c / C::kChunks, part = c % C::kChunks;
                const int t = r / G, h = r % G;
                const bool valid = t < un.n_q;
                const int64_t off =
                    (int64_t(un.q_row0 + (valid ? t : 0)) * a.n_qo_heads + un.g * G + h) * D + part * 8;
                cp_async16(base + C::kQOff + sw128_off(r, part, kPfRows), q + off, valid);
            }
        }
        const uint32_t row_bytes = uint32_t(a.n_kv_heads) * D * 2;
        const char* src = static_cast<const char*>(half ? a.v_pool : a.k_pool) +
                          (size_t(un.g) * D + (pt % C::kChunks) * 8) * 2;
        const uint32_t ring = base + (half ? C::kVOff : C::kKOff);
        using PP = PfPieces<D, G>;
        const int tokA = pt / C::kChunks, col = pt % C::kChunks;
        uint32_t lo[PP::kPeriod];
#pragma unroll
        for (int r = 0; r < PP::kPeriod; ++r)
            lo[r] = sw128_off(C::kTmaTok + tokA + r * PP::kStep, col, C::kKv);
        const int32_t* ids = a.kv_indices + un.kv_begin;
        int slot[C::kTilePieces];
        if (n_copy_tiles > 0) load_tile_slots<D, G>(ids, un.kv_hi, t0, tokA, slot);
        for (int n = 0; n < n_copy_tiles; ++n) {
            const int stages = C::stages(half);
            const int st = n % stages;
            if (n >= stages &&
                !pf_wait(empty(half, st), uint32_t((n / stages - 1) & 1), a.status, abort_flag))
                break;
            issue_tile<D, G>(src, row_bytes, ring + st * C::kKvBytes, lo, slot);
            cp_async_arrive(landed(half, st));
            if (n + 1 < n_tiles) load_tile_slots<D, G>(ids, un.kv_hi, t0 + n + 1, tokA, slot);
        }
        cp_async_wait<0>();  // nothing may still write this CTA's shared memory at exit
    } else if (warp == kPfMmaWarp) {
        // ================= MMA issuer (one warp, one lane issues) =================
        // Two streams of work, each issued as soon as its inputs are ready (polled,
        // so that neither waits behind the other): S of tile ns once its K stage has
        // been announced and P V of tile ns - 3, which read P from the same S buffer,
        // has completed (so S runs up to two tiles ahead of the softmax), and
        // P V of tile npv once its P is in TMEM (and O rescaled) and its V stage has
        // been announced. The whole warp runs the loop with lane 0's view of the
        // barriers, so the descriptors stay warp-uniform; lane 0 alone issues.
        const bool leader = lane == 0;
        const uint32_t o_tmem = tmem + uint32_t(C::kOCol);
        const uint64_t q_desc = tc::sdesc_sw128(base + C::kQOff, 16, 1024);
        const uint64_t k_desc = tc::sdesc_sw128(base + C::kKOff, 16, 1024);
        const uint64_t v_desc = tc::sdesc_sw128(base + C::kVOff, C::kKvPanel, 1024);
        int ns = 0, npv = 0;
        unsigned idle = 0;
        unsigned long long t_idle = 0;
        while (npv < n_tiles) {
            bool progress = false;
            bool go = false;
            if (leader && ns < n_tiles)
                go = mbar_test(full(0, ns % C::kKStages), uint32_t((ns / C::kKStages) & 1)) &&
                     (ns < kPfSBufs || mbar_test(o_done(ns), ph(ns - kPfSBufs)));
            if (__shfl_sync(kFullMask, go, 0)) {
                tc::fence_after_sync();
                // descriptor start addresses advance in 16-byte units (low bits)
                const uint64_t kd = k_desc + uint64_t(((ns % C::kKStages) * C::kKvBytes) >> 4);
                const uint32_t s_tmem = tmem + uint32_t((ns % kPfSBufs) * C::kKv);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = uint32_t(((ks >> 2) * C::kQPanel + (ks & 3) * 32) >> 4);
                    const uint32_t koff = uint32_t(((ks >> 2) * C::kKvPanel + (ks & 3) * 32) >> 4);
                    tc::mma_bf16_ss_if(leader, s_tmem, q_desc + off, kd + koff, C::kIdescS, ks > 0);
                }
                tc::commit_if(leader, s_full(ns));
                tc::commit_if(leader, empty(0, ns % C::kKStages));
                ++ns;
                progress = true;
            }
            go = false;
            if (leader && npv < ns)
                go = mbar_test(p_full(npv), ph(npv)) &&
                     mbar_test(full(1, npv % C::kVStages), uint32_t((npv / C::kVStages) & 1));
            if (__shfl_sync(kFullMask, go, 0)) {
                tc::fence_after_sync();
                const uint64_t vd = v_desc + uint64_t(((npv % C::kVStages) * C::kKvBytes) >> 4);
                const uint32_t p_tmem = tmem + uint32_t((npv % kPfSBufs) * C::kKv + C::kKv / 2);
#pragma unroll
                for (int ks = 0; ks < C::kKv / 16; ++ks)
                    tc::mma_bf16_ts_if(leader, o_tmem, p_tmem + uint32_t(8 * ks),
                                       vd + uint64_t((ks * 16 * 128) >> 4), C::kIdescO, npv > 0 || ks > 0);
                tc::commit_if(leader, o_done(npv));
                tc::commit_if(leader, empty(1, npv % C::kVStages));
                ++npv;
                progress = true;
            }
            if (progress) {
                idle = 0;
            } else if (++idle % 256 == 0) {  // the clocks are read now and then only
                bool stop = false;
                if (leader) {
                    if (idle == 256) t_idle = pf_global_ns();
                    if (*abort_flag) {
                        stop = true;
                    } else if (pf_global_ns() - t_idle > kPfWaitNs) {
                        atomicOr(a.status, 1);
                        *abort_flag = 1;
                        stop = true;
                    }
                }
                if (__shfl_sync(kFullMask, stop, 0)) break;
            }
        }
        // every MMA issued has completed before the CTA frees TMEM and exits (this
        // wait does not stop early for another role's failure)
        tc::commit_if(leader, drain);
        if (leader) {
            const unsigned long long t_drain = pf_global_ns();
            while (!mbar_try_wait(drain, 0u) && pf_global_ns() - t_drain < kPfWaitNs) {
            }
        }
        __syncwarp();
    } else if (warp >= kPfTmaWarp) {
        // ================= TMA gather =================
        // Tokens 0 .. kTmaTok - 1 of every K (warp kPfTmaWarp) or V tile: lane l copies
        // tokens 4l .. 4l + 3, one 4-row gather per 64-element panel, counted in bytes
        // on the stage's `landed` barrier beside the producer threads' arrivals. Rows
        // past the range repeat the range's last slot (finite rows the softmax masks).
        if constexpr (C::kTmaTok > 0) {
            const int half = warp - kPfTmaWarp;  // 0: K, 1: V
            const CUtensorMap* map = half ? &a.maps.v : &a.maps.k;
            const uint32_t ring = base + (half ? C::kVOff : C::kKOff);
            const int n_copy = a.withhold ? 0 : n_tiles;
            int sl[4] = {0, 0, 0, 0};
            const auto load_ids = [&](int t) {
                if (lane < C::kTmaTok / 4) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        sl[j] = __ldg(a.kv_indices + un.kv_begin +
                                      min(t * C::kKv + 4 * lane + j, un.kv_hi - 1));
                }
            };
            if (n_copy > 0) load_ids(t0);
            int issued = 0;
            for (int n = 0; n < n_copy; ++n) {
                const int stages = C::stages(half);
                const int st = n % stages;
                if (n >= stages) {
                    bool ok = true;
                    if (lane == 0)
                        ok = pf_wait(empty(half, st), uint32_t((n / stages - 1) & 1), a.status, abort_flag);
                    if (!__shfl_sync(kFullMask, ok, 0)) break;
                }
                if (lane == 0) mbar_arrive_expect_tx(landed(half, st), uint32_t(C::kTmaTok * D * 2));
                __syncwarp();
                if (lane < C::kTmaTok / 4) {
                    const uint32_t dst = ring + st * C::kKvBytes + lane * 512;
#pragma unroll
                    for (int pn = 0; pn < C::kPanels; ++pn)
                        tma_gather4(dst + pn * C::kKvPanel, map, un.g * D + 64 * pn, sl[0], sl[1], sl[2],
                                    sl[3], landed(half, st));
                }
                ++issued;
                if (n + 1 < n_copy) load_ids(t0 + n + 1);
            }
            // nothing may still write this CTA's shared memory at exit: wait (bounded)
            // for the last fill of every stage
            if (lane == 0) {
                for (int k = issued - C::stages(half); k < issued; ++k) {
                    if (k < 0) continue;
                    const uint32_t bar = landed(half, k % C::stages(half)),
                                   par = uint32_t((k / C::stages(half)) & 1);
                    const unsigned long long t_wait = pf_global_ns();
                    while (!mbar_try_wait(bar, par) && pf_global_ns() - t_wait < kPfWaitNs) {
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp == kPfRelayWarp) {
        // ================= relay: landed stage -> tensor core =================
        // The rows came by cp.async (generic proxy); the tensor core reads them
        // through the async proxy. One thread orders the two (proxy fence) after each
        // stage has landed, polling the K and V rings in turn (neither waits behind
        // the other), so that neither the producers nor the MMA thread wait for it.
        if (lane == 0) {
            int nr[2] = {0, 0};
            unsigned idle = 0;
            unsigned long long t_idle = 0;
            while (nr[0] < n_tiles || nr[1] < n_tiles) {
                bool progress = false;
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const int n = nr[v];
                    if (n < n_tiles &&
                        mbar_test(landed(v, n % C::stages(v)), uint32_t((n / C::stages(v)) & 1))) {
                        tc::fence_proxy_async_smem();
                        mbar_arrive(full(v, n % C::stages(v)));
                        nr[v] = n + 1;
                        progress = true;
                    }
                }
                if (progress) {
                    idle = 0;
                } else if (++idle % 256 == 0) {
                    if (idle == 256) t_idle = pf_global_ns();
                    if (*abort_flag) break;
                    if (pf_global_ns() - t_idle > kPfWaitNs) {
                        atomicOr(a.status, 1);
                        *abort_flag = 1;
                        break;
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ================= softmax: thread = query row =================
        const int r = tid;                       // TMEM lane and query row
        const int t = r / G, h = r % G;
        const int qpos = un.pos0 + t;
        const uint32_t lane_base = uint32_t(32 * warp) << 16;
        const float sl2 = a.scale_log2;
        float m = neg_inf(), l = 0.f;
        bool ok = true;
        for (int n = 0; n < n_tiles; ++n) {
            const uint32_t s_tmem = tmem + lane_base + uint32_t((n % kPfSBufs) * C::kKv);
            ok = pf_wait(s_full(n), ph(n), a.status, abort_flag);
            if (!__all_sync(kFullMask, ok)) { ok = false; break; }
            tc::fence_after_sync();
            float x[C::kKv];
            {   // the row of S in one load (complete before P is written over it)
                uint32_t v[C::kKv];
                if constexpr (C::kKv == 128)
                    tc::tmem_ld128(s_tmem, v);
                else
                    tc::tmem_ld64(s_tmem, v);
#pragma unroll
                for (int i = 0; i < C::kKv; ++i) x[i] = __uint_as_float(v[i]);
            }
            // causal mask: entry e is seen by this row iff e <= qpos and e < kv_hi
            // (raw scores; sm_scale > 0 is applied in the exponent below)
            const int e0 = (t0 + n) * C::kKv;
            const int lim = min(qpos + 1, un.kv_hi) - e0;  // entries 0 .. lim - 1 seen
            if (lim < C::kKv) {
#pragma unroll
                for (int i = 0; i < C::kKv; ++i) x[i] = i < lim ? x[i] : neg_inf();
            }
            // row maximum: eight independent chains of three-input maxima, then a tree
            float mxv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) mxv[j] = x[j];
#pragma unroll
            for (int i = 8; i < C::kKv; i += 16)
#pragma unroll
                for (int j = 0; j < 8; ++j) mxv[j] = fmax3(mxv[j], x[i + j], x[i + 8 + j]);
            const float mx = fmax3(fmax3(mxv[0], mxv[1], mxv[2]), fmax3(mxv[3], mxv[4], mxv[5]),
                                   fmaxf(mxv[6], mxv[7])) * sl2;
            // running maximum (base 2, scaled): moves when a row's maximum grows by more
            // than 2^8 (the first tile always sets it: every row sees entry kv_lo)
            const bool grow = mx > m + kRescaleLog2;
            const float m_new = grow ? mx : m;
            const float alpha = grow ? ex2(m - m_new) : 1.f;  // 0 on the first tile
            m = m_new;
            const float neg_m = -m;
            // P = 2^(s * scale - m) as bf16 pairs into this row's TMEM lane (the A
            // operand of P V) over the upper half of the S buffer, 64 entries (32
            // columns) at a time
            const uint32_t p_tmem = s_tmem + uint32_t(C::kKv / 2);
            // (the exponent arguments and the row sum two entries to an instruction:
            // the paired fp32 FMA and add of sm_100 and later)
            const float2 sl2x2 = make_float2(sl2, sl2), neg_mx2 = make_float2(neg_m, neg_m);
            float2 sums[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < C::kKv / 64; ++c) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float2 e = __ffma2_rn(make_float2(x[64 * c + 2 * i], x[64 * c + 2 * i + 1]),
                                                sl2x2, neg_mx2);
                    const float2 p = make_float2(ex2(e.x), ex2(e.y));
                    sums[i & 1] = __fadd2_rn(sums[i & 1], p);
                    pk[i] = pack_bf16x2(p.x, p.y);
                }
                tc::tmem_st32(p_tmem + uint32_t(32 * c), pk);
            }
            const float2 s2 = __fadd2_rn(sums[0], sums[1]);
            l = fmaf(l, alpha, s2.x + s2.y);
            // a row maximum moved: O (complete up to P V of tile n - 1) is rescaled
            // before P V of tile n accumulates into it
            if (n > 0 && __any_sync(kFullMask, grow)) {
                ok = pf_wait(o_done(n - 1), ph(n - 1), a.status, abort_flag);
                if (!__all_sync(kFullMask, ok)) { ok = false; break; }
                tc::fence_after_sync();
                {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        const uint32_t ta = tmem + lane_base + uint32_t(C::kOCol + 32 * c);
                        tc::tmem_ld32(ta, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                        tc::tmem_st32(ta, v);
                    }
                    tc::tmem_st_wait();
                }
            }
            tc::tmem_st_wait();
            tc::fence_before_sync();
            mbar_arrive(p_full(n));
        }
        // ---- epilogue: O of the last tile, divided by the row sum
        if (ok && n_tiles > 0) {
            ok = pf_wait(o_done(n_tiles - 1), ph(n_tiles - 1), a.status, abort_flag);
            ok = __all_sync(kFullMask, ok);
        }
        if (ok && n_tiles > 0) {
            tc::fence_after_sync();
            const bool store = t < un.n_q;
            const float inv = 1.f / l;
            const float lse2 = m + __log2f(l);
            const int64_t row = int64_t(un.q_row0 + t) * a.n_qo_heads + un.g * G + h;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + lane_base + uint32_t(C::kOCol + 32 * c), v);
                if (!store) continue;
                if (un.part >= 0) {  // a piece of a split range: fp32 partial result
                    float4* dst = reinterpret_cast<float4*>(
                        a.ws_o + (int64_t(un.part) * kPfRows + r) * D + 32 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(v[4 * i]) * inv, __uint_as_float(v[4 * i + 1]) * inv,
                                             __uint_as_float(v[4 * i + 2]) * inv, __uint_as_float(v[4 * i + 3]) * inv);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + row * D + 32 * c);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * i]) * inv, __uint_as_float(v[8 * i + 1]) * inv),
                                            pack_bf16x2(__uint_as_float(v[8 * i + 2]) * inv, __uint_as_float(v[8 * i + 3]) * inv),
                                            pack_bf16x2(__uint_as_float(v[8 * i + 4]) * inv, __uint_as_float(v[8 * i + 5]) * inv),
                                            pack_bf16x2(__uint_as_float(v[8 * i + 6]) * inv, __uint_as_float(v[8 * i + 7]) * inv));
                }
            }
            if (store) {
                if (un.part >= 0) a.ws_lse[int64_t(un.part) * kPfRows + r] = lse2;
                else if (a.lse != nullptr) a.lse[row] = lse2 * kLn2;
            }
        }
    }
    // every role is done with TMEM (and the MMAs have drained): free it
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kPfMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kPfTmemCols);
    }
}

// Log-sum-exp merge of split units: half a warp per (merge record, row of its 128),
// its 16 lanes over head_dim (D / 16 dims each), the pieces folded in chunks of
// kPfMergeChunk with every load of a chunk issued before any is used:
//     lse = log2 sum_c 2^lse_c,   out = sum_c 2^(lse_c - lse) out_c
// kept as a running maximum m, sum s = sum_c 2^(lse_c - m) and accumulator
// a = sum_c 2^(lse_c - m) out_c, rescaled when m grows. Few registers a thread, so a
// step's merges run in about one wave.
constexpr int kPfMergeWarps = 4;
constexpr int kPfMaxPieces = 16;  // pieces per split unit (the planner's cap)
constexpr int kPfMergeChunk = 4;  // pieces whose loads are in flight together

template <int D, int G>
__global__ void __launch_bounds__(32 * kPfMergeWarps) prefill_merge_kernel(const PfArgs a) {
    pdl_launch_dependents();
    constexpr int kVD = D / 16;  // dims per lane
    const int lane = threadIdx.x & 31;
    const int hw = (blockIdx.x * kPfMergeWarps + (threadIdx.x >> 5)) * 2 + (lane >> 4);  // half-warp
    if (hw >= a.n_merges * kPfRows) return;  // no warp-wide operation follows
    const PfMerge mg = a.merges[hw / kPfRows];  // plan data
    const int r = hw % kPfRows, t = r / G, h = r % G;
    if (t >= mg.n_q) return;
    const int d0 = (lane & 15) * kVD;
    pdl_wait();  // the pieces come from the kernel before
    float m = neg_inf(), sum = 0.f, acc[kVD];
#pragma unroll
    for (int i = 0; i < kVD; ++i) acc[i] = 0.f;
    for (int c0 = 0; c0 < mg.count; c0 += kPfMergeChunk) {
        float xl[kPfMergeChunk];
        float4 x[kPfMergeChunk][kVD / 4];
#pragma unroll
        for (int c = 0; c < kPfMergeChunk; ++c) {
            const bool in = c0 + c < mg.count;
            const int64_t wrow = int64_t(mg.first + (in ? c0 + c : 0)) * kPfRows + r;
            xl[c] = in ? __ldcg(a.ws_lse + wrow) : neg_inf();
#pragma unroll
            for (int i = 0; i < kVD / 4; ++i)
                x[c][i] = in ? __ldcg(reinterpret_cast<const float4*>(a.ws_o + wrow * D + d0) + i)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mc = m;
#pragma unroll
        for (int c = 0; c < kPfMergeChunk; ++c) mc = fmaxf(mc, xl[c]);
        const float scale = m == neg_inf() ? 0.f : ex2(m - mc);  // every piece has a finite lse
        sum *= scale;
#pragma unroll
        for (int i = 0; i < kVD; ++i) acc[i] *= scale;
#pragma unroll
        for (int c = 0; c < kPfMergeChunk; ++c) {
            const float wgt = ex2(xl[c] - mc);  // 0 for the chunk's padding
            sum += wgt;
#pragma unroll
            for (int i = 0; i < kVD / 4; ++i) {
                acc[4 * i] = fmaf(wgt, x[c][i].x, acc[4 * i]);
                acc[4 * i + 1] = fmaf(wgt, x[c][i].y, acc[4 * i + 1]);
                acc[4 * i + 2] = fmaf(wgt, x[c][i].z, acc[4 * i + 2]);
                acc[4 * i + 3] = fmaf(wgt, x[c][i].w, acc[4 * i + 3]);
            }
        }
        m = mc;
    }
    const float inv = 1.f / sum;
    const int64_t row = int64_t(mg.q_row0 + t) * a.n_qo_heads + mg.g * G + h;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + row * D + d0;
#pragma unroll
    for (int i = 0; i < kVD; i += 8)
        *reinterpret_cast<uint4*>(dst + i) =
            make_uint4(pack_bf16x2(acc[i] * inv, acc[i + 1] * inv), pack_bf16x2(acc[i + 2] * inv, acc[i + 3] * inv),
                       pack_bf16x2(acc[i + 4] * inv, acc[i + 5] * inv), pack_bf16x2(acc[i + 6] * inv, acc[i + 7] * inv));
    if (a.lse != nullptr && (lane & 15) == 0) a.lse[row] = (m + __log2f(sum)) * kLn2;
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
                                                      PfCfg<D, G>::kThreads, PfCfg<D, G>::kSmem) != cudaSuccess)
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
                   dim3(PfCfg<D, G>::kThreads), PfCfg<D, G>::kSmem, a, stream);
    if (e != cudaSuccess || a.n_merges == 0) return e;
    const int warps = (a.n_merges * kPfRows + 1) / 2;  // half a warp per row
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

// cuTensorMapEncodeTiled, reached through the runtime (no link against the driver
// library); NULL when the driver does not provide it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult found{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &found) != cudaSuccess ||
            found != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// Tensor map of a pool, [slots, cols] bf16 (every int32 slot id addressable; the
// kernel reads only listed slots), for 4-row gathers of 64-element panels: box
// 64 x 1, 128-byte swizzle.
bool encode_pool(CUtensorMap* map, const void* pool, uint64_t cols) {
    const EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, uint64_t(INT32_MAX)};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, 1};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box,
              elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    int tile_tokens = 0;  // query tokens per unit: 128 / G
    int max_units = 0;    // capacity of the unit list (tiles plus split pieces)
    int split_target = 0; // a step with fewer tile units than this splits long ranges
    int max_blocks = 0;   // workspace blocks of 128 rows (pieces of split units)
    int max_merges = 0;
    pkv::PfUnit* host_units = nullptr;  // pinned staging
    pkv::PfUnit* dev_units = nullptr;
    pkv::PfMerge* host_merges = nullptr;
    pkv::PfMerge* dev_merges = nullptr;
    float* ws_o = nullptr;
    float* ws_lse = nullptr;
    int* dev_status = nullptr;  // nonzero: a bounded wait of some CTA expired
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
    // Steps with fewer tile units than two waves of the grid (three at head_dim 256,
    // whose K/V tiles cost about twice as much per entry, so finer pieces pay for
    // their start-up; both measured best) split long causal ranges into pieces; a
    // split step has at most 2 x target pieces.
    p->split_target = (head_dim == 256 ? 3 : 2) * sms * per_sm;
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
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&p->dev_status), sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(p->dev_status, 0, sizeof(int));
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
    if (p->dev_status) cudaFree(p->dev_status);
    if (prev >= 0) cudaSetDevice(prev);
    delete p;
}

int paged_prefill_plan(pkv_prefill_plan* p, const int32_t* qo_indptr_host,
                       const int32_t* kv_indptr_host, int batch, pkv_stream_t stream) {
    TraceRange trace("paged_prefill_plan");
    clear_error();
    const char* who = "paged_prefill_plan";
    if (!p) return fail(PKV_ERR_PLAN, "%s: plan is NULL", who);
    p->planned = false;
    if (int rc = check_plan_device(who, p->device); rc != PKV_OK) return rc;
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

int paged_prefill_plan_status(pkv_prefill_plan* p, int* status) {
    clear_error();
    if (!p || !status) return fail(PKV_ERR_INVALID_ARG, "paged_prefill_plan_status: NULL argument");
    int v = 0;
    cudaError_t e = cudaMemcpy(&v, p->dev_status, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && v != 0) e = cudaMemset(p->dev_status, 0, sizeof v);
    if (e != cudaSuccess) return pf_cuda_fail(e, "paged_prefill_plan_status: read");
    *status = v;
    return PKV_OK;
}

int paged_prefill_attn(const void* q, const void* k_pool, const void* v_pool,
                       const int32_t* qo_indptr, const int32_t* kv_indptr,
                       const int32_t* kv_indices, int batch, int n_qo_heads, int n_kv_heads,
                       int head_dim, float sm_scale, void* out, float* lse,
                       const pkv_prefill_plan* p, pkv_stream_t stream) {
    TraceRange trace("paged_prefill_attn");
    clear_error();
    const char* who = "paged_prefill_attn";
    if (!p || !p->planned) return fail(PKV_ERR_PLAN, "%s: plan is NULL or not planned", who);
    if (int rc = check_plan_device(who, p->device); rc != PKV_OK) return rc;
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
        if (int rc = check_on_device(who, p->device,
                                     {{"q", q}, {"k_pool", k_pool}, {"v_pool", v_pool},
                                      {"qo_indptr", qo_indptr}, {"kv_indptr", kv_indptr},
                                      {"kv_indices", kv_indices}, {"out", out}, {"lse", lse}});
            rc != PKV_OK)
            return rc;
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
    a.status = p->dev_status;
    if (pf_tma_tokens(head_dim) > 0) {
        const uint64_t cols = uint64_t(n_kv_heads) * uint64_t(head_dim);
        if (!encode_pool(&a.maps.k, k_pool, cols) || !encode_pool(&a.maps.v, v_pool, cols))
            return fail(PKV_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed for the pools", who);
    }
    a.withhold = take_injected_stall();
    const cudaError_t e = prefill_dispatch<PfLaunchFn>(head_dim, n_qo_heads / n_kv_heads, a,
                                                       p->n_units, stream);
    if (e != cudaSuccess) return pf_cuda_fail(e, "paged_prefill_attn: launch");
    return PKV_OK;
}

}  // extern "C"
