// Split-KV paged decode attention with grouped-query heads, and the LSE merge of
// split contexts.
//
// What is computed ("Agent-Infer: 纯 Rust 编写的高性能 LLM 推理引擎", section
// "分页 KV 缓存": batched decode over a page-size-1 token pool; "Pegainfer:
// 纯Rust+CUDA构建的LLM推理引擎", section "1. 注意力机制优化": 32 query heads share 8
// KV heads, head_dim 128; section "2. Qwen3.5的混合架构支持": head_dim 256):
// for request b and query head h (KV head g = h / G),
//     out[b,h] = softmax_j(sm_scale * q[b,h] . K[idx_j, g]) . V[idx_j, g]
//     lse[b,h] = ln sum_j exp(sm_scale * q[b,h] . K[idx_j, g]).
//
// Design for sm_103a. The kernel is HBM-bound (about G flops per byte of K/V), so
// everything serves the gather of scattered pool rows:
//  * Persistent CTAs (two per SM), each walking the list of work units the
//    per-step plan gave it. A unit is a token range of one request for one
//    KV-head group of up to 512 bf16 per token (4 heads at head_dim 128, 2 at
//    256), so one token's K (or V) row of the group is one contiguous 1 KB run of
//    the pool.
//  * Warp specialisation: two producer warps turn slot ids into 1D bulk copies
//    (cp.async.bulk, the TMA engine) of whole rows into a 3-stage shared-memory
//    ring of 16-token tiles, signalled by mbarrier transaction counts; each
//    stage's 32 row copies (16 K rows, 16 V rows) are shared between them. One
//    warp alone issues only about 25 bulk copies per microsecond, which at 1 KB
//    per copy is below the HBM rate of an SM's two CTAs. Four consumer warps take
//    the tiles. Up to 3 x 32 KB per CTA is in flight, which covers HBM latency
//    with two CTAs per SM. The slot ids themselves travel kStages + 1 stages
//    ahead of the copies (cp.async into a small shared ring per producer warp),
//    so no stage waits a round trip for its ids. Rows read once carry an L2 evict-first policy; rows
//    of a shared prefix, which the group's other prefix units read again,
//    evict-last.
//  * Programmatic dependent launch: the plan is read before waiting for the
//    previous kernel; with PKV_PLAN_EARLY_GATHER the slot ids and old pool rows
//    are too, so a layer's ring fills while the kernel ahead of it finishes.
//  * The consumers use the tensor cores for the two small contractions of a GQA
//    group, so that all G query heads are served by one read of each K/V row and
//    the instruction count per byte stays far below the issue rate:
//      S^T[16 tokens x 8 heads]  = K_tile[16 x D] . Q^T[D x 8]     (mma m16n8k16)
//      O^T[D x 8 heads]         += V_tile^T[D x 16] . P^T[16 x 8]
//    K and V tiles come from shared memory with ldmatrix (V transposed on the
//    fly), q stays in registers for the whole unit, and the probabilities move
//    from the S^T accumulator layout to the P^T operand layout with movmatrix.
//    Heads beyond G in the 8-wide tile are zero padding.
//  * Online softmax in base 2 (scores times sm_scale * log2 e), fp32 state per
//    head; the output accumulators are rescaled only when some running maximum
//    moved.
//  * A unit covering a whole context writes bf16 out and lse directly. A unit
//    covering part of one writes its normalised fp32 output and base-2 lse to the
//    plan's workspace; a second, small kernel merges the parts of every split
//    context by the log-sum-exp identity
//        lse = log2 sum_c 2^lse_c,   out = sum_c 2^(lse_c - lse) out_c
//    with one warp per (context, query head), all parts' loads in flight at once.
//  * Every wait on an mbarrier is bounded (1 s); on expiry the kernel sets the
//    plan's status word, stops, and waits (again bounded) for its own copies in
//    flight before exiting.
//  * Host KV tier: a negative slot id names a row of pinned host pools, which the
//    producer warp's lanes copy together over NVLink-C2C with 16-byte cp.async (the
//    stage barrier counts one arrival per lane for them).
//  * Small steps run as one launch of a second kernel on thread-block clusters of 16
//    CTAs (one cluster per request and head group, no work list): each CTA reads
//    kv_indptr, takes a share of the slot list, and the cluster merges its parts
//    through distributed shared memory (see paged_decode_small_kernel).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

using namespace ptx;

constexpr int kTile = 16;           // tokens per pipeline stage (one mma M block)
constexpr int kGroupWarps = 4;      // consumer warps that cover one head group's rows of q
constexpr int kRowPad = 16;         // bytes between staged rows: conflict-free ldmatrix
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
constexpr int kProducersPerBlock = 2;  // producer warps per CTA

// ---------------------------------------------------------------------------
// bounded waits (PTX ISA: mbarrier.try_wait, %globaltimer)
// ---------------------------------------------------------------------------

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase of `bar` with the given parity. Returns false (and
// raises the CTA's abort flag and the status word) if it does not complete
// within kWaitLimitNs, or if another warp of the CTA already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status,
                                          volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, 1);
            *abort_flag = 1;
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// kernel
// ---------------------------------------------------------------------------

// Shapes of one instance: head_dim D, GQA group G, WPH consumer warps per KV
// head (so 4 / WPH KV heads per CTA) and NB 8-row query blocks per warp. A unit's
// query rows (row r = head r % G of its request r / G) are 8 NB per warp, so a
// unit serves 8 NB / G requests (NB = 2: the shared-prefix instance). Two CTAs run
// per SM. A pipeline stage holds kSub 16-token sub-tiles of K rows and of V rows
// of the CTA's kHeadsPerCta heads; kSub is chosen so that every stage carries
// 16 x kHeadGroupElems bf16 of K and as much of V (32 KB, plus row padding)
// whatever the head count.
template <int D, int G, int WPH, int NB = 1>
struct Cfg {
    static constexpr int kConsumerWarps = kGroupWarps;
    static constexpr int kProducerWarps = kProducersPerBlock;  // each issues 1 / P of the copies
    static constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
    static constexpr int kStages = 3;                           // 32 KB stages in flight
    static constexpr int kMinBlocks = 2;                        // resident CTAs per SM
    static constexpr int kWarpRows = 8 * NB;                    // query rows of one warp
    static constexpr int kHeadsPerCta = kGroupWarps / WPH;      // KV heads of one group
    static constexpr int kRow = kHeadsPerCta * D * 2;           // bytes of a staged row
    static constexpr int kRowP = kRow + kRowPad;
    static constexpr int kSub = kHeadGroupElems / (kHeadsPerCta * D);  // sub-tiles per stage
    static constexpr int kStageTokens = kTile * kSub;
    static constexpr int kStage = 2 * kStageTokens * kRowP;     // K rows then V rows
    static constexpr uint32_t kStageTx = 2u * kStageTokens * kRow;
    static constexpr int kKSteps = D / 16;                      // k-steps of S^T
    static constexpr int kMBlocks = D / 16 / WPH;               // O^T dim blocks per warp
    static constexpr int kDimsPerWarp = D / WPH;
    static constexpr int kQHeads = kHeadsPerCta * G;            // query heads of a group
    static constexpr int kAhead = kStages + 1;                  // stages of slot ids in flight
    // With early gather, the stages issued before the previous kernel has completed:
    // one fewer than the ring holds, so the next layer's start loads less of the
    // memory system while the previous layer's merge runs (measured faster than a
    // full ring or a single stage on the Qwen3-4B-shaped step)
    static constexpr int kEarlyStages = kStages - 1;
    static constexpr int kBarOffset = kStages * kStage;
    static constexpr int kIdxOffset = kBarOffset + 2 * kStages * 8 + 16;
    // copies of one stage: K then V rows of kStageTokens tokens; copy c is issued by
    // producer warp c % P, lane (c / P) % 32
    static constexpr int kCopies = 2 * kStageTokens;
    static constexpr int kCopiesPerLane = (kCopies / kProducerWarps + 31) / 32;
    static constexpr int kIdRing = kAhead * kStageTokens * 4;  // slot-id ring of one producer warp
    static constexpr int kSmem = kIdxOffset + kProducerWarps * kIdRing;
    static_assert(G >= 1 && G <= 8, "group size");
    static_assert(NB == 1 || NB == 2, "query blocks");
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    static_assert(kCopies % kProducerWarps == 0, "copies split evenly over the producer warps");
    static_assert(kHeadsPerCta * D * kSub == kHeadGroupElems, "stage budget");
    static_assert(kMBlocks >= 1, "dims per warp");
};

// Shared memory of the single-launch kernel for small steps: Cfg's layout, its one
// work unit, and its partial result as [kQHeads][D] fp32 then the kQHeads base-2 lse
// values (a region of its own, so each consumer warp writes its rows as soon as it
// is done). Two CTAs share an SM where both fit.
template <int D, int G, int WPH>
struct SmallCfg {
    using C = Cfg<D, G, WPH, 1>;
    static constexpr int kUnitOffset = (C::kSmem + 15) / 16 * 16;
    static constexpr int kPartOffset = kUnitOffset + 32;
    static constexpr int kPartBytes = C::kQHeads * D * 4 + C::kQHeads * 4;
    static constexpr int kSmem = kPartOffset + kPartBytes;
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

struct Shared {
    uint64_t* full;
    uint64_t* empty;
    volatile int* flags;  // [0] abort
    const Unit* units;    // the CTA's work units (the plan's list, or one built on the device)
    int part_offset;      // single-launch steps: shared-memory offset of the partial result
};

__device__ __forceinline__ int unit_stages(const Unit& un, int stage_tokens) {
    const int n_tok = un.tok_end - un.tok_begin;
    return n_tok > 0 ? (n_tok + stage_tokens - 1) / stage_tokens : 1;
}

// The slot ids of the stages ahead of the copies: the producer walks the CTA's
// stages twice, once here to start the slot-id loads (cp.async into a shared-memory
// ring of kAhead stages) and kAhead stages later to issue the row copies, so a
// stage's copies never wait a round trip for its slot ids.
struct SlotFetch {
    int u, t, n_stages;  // next stage to fetch: stage t of unit u
    Unit un;
    int pos;             // its place in the ring
};

template <class C>
__device__ __forceinline__ void fetch_slot_ids(const DecodeArgs& a, SlotFetch& f, int u_end,
                                               int lane, uint32_t ring, const Unit* units) {
    if (f.u < u_end) {
        const int n = min(C::kStageTokens, (f.un.tok_end - f.un.tok_begin) - f.t * C::kStageTokens);
        const int32_t* idx = a.kv_indices + f.un.idx_begin + f.t * C::kStageTokens;
        const uint32_t dst = ring + f.pos * C::kStageTokens * 4;
        for (int i = lane; i < n; i += 32) cp_async4(dst + 4 * i, idx + i);
        if (++f.t == f.n_stages) {
            f.t = 0;
            if (++f.u < u_end) {
                f.un = units[f.u];
                f.n_stages = unit_stages(f.un, C::kStageTokens);
            }
        }
    }
    cp_async_commit();  // one group per stage (empty past the end)
    if (++f.pos == C::kAhead) f.pos = 0;
}

// Producer warps: copy c of a stage (c < kStageTokens: token c's K row, else token
// c - kStageTokens's V row of the CTA's head group) is issued by warp c % P, lane
// (c / P) % 32, so the P warps share each stage's copies. Each warp arrives on the
// stage's full barrier with the bytes of its own copies and keeps its own ring of
// slot ids.
template <int D, int G, int WPH, int NB>
__device__ void producer_warp(const DecodeArgs& a, uint8_t* smem, const Shared& sh, int u_begin,
                              int u_end) {
    using C = Cfg<D, G, WPH, NB>;
    constexpr int P = C::kProducerWarps;
    const int lane = threadIdx.x & 31;
    const int pw = (threadIdx.x >> 5) - C::kConsumerWarps;  // producer warp index
    const bool fused = a.k_new != nullptr;
    const bool tiered = a.k_host != nullptr;
    const int64_t slot_bytes = int64_t(a.n_kv_heads) * D * 2;
    // this lane's copies: token, K or V, and shared-memory offset within a stage
    int tok[C::kCopiesPerLane];
    bool is_v[C::kCopiesPerLane], has[C::kCopiesPerLane];
    uint32_t dst[C::kCopiesPerLane];
#pragma unroll
    for (int i = 0; i < C::kCopiesPerLane; ++i) {
        const int c = pw + P * (lane + 32 * i);
        has[i] = c < C::kCopies;
        is_v[i] = c >= C::kStageTokens;
        tok[i] = is_v[i] ? c - C::kStageTokens : c;
        dst[i] = smem_u32(smem) + (is_v[i] ? C::kStageTokens * C::kRowP : 0) + tok[i] * C::kRowP;
    }
    const uint32_t id_ring = smem_u32(smem) + C::kIdxOffset + pw * C::kIdRing;
    const int32_t* id_ring_ptr = reinterpret_cast<const int32_t*>(smem + C::kIdxOffset + pw * C::kIdRing);
    const uint64_t stream_policy = policy_evict_first();
    const uint64_t shared_policy = policy_evict_last();
    int stage = 0;
    uint32_t empty_parity = 1;  // a fresh barrier reports the phase before it as complete
    uint32_t fill_parity = 0;
    uint32_t filled_mask = 0, parity_bits = 0;  // per stage: filled at all / parity of last fill
    bool aborted = false;
    // The next unit's descriptor is loaded one unit ahead, and (by the first producer
    // warp) its slot ids are prefetched into L2 once the current unit's first stage
    // is on its way.
    if (a.withhold) return;  // injected stall: the consumers' waits expire (bounded)
    Unit next = u_begin < u_end ? sh.units[u_begin] : Unit{};
    // Slot ids and pool rows may come from the previous kernel: wait for it, after
    // warming L2 with the first unit's slot ids (prefetches are hints, not reads).
    // With early gather they were final before the step's plan upload, so the
    // loads start at once and only the fused append's new rows wait.
    bool waited = !a.early;
    if (u_begin < u_end && pw == 0)
        for (int off = 32 * lane; off < next.tok_end - next.tok_begin && off < 32 * 32 * 4;
             off += 32 * 32)
            prefetch_l2(a.kv_indices + next.idx_begin + off);
    if (waited) pdl_wait();
    SlotFetch f{u_begin, 0, u_begin < u_end ? unit_stages(next, C::kStageTokens) : 0, next, 0};
#pragma unroll 1
    for (int i = 0; i < C::kAhead; ++i) fetch_slot_ids<C>(a, f, u_end, lane, id_ring, sh.units);
    int pos = 0;     // ring place of the stage being issued
    int issued = 0;  // stages issued so far
    for (int u = u_begin; u < u_end && !aborted; ++u) {
        const Unit un = next;
        if (u + 1 < u_end) next = sh.units[u + 1];
        const int32_t* idx = a.kv_indices + un.idx_begin;
        const int n_tok = un.tok_end - un.tok_begin;
        const int n_stages = unit_stages(un, C::kStageTokens);
        const int64_t group_off = int64_t(un.hg) * C::kRow;
        const uint64_t policy = un.len == -2 ? shared_policy : stream_policy;
        if (pw == 0)
            for (int off = 32 * (lane + 1); off < n_tok; off += 32 * 32) prefetch_l2(idx + off);
        for (int t = 0; t < n_stages; ++t) {
            if (pw == 0 && t == (n_stages > 1 ? 1 : 0) && u + 1 < u_end) {
                const int32_t* nidx = a.kv_indices + next.idx_begin;
                for (int off = 32 * lane; off < next.tok_end - next.tok_begin; off += 32 * 32)
                    prefetch_l2(nidx + off);
            }
            const int n = min(C::kStageTokens, n_tok - t * C::kStageTokens);
            const uint32_t full_bar = smem_u32(&sh.full[stage]);
            if (lane == 0 && !mbar_wait(smem_u32(&sh.empty[stage]), empty_parity, a.status, sh.flags))
                sh.flags[0] = 1;
            __syncwarp();
            if (sh.flags[0]) {
                aborted = true;
                break;
            }
            // this stage's slot ids (the oldest group in flight) have landed
            cp_async_wait<C::kAhead - 1>();
            __syncwarp();
            // slot id of each copy of this lane; a copy past the stage's tokens pads
            // the tile with the zero row
            int slot[C::kCopiesPerLane];
            bool row[C::kCopiesPerLane];
#pragma unroll
            for (int i = 0; i < C::kCopiesPerLane; ++i) {
                row[i] = has[i] && tok[i] < n;
                slot[i] = row[i] ? id_ring_ptr[pos * C::kStageTokens + tok[i]] : 0;
            }
            __syncwarp();  // every lane has read its ids before the place is refilled below
            if (!waited && issued == C::kEarlyStages) {
                pdl_wait();
                waited = true;
            }
            ++issued;
            // k_new / v_new may come from the previous kernel
            const int first = un.tok_begin + t * C::kStageTokens;
            if (!waited && fused && un.len - 1 >= first && un.len - 1 < first + n) {
                pdl_wait();
                waited = true;
            }
            if (!tiered) {
                if (lane == 0) mbar_arrive_expect_tx(full_bar, n > 0 ? C::kStageTx / P : 0u);
                __syncwarp();
                if (n > 0) {
#pragma unroll
                    for (int i = 0; i < C::kCopiesPerLane; ++i) {
                        if (!has[i]) continue;
                        const char* pool = static_cast<const char*>(is_v[i] ? a.v_pool : a.k_pool);
                        const void* src = row[i] ? static_cast<const void*>(pool + slot[i] * slot_bytes + group_off)
                                                 : a.zero_row;
                        // fused append: the request's newest token comes from its new row
                        if (fused && first + tok[i] == un.len - 1)
                            src = static_cast<const char*>(is_v[i] ? a.v_new : a.k_new) + un.b * slot_bytes +
                                  group_off;
                        bulk_g2s_hint(dst[i] + stage * C::kStage, src, C::kRow, full_bar, policy);
                    }
                }
            } else {
                // Host KV tier: a negative slot id -1 - h names row h of the pinned host
                // pools, read over NVLink-C2C by the warp's lanes together with 16-byte
                // cp.async (each row 16 bytes a lane); the other rows are bulk copies.
                // The barrier tracks the lanes' copies (one .noinc arrival per lane and
                // stage) and the bulk bytes.
                bool by_lanes[C::kCopiesPerLane];
                int n_by_lanes = 0;
#pragma unroll
                for (int i = 0; i < C::kCopiesPerLane; ++i) {
                    by_lanes[i] = n > 0 && has[i] && row[i] && slot[i] < 0;
                    n_by_lanes += by_lanes[i] ? 1 : 0;
                }
                const int warp_by_lanes = __reduce_add_sync(kFull, n_by_lanes);
                if (lane == 0)
                    mbar_arrive_expect_tx(full_bar,
                                          n > 0 ? C::kStageTx / P - uint32_t(warp_by_lanes) * C::kRow : 0u);
                __syncwarp();
                if (n > 0) {
#pragma unroll
                    for (int i = 0; i < C::kCopiesPerLane; ++i) {
                        const char* src = nullptr;
                        if (has[i]) {
                            if (tiered && row[i] && slot[i] < 0) {
                                src = static_cast<const char*>(is_v[i] ? a.v_host : a.k_host) +
                                      int64_t(-1 - slot[i]) * slot_bytes + group_off;
                            } else {
                                const char* pool = static_cast<const char*>(is_v[i] ? a.v_pool : a.k_pool);
                                src = row[i] ? pool + slot[i] * slot_bytes + group_off
                                             : static_cast<const char*>(a.zero_row);
                                // fused append: the request's newest token comes from its new row
                                if (fused && first + tok[i] == un.len - 1)
                                    src = static_cast<const char*>(is_v[i] ? a.v_new : a.k_new) +
                                          un.b * slot_bytes + group_off;
                            }
                        }
                        const uint32_t d_mine = dst[i] + stage * C::kStage;
                        if (has[i] && !by_lanes[i]) bulk_g2s_hint(d_mine, src, C::kRow, full_bar, policy);
                        // the rows of copy i of every lane, one after another, 16 bytes a lane
                        unsigned todo = __ballot_sync(kFull, by_lanes[i]);
                        while (todo) {
                            const int l = __ffs(todo) - 1;
                            todo &= todo - 1;
                            const char* s = reinterpret_cast<const char*>(
                                __shfl_sync(kFull, reinterpret_cast<unsigned long long>(src), l));
                            const uint32_t d = __shfl_sync(kFull, d_mine, l);
                            for (int c = lane; c < C::kRow / 16; c += 32) cp_async16(d + 16 * c, s + 16 * c, true);
                        }
                    }
                }
                cp_async_arrive_noinc(full_bar);  // fires once this lane's copies have landed
            }
            fetch_slot_ids<C>(a, f, u_end, lane, id_ring, sh.units);  // refills place `pos`
            if (++pos == C::kAhead) pos = 0;
            filled_mask |= 1u << stage;
            parity_bits = (parity_bits & ~(1u << stage)) | (fill_parity << stage);
            if (++stage == C::kStages) {
                stage = 0;
                empty_parity ^= 1;
                fill_parity ^= 1;
            }
        }
    }
    // No copy (bulk or slot-id) may still be writing this CTA's shared memory when
    // it exits.
    cp_async_wait<0>();
    if (lane == 0) {
        for (int s = 0; s < C::kStages; ++s)
            if (filled_mask & (1u << s)) {
                const uint32_t bar = smem_u32(&sh.full[s]);
                const uint32_t par = (parity_bits >> s) & 1u;
                if (!mbar_try_wait(bar, par)) {
                    const unsigned long long t0 = global_ns();
                    while (!mbar_try_wait(bar, par) && global_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
    }
}

// Q^T as the B operand of S^T = K Q^T: query block nb of a warp with row base r0
// holds the rows r0 + 8 nb .. r0 + 8 nb + 7 of the unit's query set, row r being
// head r % G of request b + r / G; lane l holds row r0 + 8 nb + l / 4, dims
// 2 (l % 4) .. of each k-step. Rows beyond the unit's requests are zero.
template <int D, int G, int WPH, int NB>
__device__ __forceinline__ void load_q_fragments(const DecodeArgs& a, const Unit& un, int hh, int r0,
                                                 int g, int t4,
                                                 uint32_t (&qf)[NB][Cfg<D, G, WPH, NB>::kKSteps][2]) {
    using C = Cfg<D, G, WPH, NB>;
    const int kvh = un.hg * C::kHeadsPerCta + hh;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int r = r0 + 8 * nb + g;
        const bool valid = r / G < un.nreq;
        const uint32_t* row = reinterpret_cast<const uint32_t*>(
            static_cast<const __nv_bfloat16*>(a.q) +
            (int64_t(un.b + (valid ? r / G : 0)) * a.n_qo_heads + kvh * G + r % G) * D + 2 * t4);
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
            qf[nb][ks][0] = valid ? __ldg(row + ks * 8) : 0u;
            qf[nb][ks][1] = valid ? __ldg(row + ks * 8 + 4) : 0u;
        }
    }
}

// Fused append: copy this warp's part (head hh, dims of `part`) of the staged new
// K and V rows of request un.b from shared memory to pool slot slot_ids[un.b].
template <int D, int G, int WPH, int NB>
__device__ __forceinline__ void store_new_rows(const DecodeArgs& a, const Unit& un,
                                               const uint8_t* smem, int stage, int row, int hh,
                                               int part, int lane) {
    using C = Cfg<D, G, WPH, NB>;
    constexpr int kBytes = C::kDimsPerWarp * 2;  // bytes of this warp's share of one row
    const int64_t slot = __ldg(a.slot_ids + un.b);
    const int64_t dst_off = slot * int64_t(a.n_kv_heads) * D * 2 +
                            (int64_t(un.hg) * C::kHeadsPerCta + hh) * D * 2 + part * kBytes;
    const uint8_t* src_row = smem + stage * C::kStage + row * C::kRowP + (hh * D) * 2 + part * kBytes;
    for (int off = lane * 16; off < 2 * kBytes; off += 32 * 16) {
        const bool is_v = off >= kBytes;
        const int o = is_v ? off - kBytes : off;
        const uint4 v = *reinterpret_cast<const uint4*>(src_row + (is_v ? C::kStageTokens * C::kRowP : 0) + o);
        char* pool = static_cast<char*>(const_cast<void*>(is_v ? a.v_pool : a.k_pool));
        *reinterpret_cast<uint4*>(pool + dst_off + o) = v;
    }
}

// kSmall: the single-launch kernel for small steps, whose one unit writes its partial
// result to the CTA's shared memory for the cluster's merge.
template <int D, int G, int WPH, int NB, bool kSmall = false>
__device__ void consumer_warp(const DecodeArgs& a, uint8_t* smem, const Shared& sh, int u_begin,
                              int u_end) {
    using C = Cfg<D, G, WPH, NB>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hh = warp / WPH;    // KV head within the group
    const int part = warp % WPH;  // which slice of head_dim this warp accumulates
    const int g = lane >> 2, t4 = lane & 3;
    const int hq = a.n_qo_heads;
    const float scale_log2 = a.sm_scale * kLog2e;
    // ldmatrix row addresses within a stage (see the fragment layouts of mma.m16n8k16):
    // K tile as the A operand (rows = tokens, k = dims)
    const uint32_t k_lane = smem_u32(smem) + ((lane & 7) + ((lane >> 3) & 1) * 8) * C::kRowP +
                            (hh * D + (lane >> 4) * 8) * 2;
    // V tile, transposed on load, as the A operand (rows = dims, k = tokens)
    const uint32_t v_lane = smem_u32(smem) + C::kStageTokens * C::kRowP +
                            ((lane & 7) + (lane >> 4) * 8) * C::kRowP +
                            (hh * D + part * C::kDimsPerWarp + ((lane >> 3) & 1) * 8) * 2;
    int stage = 0;
    uint32_t full_parity = 0;

    // With one query block the next unit's q fragments are loaded while the current
    // unit streams; with two (shared prefixes) they are loaded at the unit's start.
    constexpr bool kPrefetchQ = NB == 1;
    uint32_t qb[NB][C::kKSteps][2], qn[NB][C::kKSteps][2];
    Unit next = u_begin < u_end ? sh.units[u_begin] : Unit{};
    // Warm L2 with the first unit's q rows (a hint, safe before the wait): lane l
    // touches query row l of this warp's KV head.
    if (u_begin < u_end && lane < C::kWarpRows && lane / G < next.nreq) {
        const int kvh = next.hg * C::kHeadsPerCta + hh;
        const int r = lane;
        prefetch_l2(static_cast<const __nv_bfloat16*>(a.q) +
                    (int64_t(next.b + r / G) * a.n_qo_heads + kvh * G + r % G) * D);
    }
    pdl_wait();  // q may come from the previous kernel
    if constexpr (kPrefetchQ) {
        if (u_begin < u_end) load_q_fragments<D, G, WPH, NB>(a, next, hh, 0, g, t4, qn);
    }
    for (int u = u_begin; u < u_end; ++u) {
        const Unit un = next;
        const int kvh = un.hg * C::kHeadsPerCta + hh;
        constexpr int r0 = 0;  // first query row of this warp
        if constexpr (kPrefetchQ) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int ks = 0; ks < C::kKSteps; ++ks) {
                    qb[nb][ks][0] = qn[nb][ks][0];
                    qb[nb][ks][1] = qn[nb][ks][1];
                }
        } else {
            load_q_fragments<D, G, WPH, NB>(a, un, hh, r0, g, t4, qb);
        }
        if (u + 1 < u_end) {
            next = sh.units[u + 1];
            if constexpr (kPrefetchQ) load_q_fragments<D, G, WPH, NB>(a, next, hh, r0, g, t4, qn);
        }
        // A warp whose rows are all beyond the unit's requests only passes the stages on.
        const bool active = r0 / G < un.nreq;
        // softmax state per query block and column (heads 2 t4, 2 t4 + 1 of the block)
        float m[NB][2], l[NB][2];
        float o[NB][C::kMBlocks][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            m[nb][0] = m[nb][1] = neg_inf();
            l[nb][0] = l[nb][1] = 0.f;
#pragma unroll
            for (int mb = 0; mb < C::kMBlocks; ++mb)
                o[nb][mb][0] = o[nb][mb][1] = o[nb][mb][2] = o[nb][mb][3] = 0.f;
        }

        const int n_tok = un.tok_end - un.tok_begin;
        const int n_stages = n_tok > 0 ? (n_tok + C::kStageTokens - 1) / C::kStageTokens : 1;
        for (int t = 0; t < n_stages; ++t) {
            const bool ok = mbar_wait(smem_u32(&sh.full[stage]), full_parity, a.status, sh.flags);
            if (!__all_sync(kFull, ok)) return;  // uniform exit: no lane is left in a shuffle
            const int n_stage = n_tok - t * C::kStageTokens;
            // Fused append: the stage holding the request's newest token has its new
            // K/V rows (copied from k_new / v_new); each warp writes its share of them
            // to the pool slot before the stage is released.
            if (a.k_new != nullptr) {
                const int row = un.len - 1 - (un.tok_begin + t * C::kStageTokens);
                if (row >= 0 && row < n_stage && row < C::kStageTokens)
                    store_new_rows<D, G, WPH, NB>(a, un, smem, stage, row, hh, part, lane);
            }
#pragma unroll
            for (int j = 0; j < C::kSub; ++j) {
                const int n = active ? n_stage - j * kTile : 0;  // valid rows of this sub-tile
                if (n <= 0) break;
                const uint32_t st = stage * C::kStage + j * kTile * C::kRowP;
                float s[NB][4];
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < C::kKSteps; ++ks) {
                    uint32_t ka[4];
                    ldsm_x4(k_lane + st + ks * 32, ka);
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) mma_bf16(s[nb], ka, qb[nb][ks][0], qb[nb][ks][1]);
                }
                uint32_t pb[NB][2];
                bool rescale = false;
                float al[NB][2];
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    // s[nb][0], [1]: token g, columns 2t4, 2t4+1; [2], [3]: token g + 8
                    const float x0 = g < n ? s[nb][0] * scale_log2 : neg_inf();
                    const float x1 = g < n ? s[nb][1] * scale_log2 : neg_inf();
                    const float x2 = g + 8 < n ? s[nb][2] * scale_log2 : neg_inf();
                    const float x3 = g + 8 < n ? s[nb][3] * scale_log2 : neg_inf();
                    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
                    }
                    const float mn0 = fmaxf(m[nb][0], mx0), mn1 = fmaxf(m[nb][1], mx1);
                    al[nb][0] = ex2(m[nb][0] - mn0);
                    al[nb][1] = ex2(m[nb][1] - mn1);
                    rescale |= (al[nb][0] != 1.f) || (al[nb][1] != 1.f);
                    m[nb][0] = mn0;
                    m[nb][1] = mn1;
                    const float p0 = ex2(x0 - mn0), p1 = ex2(x1 - mn1);
                    const float p2 = ex2(x2 - mn0), p3 = ex2(x3 - mn1);
                    l[nb][0] = fmaf(l[nb][0], al[nb][0], p0 + p2);
                    l[nb][1] = fmaf(l[nb][1], al[nb][1], p1 + p3);
                    // P^T operand: tokens 0-7 and 8-15 of the sub-tile, rows in columns
                    pb[nb][0] = movmatrix_trans(pack_bf16x2(p0, p1));
                    pb[nb][1] = movmatrix_trans(pack_bf16x2(p2, p3));
                }
                if (__any_sync(kFull, rescale)) {
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                        for (int mb = 0; mb < C::kMBlocks; ++mb) {
                            o[nb][mb][0] *= al[nb][0];
                            o[nb][mb][1] *= al[nb][1];
                            o[nb][mb][2] *= al[nb][0];
                            o[nb][mb][3] *= al[nb][1];
                        }
                }
#pragma unroll
                for (int mb = 0; mb < C::kMBlocks; ++mb) {
                    uint32_t va[4];
                    ldsm_x4_trans(v_lane + st + mb * 32, va);
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) mma_bf16(o[nb][mb], va, pb[nb][0], pb[nb][1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.empty[stage]));
            if (++stage == C::kStages) {
                stage = 0;
                full_parity ^= 1;
            }
        }

        // ---- epilogue: o[nb][mb][0..3] = (dim 16*mb' + g (+8), rows r0 + 8nb + 2t4, +1)
        if (!active) continue;
        const int dim0 = part * C::kDimsPerWarp + g;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
            for (int jc = 0; jc < 2; ++jc) {
                float lt = l[nb][jc];
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) lt += __shfl_xor_sync(kFull, lt, off);
                const int r = r0 + 8 * nb + 2 * t4 + jc;
                const int req = r / G, h = r % G;
                if (req >= un.nreq) continue;
                const float inv = lt == 0.f ? 0.f : 1.f / lt;
                const float lse2 = lt == 0.f ? neg_inf() : m[nb][jc] + __log2f(lt);
                if (un.partial < 0) {
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) +
                                         (int64_t(un.b + req) * hq + kvh * G + h) * D + dim0;
#pragma unroll
                    for (int mb = 0; mb < C::kMBlocks; ++mb) {
                        dst[mb * 16] = __float2bfloat16_rn(o[nb][mb][jc] * inv);
                        dst[mb * 16 + 8] = __float2bfloat16_rn(o[nb][mb][2 + jc] * inv);
                    }
                    if (a.lse != nullptr && part == 0 && g == 0)
                        a.lse[int64_t(un.b + req) * hq + kvh * G + h] = lse2 * kLn2;
                } else {
                    const int64_t prow = kSmall ? hh * G + h
                                                : int64_t(un.partial + req) * C::kQHeads + hh * G + h;
                    float* part_o = kSmall ? reinterpret_cast<float*>(smem + sh.part_offset) : a.ws_o;
                    float* part_lse = kSmall ? part_o + C::kQHeads * D : a.ws_lse;
                    float* dst = part_o + prow * D + dim0;
#pragma unroll
                    for (int mb = 0; mb < C::kMBlocks; ++mb) {
                        dst[mb * 16] = o[nb][mb][jc] * inv;
                        dst[mb * 16 + 8] = o[nb][mb][2 + jc] * inv;
                    }
                    if (part == 0 && g == 0) part_lse[prow] = lse2;
                }
            }
        }
    }
}

template <int D, int G, int WPH, int NB>
__global__ void __launch_bounds__(Cfg<D, G, WPH, NB>::kThreads, Cfg<D, G, WPH, NB>::kMinBlocks)
    paged_decode_kernel(const DecodeArgs a) {
    using C = Cfg<D, G, WPH, NB>;
    extern __shared__ __align__(128) uint8_t smem[];
    Shared sh;
    sh.full = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    sh.empty = sh.full + C::kStages;
    sh.flags = reinterpret_cast<volatile int*>(sh.full + 2 * C::kStages);
    sh.units = a.units;
    sh.part_offset = 0;
    if (threadIdx.x == 0) {
        // a stage completes on one arrival per producer warp (plus, with the host KV
        // tier, one per producer lane for its cp.async copies) and the bulk bytes
        const uint32_t full_arrivals = C::kProducerWarps * (a.k_host != nullptr ? 33 : 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), full_arrivals);
            mbar_init(smem_u32(&sh.empty[s]), C::kConsumerWarps);
        }
        sh.flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Only plan data (uploaded before the previous kernel ran) is read before
    // each role's pdl_wait(), so the next kernel may be scheduled right away.
    pdl_launch_dependents();
    const int u_begin = a.cta_begin[blockIdx.x];
    const int u_end = a.cta_begin[blockIdx.x + 1];
    if ((threadIdx.x >> 5) >= C::kConsumerWarps)
        producer_warp<D, G, WPH, NB>(a, smem, sh, u_begin, u_end);
    else
        consumer_warp<D, G, WPH, NB>(a, smem, sh, u_begin, u_end);
}

// ---------------------------------------------------------------------------
// Small steps in one launch: a thread-block cluster per (request, head group)
// ---------------------------------------------------------------------------
// A plan whose capacity is small (a few requests of short contexts, the
// latency-bound single-request decode) runs each step as one launch with no work
// list: cluster c serves (request c / groups, head group c % groups), and its CTA of
// rank r takes the r-th of cs stage-aligned shares of the request's slot list, read
// from kv_indptr on the device. Every CTA ends with a partial result in its own
// shared memory; after a cluster barrier the consumer warps of the cluster merge
// the query heads' parts by the log-sum-exp identity, reading the peers' results
// through distributed shared memory (ld.shared::cluster), and write out and lse. A
// second cluster barrier keeps every CTA's shared memory alive until its peers have
// read it. Every thread reaches both barriers, also after a bounded wait ran out.

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
template <int D, int G, int WPH, int CS>
__global__ void __launch_bounds__(SmallCfg<D, G, WPH>::C::kThreads, 2)
    paged_decode_small_kernel(const DecodeArgs a) {
    using C = typename SmallCfg<D, G, WPH>::C;
    extern __shared__ __align__(128) uint8_t smem[];
    Shared sh;
    sh.full = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    sh.empty = sh.full + C::kStages;
    sh.flags = reinterpret_cast<volatile int*>(sh.full + 2 * C::kStages);
    using SC = SmallCfg<D, G, WPH>;
    Unit* unit = reinterpret_cast<Unit*>(smem + SC::kUnitOffset);
    sh.units = unit;
    sh.part_offset = SC::kPartOffset;
    constexpr int cs = CS;  // CTAs of a cluster: the ways each request is split
    const uint32_t rank = cluster_rank();
    const int item = blockIdx.x / cs;
    const int n_groups = a.n_kv_heads / C::kHeadsPerCta;
    const bool has_item = item < a.batch * n_groups;  // the same for the whole cluster
    pdl_launch_dependents();
    if (threadIdx.x == 0) {
        const uint32_t full_arrivals = C::kProducerWarps * (a.k_host != nullptr ? 33 : 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), full_arrivals);
            mbar_init(smem_u32(&sh.empty[s]), C::kConsumerWarps);
        }
        sh.flags[0] = 0;
        if (has_item) {
            // with early gather kv_indptr was final before the step's plan call
            if (!a.early) pdl_wait();
            const int b = item / n_groups;
            const int ip0 = a.kv_indptr[b], ip1 = a.kv_indptr[b + 1];
            const int L = ip1 - ip0;
            const int st = C::kStageTokens;
            const int share = ((L + cs - 1) / cs + st - 1) / st * st;
            const int t0 = min(int(rank) * share, L), t1 = min(t0 + share, L);
            *unit = Unit{b, item % n_groups, t0, t1, int(rank), 1, ip0 + t0, L};
        }
        fence_mbar_init();
    }
    __syncthreads();
    const int n_units = has_item ? 1 : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= C::kConsumerWarps)
        producer_warp<D, G, WPH, 1>(a, smem, sh, 0, n_units);
    else
        consumer_warp<D, G, WPH, 1, true>(a, smem, sh, 0, n_units);
    __syncwarp();
    cluster_sync_all();  // every CTA's partial result is in its shared memory
    if (has_item && warp < C::kConsumerWarps) {
        // CTA r merges query heads r, r + cs, ...; its consumer warps split head_dim,
        // kDL dims per lane
        constexpr int kDL = D / (32 * C::kConsumerWarps);
        const Unit un = *unit;
        const uint32_t part_base = smem_u32(smem + SC::kPartOffset);
        const int dim0 = warp * 32 * kDL + lane * kDL;
        for (int qh = int(rank); qh < C::kQHeads; qh += cs) {
            // lane p < cs holds part p's base-2 lse (the other lanes read part 0's and drop it)
            const float lv = dsmem_ld_f32(dsmem_addr(part_base + (C::kQHeads * D + qh) * 4,
                                                     lane < cs ? lane : 0));
            const float lp = lane < cs ? lv : neg_inf();
            float x[cs][kDL];
#pragma unroll
            for (int p = 0; p < cs; ++p)
#pragma unroll
                for (int i = 0; i < kDL; ++i)
                    x[p][i] = dsmem_ld_f32(dsmem_addr(part_base + (qh * D + dim0 + i) * 4, p));
            float mx = lp;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
            const float e = lp == neg_inf() ? 0.f : ex2(lp - mx);
            float sm = e;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sm += __shfl_xor_sync(kFull, sm, off);
            float acc[kDL];
#pragma unroll
            for (int i = 0; i < kDL; ++i) acc[i] = 0.f;
#pragma unroll
            for (int p = 0; p < cs; ++p) {
                const float w = __shfl_sync(kFull, e, p);
#pragma unroll
                for (int i = 0; i < kDL; ++i) acc[i] = fmaf(w, x[p][i], acc[i]);
            }
            const float inv = sm > 0.f ? 1.f / sm : 0.f;
            const int h = (un.hg * C::kHeadsPerCta) * G + qh;  // query head index
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) +
                                 (int64_t(un.b) * a.n_qo_heads + h) * D + dim0;
            if constexpr (kDL == 1) {
                dst[0] = __float2bfloat16_rn(acc[0] * inv);
            } else {
#pragma unroll
                for (int i = 0; i < kDL; i += 2)
                    *reinterpret_cast<uint32_t*>(dst + i) = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
            }
            if (a.lse != nullptr && warp == 0 && lane == 0)
                a.lse[int64_t(un.b) * a.n_qo_heads + h] = sm > 0.f ? (mx + __log2f(sm)) * kLn2 : neg_inf();
        }
    }
    __syncwarp();
    cluster_sync_all();  // no CTA leaves while a peer may still read its shared memory
}

// ---------------------------------------------------------------------------
// LSE merge of split contexts
// ---------------------------------------------------------------------------
// One warp per (merge record, query head of the group): lanes first take parts
// c = lane, lane + 32, ... to form the merged log-sum-exp (online max/sum, then a
// warp reduction), then every lane owns head_dim/32 consecutive dimensions and
// sums w_c * out_c over all parts, with w_c = 2^(lse_c - lse) broadcast from the
// lane that read part c; the parts' loads of a chunk of 16 (8 at head_dim 256)
// are all issued before any is used. Launched right after the decode kernel on a
// fixed grid (warps loop over the work), so the launch does not depend on the step.
constexpr int kMergeThreads = 128;

// Issue the loads of parts c0 .. c0 + kChunk - 1 of one merged context's query
// head: lane l receives dims l * D / 32 .. of every part (zeros past the count).
template <int D, int kChunk>
__device__ __forceinline__ void merge_load_chunk(const DecodeArgs& a, const int32_t* parts,
                                                 int count, int c0, int slot_l, int qheads,
                                                 int qh, int lane,
                                                 float4 (&x)[kChunk][D / 128]) {
    constexpr int kVD = D / 32;
    const int c = c0 + (lane % kChunk);
    const int from_lane = __shfl_sync(kFull, slot_l, c & 31);  // every lane shuffles
    const int slot_c = c < count ? (c < 32 ? from_lane : __ldg(parts + c)) : 0;
#pragma unroll
    for (int j = 0; j < kChunk; ++j) {
        const int slot = __shfl_sync(kFull, slot_c, j);
        const float* src = a.ws_o + (int64_t(slot) * qheads + qh) * D + lane * kVD;
#pragma unroll
        for (int i = 0; i < kVD / 4; ++i)
            x[j][i] = c0 + j < count ? __ldcg(reinterpret_cast<const float4*>(src) + i)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads, 2) lse_merge_kernel(const DecodeArgs a) {
    pdl_launch_dependents();
    constexpr int kVD = D / 32;  // dims per lane
    const int lane = threadIdx.x & 31;
    const int n_merges = a.meta_header[0];
    const int qheads = a.heads_per_cta * (a.n_qo_heads / a.n_kv_heads);
    const int G = a.n_qo_heads / a.n_kv_heads;
    const int items = n_merges * qheads;
    const int warps = gridDim.x * (kMergeThreads / 32);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    // The merge record and the slots of its first 32 parts are plan data: read them
    // before waiting for the decode kernel, so only the partial results are loaded
    // after it.
    int w = blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);
    Merge mg{};
    int slot_l = 0;  // slot of part `lane` (parts < 32)
    if (w < items) {
        mg = a.merges[w / qheads];
        if (lane < mg.count) slot_l = __ldg(a.part_list + mg.first + lane);
    }
    pdl_wait();  // the partial results come from the decode kernel
    // Parts in chunks of kChunk: every load of a chunk is issued before the first
    // use, so a chunk costs one round trip to L2; the first chunk's outputs are
    // issued together with the log-sum-exp pass, which does not need them.
    constexpr int kChunk = kVD == 4 ? 32 : 16;
    for (; w < items; w += warps) {
        const int qh = w % qheads;
        const int32_t* parts = a.part_list + mg.first;
        float4 x[kChunk][kVD / 4];
        merge_load_chunk<D, kChunk>(a, parts, mg.count, 0, slot_l, qheads, qh, lane, x);
        float mx = neg_inf(), sm = 0.f, lse_l = neg_inf();  // lse_l: part `lane`'s lse
        for (int c = lane; c < mg.count; c += 32) {
            const int slot = c < 32 ? slot_l : __ldg(parts + c);
            const float xl = __ldcg(a.ws_lse + int64_t(slot) * qheads + qh);
            if (c < 32) lse_l = xl;
            const float mn = fmaxf(mx, xl);
            sm = (mx == neg_inf() ? 0.f : sm * ex2(mx - mn)) + ex2(xl - mn);
            mx = mn;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float mo = __shfl_xor_sync(kFull, mx, off);
            const float so = __shfl_xor_sync(kFull, sm, off);
            const float mn = fmaxf(mx, mo);
            sm = (mx == neg_inf() ? 0.f : sm * ex2(mx - mn)) + (mo == neg_inf() ? 0.f : so * ex2(mo - mn));
            mx = mn;
        }
        const float total = mx + __log2f(sm);
        float acc[kVD];
#pragma unroll
        for (int i = 0; i < kVD; ++i) acc[i] = 0.f;
        for (int c0 = 0; c0 < mg.count; c0 += kChunk) {
            if (c0 > 0) merge_load_chunk<D, kChunk>(a, parts, mg.count, c0, slot_l, qheads, qh, lane, x);
            // weight of part c0 + lane % kChunk (lse from the pass above for parts < 32)
            const int c = c0 + (lane % kChunk);
            const float from_lane = __shfl_sync(kFull, lse_l, c & 31);
            float wl = 0.f;
            if (c < mg.count)
                wl = ex2((c < 32 ? from_lane
                                 : __ldcg(a.ws_lse + int64_t(__ldg(parts + c)) * qheads + qh)) -
                         total);
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
                const float wj = __shfl_sync(kFull, wl, j);
#pragma unroll
                for (int i = 0; i < kVD / 4; ++i) {
                    acc[4 * i] = fmaf(wj, x[j][i].x, acc[4 * i]);
                    acc[4 * i + 1] = fmaf(wj, x[j][i].y, acc[4 * i + 1]);
                    acc[4 * i + 2] = fmaf(wj, x[j][i].z, acc[4 * i + 2]);
                    acc[4 * i + 3] = fmaf(wj, x[j][i].w, acc[4 * i + 3]);
                }
            }
        }
        const int h = (mg.hg * a.heads_per_cta) * G + qh;  // query head index
        __nv_bfloat16* dst = out + (int64_t(mg.b) * a.n_qo_heads + h) * D + lane * kVD;
#pragma unroll
        for (int i = 0; i < kVD; i += 4) {
            uint2 packed;
            packed.x = pack_bf16x2(acc[i], acc[i + 1]);
            packed.y = pack_bf16x2(acc[i + 2], acc[i + 3]);
            *reinterpret_cast<uint2*>(dst + i) = packed;
        }
        if (a.lse != nullptr && lane == 0) a.lse[int64_t(mg.b) * a.n_qo_heads + h] = total * kLn2;
        // next item of this warp
        if (w + warps < items) {
            mg = a.merges[(w + warps) / qheads];
            slot_l = lane < mg.count ? __ldg(a.part_list + mg.first + lane) : 0;
        }
    }
}

template <int D>
cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.merge_ctas);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, lse_merge_kernel<D>, a);
}

template <int D, int G, int WPH, int NB>
cudaError_t prepare() {
    // Raise the dynamic shared memory limit once per instance.
    static cudaError_t status = cudaFuncSetAttribute(
        paged_decode_kernel<D, G, WPH, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        Cfg<D, G, WPH, NB>::kSmem);
    return status;
}

template <int D, int G, int WPH, int NB>
int occupancy() {
    using C = Cfg<D, G, WPH, NB>;
    if (prepare<D, G, WPH, NB>() != cudaSuccess) return 0;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, paged_decode_kernel<D, G, WPH, NB>,
                                                      C::kThreads, C::kSmem) != cudaSuccess)
        return 0;
    return blocks;
}

template <int D, int G, int WPH, int NB>
cudaError_t launch(const DecodeArgs& a, cudaStream_t stream) {
    using C = Cfg<D, G, WPH, NB>;
    cudaError_t e = prepare<D, G, WPH, NB>();
    if (e != cudaSuccess) return e;
    if (a.n_ctas == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_ctas);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, G, WPH, NB>, a);
}

template <int D, int G, int WPH, int CS>
cudaError_t prepare_small() {
    static cudaError_t status = [] {
        auto k = paged_decode_small_kernel<D, G, WPH, CS>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SmallCfg<D, G, WPH>::kSmem);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return e;
    }();
    return status;
}

template <int D, int G, int WPH, int CS>
cudaLaunchConfig_t small_config(int grid, cudaStream_t stream, cudaLaunchAttribute (&attr)[2]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(SmallCfg<D, G, WPH>::C::kThreads);
    cfg.dynamicSmemBytes = SmallCfg<D, G, WPH>::kSmem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cfg;
}

// Clusters of the single-launch kernel that fit on the device at once (0: the kernel
// cannot run, e.g. no 16-CTA clusters).
template <int D, int G, int WPH, int CS>
int small_clusters() {
    if (prepare_small<D, G, WPH, CS>() != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = small_config<D, G, WPH, CS>(CS, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, paged_decode_small_kernel<D, G, WPH, CS>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int D, int G, int WPH, int CS>
cudaError_t launch_small(const DecodeArgs& a, cudaStream_t stream) {
    cudaError_t e = prepare_small<D, G, WPH, CS>();
    if (e != cudaSuccess) return e;
    if (a.n_ctas == 0) return cudaSuccess;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = small_config<D, G, WPH, CS>(a.n_ctas, stream, attr);
    return cudaLaunchKernelEx(&cfg, paged_decode_small_kernel<D, G, WPH, CS>, a);
}

// Calls FN<D, G, WPH, NB>::run(args...) for the runtime shape. `shared` selects
// the shared-prefix instance (two query blocks per warp), which exists only at
// head_dim 128 with one warp per KV head.
template <template <int, int, int, int> class FN, typename... Args>
auto dispatch(int head_dim, int group, int wph, bool shared, Args&&... args)
    -> decltype(FN<128, 1, 1, 1>::run(args...)) {
#define PKV_G(D_, W_, NB_)                                     \
    switch (group) {                                           \
        case 1: return FN<D_, 1, W_, NB_>::run(args...);       \
        case 2: return FN<D_, 2, W_, NB_>::run(args...);       \
        case 4: return FN<D_, 4, W_, NB_>::run(args...);       \
        case 8: return FN<D_, 8, W_, NB_>::run(args...);       \
        default: break;                                        \
    }
    if (!shared) {
        if (head_dim == 128) {
            if (wph == 1) { PKV_G(128, 1, 1) }
            if (wph == 2) { PKV_G(128, 2, 1) }
            if (wph == 4) { PKV_G(128, 4, 1) }
        } else if (head_dim == 256) {
            if (wph == 2) { PKV_G(256, 2, 1) }
            if (wph == 4) { PKV_G(256, 4, 1) }
        }
    } else if (head_dim == 128 && wph == 1) {
        PKV_G(128, 1, 2)
    }
#undef PKV_G
    return FN<128, 1, 1, 1>::unsupported();
}

template <int D, int G, int WPH, int NB>
struct OccupancyFn {
    static int run() { return occupancy<D, G, WPH, NB>(); }
    static int unsupported() { return 0; }
};
template <int D, int G, int WPH, int NB>
struct LaunchFn {
    static cudaError_t run(const DecodeArgs& a, cudaStream_t s) {
        return launch<D, G, WPH, NB>(a, s);
    }
    static cudaError_t unsupported() { return cudaErrorInvalidValue; }
};
template <int D, int G, int WPH, int NB>
struct SmallClustersFn {
    static int run(int cs) {
        if constexpr (NB != 1) {
            return 0;
        } else {
            switch (cs) {
                case 16: return small_clusters<D, G, WPH, 16>();
                case 8: return small_clusters<D, G, WPH, 8>();
                case 4: return small_clusters<D, G, WPH, 4>();
                default: return 0;
            }
        }
    }
    static int unsupported() { return 0; }
};
template <int D, int G, int WPH, int NB>
struct SmallLaunchFn {
    static cudaError_t run(const DecodeArgs& a, cudaStream_t s) {
        switch (a.small) {
            case 16: return launch_small<D, G, WPH, 16>(a, s);
            case 8: return launch_small<D, G, WPH, 8>(a, s);
            case 4: return launch_small<D, G, WPH, 4>(a, s);
            default: return cudaErrorInvalidValue;
        }
    }
    static cudaError_t unsupported() { return cudaErrorInvalidValue; }
};
template <int D, int G, int WPH, int NB>
struct RowsFn {
    static int run() { return Cfg<D, G, WPH, NB>::kWarpRows; }
    static int unsupported() { return 0; }
};

int warps_per_head(int heads_per_cta) { return kGroupWarps / heads_per_cta; }

}  // namespace

bool decode_shape_supported(int n_qo_heads, int n_kv_heads, int head_dim) {
    if (n_kv_heads <= 0 || n_qo_heads <= 0 || n_qo_heads % n_kv_heads != 0) return false;
    const int G = n_qo_heads / n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return false;
    if (head_dim != 128 && head_dim != 256) return false;
    return n_kv_heads == 1 || n_kv_heads == 2 || n_kv_heads == 4 || n_kv_heads == 8;
}

int decode_shared_rows(int n_qo_heads, int n_kv_heads, int head_dim, int heads_per_cta) {
    if (!decode_shape_supported(n_qo_heads, n_kv_heads, head_dim) || heads_per_cta < 1 ||
        kGroupWarps % heads_per_cta != 0)
        return 0;
    return dispatch<RowsFn>(head_dim, n_qo_heads / n_kv_heads, warps_per_head(heads_per_cta), true);
}

int decode_ctas_per_sm(int n_qo_heads, int n_kv_heads, int head_dim, int heads_per_cta,
                       bool shared) {
    if (!decode_shape_supported(n_qo_heads, n_kv_heads, head_dim)) return 0;
    if (heads_per_cta < 1 || heads_per_cta > heads_per_group(n_kv_heads, head_dim) ||
        n_kv_heads % heads_per_cta != 0)
        return 0;
    return dispatch<OccupancyFn>(head_dim, n_qo_heads / n_kv_heads, warps_per_head(heads_per_cta),
                                 shared);
}

int decode_small_clusters(int n_qo_heads, int n_kv_heads, int head_dim, int cluster_size) {
    if (!decode_shape_supported(n_qo_heads, n_kv_heads, head_dim)) return 0;
    const int hpc = heads_per_group(n_kv_heads, head_dim);
    return dispatch<SmallClustersFn>(head_dim, n_qo_heads / n_kv_heads, warps_per_head(hpc), false,
                                     cluster_size);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    if (a.small)
        return dispatch<SmallLaunchFn>(a.head_dim, a.n_qo_heads / a.n_kv_heads,
                                       warps_per_head(a.heads_per_cta), false, a, stream);
    cudaError_t e = dispatch<LaunchFn>(a.head_dim, a.n_qo_heads / a.n_kv_heads,
                                       warps_per_head(a.heads_per_cta), a.shared, a, stream);
    if (e != cudaSuccess) return e;
    return a.head_dim == 128 ? launch_merge<128>(a, stream) : launch_merge<256>(a, stream);
}

}  // namespace pkv
