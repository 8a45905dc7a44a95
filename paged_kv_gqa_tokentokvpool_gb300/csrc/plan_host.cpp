// Per-step work partitioner for split-KV decode (host only, no CUDA calls).
//
// The plan is built once per decode step and reused by every layer ("Agent-Infer:
// 纯 Rust 编写的高性能 LLM 推理引擎", section "分页 KV 缓存"; section "优化历程",
// stage 3). Its job on this hardware: a decode batch mixes short and very long
// contexts, and the attention kernel runs a fixed grid of persistent CTAs
// (resident CTAs per SM x SMs). The work of a layer is the set of
// (request, KV-head group) pairs, each a run of L_b tokens; head groups are
// independent, so cutting along heads costs nothing, while cutting a context
// into token chunks costs one fp32 partial result per extra chunk plus a
// log-sum-exp merge. The planner:
//   1. picks a chunk length c (a multiple of kChunkQuantum) by estimating, for a
//      handful of candidates, the makespan of a longest-first assignment of the
//      resulting units to the CTAs (average load plus half the largest unit),
//      charging each unit a fixed cost and each split unit the traffic of its
//      partial;
//   2. cuts every (request, head group) longer than c into near-equal parts;
//   3. assigns units to CTAs longest first, each to the least-loaded CTA
//      (longest-processing-time-first list scheduling), and lists every CTA's
//      units contiguously.
#include <algorithm>
#include <cstdint>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "pkv_internal.h"

namespace pkv {

namespace {

// Cost model, in "token rows" (one token of one head group = 2 * row bytes).
constexpr int64_t kUnitOverheadTokens = 16;   // q load, pipeline hand-over, epilogue
constexpr int64_t kPartialOverheadTokens = 8; // fp32 partial written + read back

int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }

struct Work {
    int32_t b;
    int32_t len;
};

int64_t units_for_chunk(const std::vector<Work>& work, int64_t chunk) {
    int64_t n = 0;
    for (const Work& w : work) n += (w.len <= chunk) ? 1 : (w.len + chunk - 1) / chunk;
    return n;
}

int64_t unit_cost(int64_t len, bool split) {
    return len + kUnitOverheadTokens + (split ? kPartialOverheadTokens : 0);
}

// Estimated makespan of longest-first list scheduling of the units chunk c
// creates, without running it: the average load per CTA plus half the largest
// unit (the last unit placed on the busiest CTA), and never below the largest.
int64_t estimate_makespan(const std::vector<Work>& work, int64_t chunk, int ctas) {
    int64_t sum = 0, biggest = 0;
    for (const Work& w : work) {
        if (w.len <= chunk) {
            const int64_t c = unit_cost(w.len, false);
            sum += c;
            biggest = std::max(biggest, c);
            continue;
        }
        const int64_t parts = (w.len + chunk - 1) / chunk;
        sum += w.len + parts * (kUnitOverheadTokens + kPartialOverheadTokens);
        biggest = std::max(biggest, unit_cost((w.len + parts - 1) / parts, true));
    }
    return std::max(biggest, (sum + ctas - 1) / ctas + biggest / 2);
}

}  // namespace

int plan_max_units(int ctas, int max_batch, int n_groups) {
    return kMaxUnitsPerCta * ctas + max_batch * n_groups;
}

int plan_compute(const int32_t* indptr, int batch, int n_groups, int ctas, const PlanLimits& lim,
                 Unit* units, int* cta_begin, Merge* merges, PlanCounts* out) {
    if (batch < 0) return fail(PKV_ERR_INVALID_ARG, "plan: batch %d < 0", batch);
    if (n_groups < 1 || ctas < 1) return fail(PKV_ERR_INVALID_ARG, "plan: bad head groups / CTAs");
    if (batch > 0 && indptr == nullptr) return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr is NULL");
    if (batch > 0 && indptr[0] != 0)
        return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr[0] = %d, expected 0", indptr[0]);
    std::vector<Work> work;
    work.reserve(size_t(batch) * n_groups);
    int64_t total = 0;
    int32_t lmax = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t L = int64_t(indptr[b + 1]) - indptr[b];
        if (L < 0) return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr decreases at %d", b);
        lmax = std::max<int32_t>(lmax, static_cast<int32_t>(L));
        for (int g = 0; g < n_groups; ++g) work.push_back(Work{b, static_cast<int32_t>(L)});
        total += L * n_groups;
    }

    // Candidate chunks: from about total / (kMaxUnitsPerCta * ctas) up to the
    // longest context, growing by ~1.25x; the largest means "never split".
    int64_t chunk = std::max<int64_t>(lmax, 1);
    if (lmax > kMinChunkTokens) {
        const int64_t lo = std::max<int64_t>(
            kMinChunkTokens,
            round_up((total + int64_t(kMaxUnitsPerCta) * ctas - 1) / (int64_t(kMaxUnitsPerCta) * ctas),
                     kChunkQuantum));
        std::vector<int64_t> cands;
        for (int64_t c = round_up(lo, kChunkQuantum); c < lmax;
             c = round_up(c + std::max<int64_t>(kChunkQuantum, c / 4), kChunkQuantum))
            cands.push_back(c);
        cands.push_back(lmax);
        int64_t best = -1;
        for (int64_t c : cands) {
            if (units_for_chunk(work, c) > lim.max_units) continue;
            const int64_t ms = estimate_makespan(work, c, ctas);
            // prefer the larger chunk (fewer partials) unless a smaller one is
            // at least 1% faster
            if (best < 0 || ms * 100 < best * 99) {
                best = ms;
                chunk = c;
            }
        }
    }

    // Cut the work into units.
    std::vector<Unit> all;
    all.reserve(size_t(units_for_chunk(work, chunk)));
    int n_merges = 0, next_partial = 0;
    for (size_t i = 0; i < work.size(); ++i) {
        const Work& w = work[i];
        const int32_t g = static_cast<int32_t>(i % n_groups);
        if (w.len <= chunk) {
            all.push_back(Unit{w.b, g, 0, w.len, -1, -1, 0, 0});
            continue;
        }
        const int32_t parts = static_cast<int32_t>((w.len + chunk - 1) / chunk);
        if (n_merges >= lim.max_merges)
            return fail(PKV_ERR_PLAN, "plan: more split contexts than capacity %d", lim.max_merges);
        merges[n_merges] = Merge{w.b, g, next_partial, parts};
        const int32_t base = w.len / parts, rem = w.len % parts;
        int32_t start = 0;
        for (int32_t p = 0; p < parts; ++p) {
            const int32_t len = base + (p < rem ? 1 : 0);
            all.push_back(Unit{w.b, g, start, start + len, next_partial++, n_merges, 0, 0});
            start += len;
        }
        ++n_merges;
    }
    const int n_units = static_cast<int>(all.size());
    if (n_units > lim.max_units)
        return fail(PKV_ERR_PLAN, "plan: %d work units exceed the plan's capacity %d", n_units,
                    lim.max_units);

    // Longest-first list scheduling onto min(ctas, units) CTAs.
    const int used = std::max(1, std::min(ctas, n_units));
    std::vector<int> order(n_units);
    for (int i = 0; i < n_units; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
        return (all[x].tok_end - all[x].tok_begin) > (all[y].tok_end - all[y].tok_begin);
    });
    using Slot = std::pair<int64_t, int>;  // (load, cta)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int c = 0; c < used; ++c) heap.push(Slot{0, c});
    std::vector<std::vector<int>> lists(used);
    for (int i : order) {
        Slot s = heap.top();
        heap.pop();
        const Unit& u = all[i];
        s.first += unit_cost(u.tok_end - u.tok_begin, u.partial >= 0);
        lists[s.second].push_back(i);
        heap.push(s);
    }
    int pos = 0, n_ctas = 0;
    for (int c = 0; c < used; ++c) {
        if (lists[c].empty()) continue;
        cta_begin[n_ctas++] = pos;
        for (int i : lists[c]) units[pos++] = all[i];
    }
    cta_begin[n_ctas] = pos;
    out->n_units = n_units;
    out->n_ctas = n_ctas;
    out->n_merges = n_merges;
    out->n_partials = next_partial;
    out->chunk_tokens = static_cast<int>(chunk);
    return PKV_OK;
}

}  // namespace pkv
