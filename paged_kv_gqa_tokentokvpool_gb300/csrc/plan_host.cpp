// Per-step work partitioner for split-KV decode (host only, no CUDA calls).
//
// The plan is built once per decode step and reused by every layer ("Agent-Infer:
// 纯 Rust 编写的高性能 LLM 推理引擎", section "分页 KV 缓存"; section "优化历程",
// stage 3). Its job on this hardware: a decode batch mixes short and very long
// contexts, and the attention kernel runs a fixed grid of persistent CTAs
// (resident CTAs per SM x SMs). The work of a layer is the list of items
// (request b, KV-head group hg), each a run of L_b tokens; head groups are
// independent, so cutting along heads costs nothing, while cutting a context into
// token ranges costs one fp32 partial result per extra range plus a log-sum-exp
// merge. The planner therefore:
//   1. lays the items end to end (request-major) and cuts that sequence into
//      `ctas` ranges of equal token count (fewer if a range would drop below
//      kMinChunkTokens), so every CTA streams the same number of bytes whatever
//      the mix of lengths, and an item is only split where a range boundary
//      falls inside it (at most ctas - 1 splits in total);
//   2. moves each boundary to the nearest item edge when it falls within
//      min(kSnapTokens, range / 8) tokens of it, so no split creates a sliver of
//      a unit while the ranges stay within 25% of equal;
//   3. lists each CTA's pieces of split items before its whole items, so the
//      parts of a split context finish early and the CTA that completes a
//      context's last part merges it while the other CTAs are still streaming.
// Empty contexts (L_b = 0) become zero-token units that only write out = 0 and
// lse = -inf; they are dealt round-robin at the end of the CTA lists.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "pkv_internal.h"

namespace pkv {

namespace {

// A range boundary closer than this to an item edge moves onto the edge (the
// distance is also capped at an eighth of the range).
constexpr int64_t kSnapTokens = 32;

}  // namespace

int plan_max_units(int ctas, int max_batch, int n_groups) {
    // each CTA holds at most two split pieces besides whole items
    return 2 * ctas + max_batch * n_groups;
}

int plan_compute(const int32_t* indptr, int batch, int n_groups, int ctas, const PlanLimits& lim,
                 Unit* units, int* cta_begin, Merge* merges, PlanCounts* out) {
    if (batch < 0) return fail(PKV_ERR_INVALID_ARG, "plan: batch %d < 0", batch);
    if (n_groups < 1 || ctas < 1) return fail(PKV_ERR_INVALID_ARG, "plan: bad head groups / CTAs");
    if (batch > 0 && indptr == nullptr) return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr is NULL");
    if (batch > 0 && indptr[0] != 0)
        return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr[0] = %d, expected 0", indptr[0]);
    const int n_items = batch * n_groups;
    std::vector<int64_t> start(n_items + 1, 0);  // item k covers [start[k], start[k+1])
    for (int b = 0; b < batch; ++b) {
        const int64_t L = int64_t(indptr[b + 1]) - indptr[b];
        if (L < 0) return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr decreases at %d", b);
        for (int g = 0; g < n_groups; ++g) {
            const int k = b * n_groups + g;
            start[k + 1] = start[k] + L;
        }
    }
    const int64_t total = start[n_items];

    // 1-2. range boundaries, snapped and quantised inside items; a small step uses
    // fewer CTAs so that no range is shorter than kMinChunkTokens
    const int used = static_cast<int>(
        std::max<int64_t>(1, std::min<int64_t>(ctas, total / kMinChunkTokens)));
    std::vector<int64_t> cut(used + 1);
    cut[0] = 0;
    cut[used] = total;
    const int64_t snap = std::min<int64_t>(kSnapTokens, total / used / 8);
    int k = 0;
    for (int c = 1; c < used; ++c) {
        int64_t p = total * c / used;
        while (k < n_items && start[k + 1] <= p) ++k;  // item k: start[k] <= p < start[k+1]
        if (k < n_items && p > start[k]) {
            if (p - start[k] < snap) p = start[k];
            else if (start[k + 1] - p < snap) p = start[k + 1];
        }
        cut[c] = std::max(cut[c - 1], std::min(p, total));
    }

    // pieces: walk every range over the items it touches
    std::vector<int> parts(n_items, 0);
    struct Piece {
        int cta, item;
        int64_t t0, t1;  // token offsets within the item
    };
    std::vector<Piece> pieces;
    pieces.reserve(size_t(n_items) + 2 * used);
    int item = 0;
    for (int c = 0; c < used; ++c) {
        const int64_t a = cut[c], b = cut[c + 1];
        if (a == b) continue;
        while (item < n_items && start[item + 1] <= a) ++item;
        for (int i = item; i < n_items && start[i] < b; ++i) {
            const int64_t t0 = std::max(a, start[i]) - start[i];
            const int64_t t1 = std::min(b, start[i + 1]) - start[i];
            if (t1 <= t0) continue;
            pieces.push_back(Piece{c, i, t0, t1});
            ++parts[i];
        }
    }
    // empty items still need a unit each
    int rr = 0;
    for (int i = 0; i < n_items; ++i)
        if (start[i + 1] == start[i]) {
            pieces.push_back(Piece{rr, i, 0, 0});
            parts[i] = 1;
            rr = (rr + 1) % used;
        }
    const int n_units = static_cast<int>(pieces.size());
    if (n_units > lim.max_units)
        return fail(PKV_ERR_PLAN, "plan: %d work units exceed the plan's capacity %d", n_units,
                    lim.max_units);

    // merge records and partial slots, in item order
    std::vector<int> merge_of(n_items, -1), next_slot(n_items, 0);
    int n_merges = 0, n_partials = 0;
    for (int i = 0; i < n_items; ++i) {
        if (parts[i] < 2) continue;
        if (n_merges >= lim.max_merges)
            return fail(PKV_ERR_PLAN, "plan: more split contexts than capacity %d", lim.max_merges);
        merges[n_merges] = Merge{i / n_groups, i % n_groups, n_partials, parts[i]};
        merge_of[i] = n_merges++;
        next_slot[i] = n_partials;
        n_partials += parts[i];
    }
    std::vector<Unit> all(n_units);
    for (int u = 0; u < n_units; ++u) {
        const Piece& pc = pieces[u];  // pieces of an item appear in token order
        const int m = merge_of[pc.item];
        const int b = pc.item / n_groups;
        all[u] = Unit{b, pc.item % n_groups, static_cast<int32_t>(pc.t0),
                      static_cast<int32_t>(pc.t1), m >= 0 ? next_slot[pc.item]++ : -1, m,
                      static_cast<int32_t>(indptr[b] + pc.t0),
                      static_cast<int32_t>(start[pc.item + 1] - start[pc.item])};
    }

    // 3. per-CTA lists: split pieces first, then whole items
    std::vector<int> order(n_units);
    for (int u = 0; u < n_units; ++u) order[u] = u;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
        if (pieces[x].cta != pieces[y].cta) return pieces[x].cta < pieces[y].cta;
        return (all[x].partial >= 0) > (all[y].partial >= 0);
    });
    // Every CTA of the grid gets an entry: CTAs without work get empty ranges, so
    // the launch shape does not depend on the step.
    int pos = 0, o = 0;
    for (int c = 0; c < ctas; ++c) {
        cta_begin[c] = pos;
        while (o < n_units && pieces[order[o]].cta == c) units[pos++] = all[order[o++]];
    }
    cta_begin[ctas] = pos;
    out->n_units = n_units;
    out->n_ctas = used;
    out->n_merges = n_merges;
    out->n_partials = n_partials;
    out->chunk_tokens = static_cast<int>((total + used - 1) / used);
    return PKV_OK;
}

}  // namespace pkv
