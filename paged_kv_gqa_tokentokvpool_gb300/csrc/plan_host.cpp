// Per-step work partitioner for split-KV decode (host only, no CUDA calls).
//
// The plan is built once per decode step and reused by every layer ("Agent-Infer:
// 纯 Rust 编写的高性能 LLM 推理引擎", section "分页 KV 缓存"; section "优化历程",
// stage 3). Its job on this hardware: a decode batch mixes short and very long
// contexts, and the attention kernel runs a fixed grid of persistent CTAs
// (resident CTAs per SM x SMs). The work of a layer is a list of items, each a run
// of slots of one KV-head group hg to be attended by a set of requests:
//   * a plain item: all L_b slots of request b, for request b;
//   * with shared prefixes (the same first P slots listed by a run of consecutive
//     requests, as a prefix cache produces; "Agent-Infer", section "前缀缓存"): a
//     prefix item covers the P shared slots once for up to R requests of the group
//     (the query rows of R requests fill the kernel's tile), and a suffix item
//     covers the L_b - P private slots of each member.
// Head groups are independent, so cutting along heads costs nothing, while cutting
// a run into token ranges costs one fp32 partial result per extra range (per
// request of the item) plus a log-sum-exp merge. The planner therefore:
//   1. lays the items end to end and gives each CTA a contiguous range of that
//      sequence, costed in tokens as the kernel spends its time: whole pipeline
//      stages (a ragged last stage costs a full one) plus a fixed cost per unit.
//      A CTA takes whole items while they fit its budget, then as many whole stages
//      of the next item as fit, so only an item's last piece has a ragged stage and
//      no piece of a split item is shorter than kMinChunkTokens;
//   2. takes the smallest budget for which that greedy fill needs at most `ctas`
//      CTAs (a bisection over the budget), so the slowest CTA,
//      which sets the launch's duration, is as fast as the cost model allows. An
//      item is only split where a range boundary falls inside it;
//   3. gives every piece of a split item, and every piece of a prefix or suffix
//      item, a partial slot per request it serves, and every (request, head group)
//      with partial results a merge record whose part list names those slots in
//      token order;
//   4. lists each CTA's partial pieces before its whole items, so the parts of a
//      split context finish early.
// Empty contexts (L_b = 0) become zero-token units that only write out = 0 and
// lse = -inf; they are dealt round-robin at the end of the CTA lists.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "pkv_internal.h"

namespace pkv {

namespace {

struct Item {
    int32_t b;        // (first) request
    int32_t nreq;     // requests served
    int32_t hg;       // KV-head group
    int32_t tok0;     // first token within the request's slot list
    int32_t len;      // tokens
    int32_t req_len;  // context length of the request (-1 / -2 for a prefix item)
    int32_t idx0;     // kv_indptr[b] + tok0
    bool partial;     // its pieces always write partial results (prefix, suffix)
};


// Cost of a CTA streaming a piece of t tokens, in tokens: the kernel moves K/V in
// pipeline stages of stage_tokens tokens, and a ragged last stage takes a whole
// stage's turn; every unit also pays a fixed cost (its epilogue, the switch of
// query rows).
// stage_tokens is a power of two.
int64_t piece_cost(int64_t t, int64_t stage_tokens, int64_t unit_cost) {
    return ((t + stage_tokens - 1) & ~(stage_tokens - 1)) + unit_cost;
}

// Cuts the items, laid end to end, into CTA ranges of cost at most T: each CTA
// takes the sequence in order, whole items while they fit and then as many whole
// stages of the next item as fit, so that only an item's last piece has a ragged
// stage. No piece of a split item is shorter than kMinChunkTokens. Returns the
// number of CTAs used (writing cut[0 .. used] when cut is not NULL), or
// max_ctas + 1 once more than max_ctas would be needed or a piece cannot fit an
// empty CTA.
int greedy_fill(const std::vector<Item>& items, const std::vector<int64_t>& start, int64_t T,
                int64_t stage_tokens, int64_t unit_cost, int max_ctas, int64_t* cut) {
    const int64_t kMin = kMinChunkTokens;
    int n = 0;              // index of the CTA being filled
    int64_t budget = T;     // its budget left
    if (cut) cut[0] = 0;
    for (size_t k = 0; k < items.size(); ++k) {
        int64_t r = items[k].len;  // tokens of item k not yet placed
        while (r > 0) {
            const int64_t c = piece_cost(r, stage_tokens, unit_cost);
            if (c <= budget) {
                budget -= c;
                break;
            }
            // split: whole stages that fit, leaving at least kMin tokens behind
            int64_t p = budget > unit_cost ? (budget - unit_cost) & ~(stage_tokens - 1) : 0;
            if (r - p < kMin) p = r >= kMin ? (r - kMin) & ~(stage_tokens - 1) : 0;
            if (p >= kMin) {
                r -= p;
            } else if (budget == T) {
                return max_ctas + 1;  // not even a minimum piece fits an empty CTA
            } else {
                p = 0;
            }
            // the range ends here
            if (++n >= max_ctas) return max_ctas + 1;
            if (cut) cut[n] = start[k + 1] - r;
            budget = T;
        }
    }
    if (budget == T && n > 0) {
        // the last range is empty: the previous cut already ends the sequence
        if (cut) cut[n] = start[items.size()];
        return n;
    }
    if (cut) cut[n + 1] = start[items.size()];
    return n + 1;
}

}  // namespace

int plan_max_units(int ctas, int max_batch, int n_groups) {
    // at most two items per (request, head group) (a suffix and a share of a
    // prefix), plus one extra piece per range boundary
    return 2 * ctas + 2 * max_batch * n_groups;
}

int plan_compute(const int32_t* indptr, int batch, int n_groups, int ctas, int stage_tokens,
                 const PlanLimits& lim,
                 const PlanSharing* sharing, Unit* units, int* cta_begin, Merge* merges,
                 int32_t* part_list, PlanCounts* out) {
    if (batch < 0) return fail(PKV_ERR_INVALID_ARG, "plan: batch %d < 0", batch);
    if (n_groups < 1 || ctas < 1) return fail(PKV_ERR_INVALID_ARG, "plan: bad head groups / CTAs");
    if (batch > 0 && indptr == nullptr) return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr is NULL");
    if (batch > 0 && indptr[0] != 0)
        return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr[0] = %d, expected 0", indptr[0]);
    for (int b = 0; b < batch; ++b)
        if (indptr[b + 1] < indptr[b])
            return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr decreases at %d", b);
    const auto L = [&](int b) { return indptr[b + 1] - indptr[b]; };

    // items, in batch order; a sharing group contributes its prefix items, then
    // its members' suffix items
    std::vector<Item> items;
    items.reserve(size_t(2) * batch * n_groups);
    int s = 0;
    for (int b = 0; b < batch;) {
        while (sharing && s < sharing->n && sharing->indptr[s + 1] <= b) ++s;
        if (sharing && s < sharing->n && sharing->indptr[s] == b && sharing->len[s] > 0) {
            const int m1 = sharing->indptr[s + 1];
            const int32_t P = sharing->len[s];
            // -2 marks a prefix that other items of the group read again (the
            // kernel then asks L2 to keep its rows), -1 one read by this item only
            const int32_t tag = m1 - b > sharing->requests_per_unit ? -2 : -1;
            for (int c0 = b; c0 < m1; c0 += sharing->requests_per_unit) {
                const int nreq = std::min(sharing->requests_per_unit, m1 - c0);
                for (int g = 0; g < n_groups; ++g)
                    items.push_back(Item{c0, nreq, g, 0, P, tag, indptr[c0], true});
            }
            for (int m = b; m < m1; ++m)
                for (int g = 0; g < n_groups; ++g)
                    items.push_back(Item{m, 1, g, P, L(m) - P, L(m), indptr[m] + P, true});
            b = m1;
            ++s;
            continue;
        }
        for (int g = 0; g < n_groups; ++g)
            items.push_back(Item{b, 1, g, 0, L(b), L(b), indptr[b], false});
        ++b;
    }
    const int n_items = static_cast<int>(items.size());
    std::vector<int64_t> start(n_items + 1, 0);  // item k covers [start[k], start[k+1])
    for (int k = 0; k < n_items; ++k) start[k + 1] = start[k] + items[k].len;
    const int64_t total = start[n_items];

    // 1-2. range boundaries: the smallest budget whose greedy fill needs at most
    // `ctas` CTAs
    std::vector<int64_t> cut(size_t(ctas) + 1);
    const int64_t unit_cost = std::max<int64_t>(1, stage_tokens / 4);
    int64_t lb = 0;  // sum of the items' costs, unsplit
    for (int k = 0; k < n_items; ++k)
        if (items[k].len > 0) lb += piece_cost(items[k].len, stage_tokens, unit_cost);
    int used = 1;
    cut[0] = 0;
    cut[1] = total;
    if (total > 0) {
        // lo: infeasible, as `ctas` CTAs of a smaller budget than lb / ctas cannot
        // hold costs that add up to at least lb. hi: feasible; a minimum piece, two
        // stages and a unit above lb / ctas usually is, else the step doubles (all
        // items in one CTA, a budget of lb, always are)
        const int64_t base = (lb + ctas - 1) / ctas;
        int64_t lo = base - 1, step = kMinChunkTokens + 2 * stage_tokens + unit_cost;
        int64_t hi = std::min(lb, base + step);
        while (hi < lb && greedy_fill(items, start, hi, stage_tokens, unit_cost, ctas, nullptr) > ctas) {
            lo = hi;
            step *= 2;
            hi = std::min(lb, base + step);
        }
        while (hi - lo > 1) {
            const int64_t mid = lo + (hi - lo) / 2;
            if (greedy_fill(items, start, mid, stage_tokens, unit_cost, ctas, nullptr) <= ctas)
                hi = mid;
            else
                lo = mid;
        }
        used = greedy_fill(items, start, hi, stage_tokens, unit_cost, ctas, cut.data());
    }

    // pieces: walk every range over the items it touches
    struct Piece {
        int cta, item;
        int64_t t0, t1;  // token offsets within the item
        int slot;        // first partial slot, or -1 for a direct write
    };
    std::vector<Piece> pieces;
    pieces.reserve(size_t(n_items) + 2 * used);
    std::vector<int> n_pieces(n_items, 0);
    int item = 0;
    for (int c = 0; c < used; ++c) {
        const int64_t a = cut[c], b = cut[c + 1];
        if (a == b) continue;
        while (item < n_items && start[item + 1] <= a) ++item;
        for (int i = item; i < n_items && start[i] < b; ++i) {
            const int64_t t0 = std::max(a, start[i]) - start[i];
            const int64_t t1 = std::min(b, start[i + 1]) - start[i];
            if (t1 <= t0) continue;
            pieces.push_back(Piece{c, i, t0, t1, -1});
            ++n_pieces[i];
        }
    }
    // empty items (empty contexts) still need a unit each
    int rr = 0;
    for (int i = 0; i < n_items; ++i)
        if (items[i].len == 0) {
            pieces.push_back(Piece{rr, i, 0, 0, -1});
            n_pieces[i] = 1;
            rr = (rr + 1) % used;
        }
    const int n_units = static_cast<int>(pieces.size());
    if (n_units > lim.max_units)
        return fail(PKV_ERR_PLAN, "plan: %d work units exceed the plan's capacity %d", n_units,
                    lim.max_units);

    // 3. partial slots, in piece order (pieces of an item are in token order)
    int n_partials = 0;
    for (Piece& pc : pieces) {
        const Item& it = items[pc.item];
        if (it.partial || n_pieces[pc.item] > 1) {
            pc.slot = n_partials;
            n_partials += it.nreq;
        }
    }
    if (n_partials > lim.max_partials)
        return fail(PKV_ERR_PLAN, "plan: %d partial results exceed the plan's capacity %d",
                    n_partials, lim.max_partials);
    // Merge records: one per (request, head group) with partial results; its part
    // list gives that request's slot in every piece serving it. Items are emitted
    // prefix before suffix and pieces in token order, so every list is in token
    // order.
    std::vector<std::vector<int>> parts_of(size_t(batch) * n_groups);
    for (const Piece& pc : pieces) {
        if (pc.slot < 0) continue;
        const Item& it = items[pc.item];
        for (int r = 0; r < it.nreq; ++r)
            parts_of[size_t(it.b + r) * n_groups + it.hg].push_back(pc.slot + r);
    }
    int n_merges = 0, n_list = 0;
    for (int b = 0; b < batch; ++b)
        for (int g = 0; g < n_groups; ++g) {
            const std::vector<int>& pl = parts_of[size_t(b) * n_groups + g];
            if (pl.empty()) continue;
            if (n_merges >= lim.max_merges)
                return fail(PKV_ERR_PLAN, "plan: more merged contexts than capacity %d",
                            lim.max_merges);
            merges[n_merges++] = Merge{b, g, n_list, static_cast<int32_t>(pl.size())};
            for (int slot : pl) part_list[n_list++] = slot;
        }

    std::vector<Unit> all(n_units);
    for (int u = 0; u < n_units; ++u) {
        const Piece& pc = pieces[u];
        const Item& it = items[pc.item];
        all[u] = Unit{it.b,
                      it.hg,
                      static_cast<int32_t>(it.tok0 + pc.t0),
                      static_cast<int32_t>(it.tok0 + pc.t1),
                      pc.slot,
                      it.nreq,
                      static_cast<int32_t>(it.idx0 + pc.t0),
                      it.req_len};
    }

    // 4. per-CTA lists: partial pieces first, then whole items
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
