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
//   1. lays the items end to end and cuts that sequence into `ctas` ranges of equal
//      token count (fewer if a range would drop below kMinChunkTokens), so every
//      CTA streams the same number of bytes whatever the mix of lengths, and an
//      item is only split where a range boundary falls inside it;
//   2. moves each boundary to the nearest item edge when it falls within
//      min(kSnapTokens, range / 8) tokens of it, so no split creates a sliver of a
//      unit while the ranges stay within 25% of equal;
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

// A range boundary closer than this to an item edge moves onto the edge (the
// distance is also capped at an eighth of the range).
constexpr int64_t kSnapTokens = 32;

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

}  // namespace

int plan_max_units(int ctas, int max_batch, int n_groups) {
    // at most two items per (request, head group) (a suffix and a share of a
    // prefix), plus one extra piece per range boundary
    return 2 * ctas + 2 * max_batch * n_groups;
}

int plan_compute(const int32_t* indptr, int batch, int n_groups, int ctas, const PlanLimits& lim,
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

    // 1-2. range boundaries, snapped near item edges; a small step uses fewer CTAs
    // so that no range is shorter than kMinChunkTokens
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
