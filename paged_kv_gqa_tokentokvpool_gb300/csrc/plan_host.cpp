// Per-step work partitioner for split-KV decode (host only, no CUDA calls).
//
// The plan is built once per decode step and reused by every layer ("Agent-Infer:
// 纯 Rust 编写的高性能 LLM 推理引擎", section "分页 KV 缓存"; section "优化历程",
// stage 3). Its job on this hardware: a decode batch mixes short and very long
// contexts, and one CTA per request would leave most of the 152 SMs idle behind
// the longest one. So every context longer than a chunk is cut into near-equal
// parts, each part is one work unit, and the chunk length is the smallest one
// (a multiple of kChunkQuantum, at least kMinChunkTokens) for which the number of
// units stays within kWavesTarget waves of resident CTAs. Units are listed
// longest first, so the hardware block scheduler hands the long ones out first
// and the short ones fill the tail (longest-processing-time-first order).
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "pkv_internal.h"

namespace pkv {

int plan_target_units(const PlanShape& s) {
    const int sms = std::max(1, s.num_sms);
    const int per_sm = std::max(1, s.ctas_per_sm);
    return sms * per_sm * kWavesTarget;
}

namespace {

int64_t units_for_chunk(const std::vector<int32_t>& lengths, int64_t chunk) {
    int64_t n = 0;
    for (int32_t L : lengths) n += (L <= chunk) ? 1 : (L + chunk - 1) / chunk;
    return n;
}

int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }

}  // namespace

int plan_compute(const int32_t* indptr, int batch, const PlanShape& shape, Unit* units,
                 int max_units, Merge* merges, int max_merges, int* n_units_out,
                 int* n_merges_out, int* chunk_out) {
    if (batch < 0) return fail(PKV_ERR_INVALID_ARG, "plan: batch %d < 0", batch);
    if (batch > 0 && indptr == nullptr) return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr is NULL");
    if (batch > 0 && indptr[0] != 0)
        return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr[0] = %d, expected 0", indptr[0]);
    std::vector<int32_t> lengths(batch);
    int32_t lmax = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t L = int64_t(indptr[b + 1]) - indptr[b];
        if (L < 0) return fail(PKV_ERR_INVALID_ARG, "plan: kv_indptr decreases at %d", b);
        lengths[b] = static_cast<int32_t>(L);
        lmax = std::max(lmax, lengths[b]);
    }
    const int64_t cap = std::max<int64_t>(plan_target_units(shape), batch);

    // Smallest admissible chunk whose unit count fits in `cap`. The largest
    // candidate (round_up(lmax)) gives exactly `batch` units, which always fits.
    int64_t chunk;
    if (lmax <= kMinChunkTokens) {
        chunk = std::max<int64_t>(lmax, 1);
    } else {
        int64_t lo = round_up(kMinChunkTokens, kChunkQuantum) / kChunkQuantum;
        int64_t hi = round_up(lmax, kChunkQuantum) / kChunkQuantum;
        while (lo < hi) {
            const int64_t mid = (lo + hi) / 2;
            if (units_for_chunk(lengths, mid * kChunkQuantum) <= cap) hi = mid;
            else lo = mid + 1;
        }
        chunk = lo * kChunkQuantum;
    }

    const int64_t total = units_for_chunk(lengths, chunk);
    if (total > max_units)
        return fail(PKV_ERR_PLAN, "plan: %lld work units exceed the plan's capacity %d",
                    (long long)total, max_units);
    int nu = 0, nm = 0, next_partial = 0;
    for (int b = 0; b < batch; ++b) {
        const int32_t L = lengths[b];
        const int32_t parts = (L <= chunk) ? 1 : static_cast<int32_t>((L + chunk - 1) / chunk);
        if (parts == 1) {
            units[nu++] = Unit{b, 0, L, -1};
            continue;
        }
        if (nm >= max_merges)
            return fail(PKV_ERR_PLAN, "plan: more split requests than capacity %d", max_merges);
        merges[nm++] = Merge{b, next_partial, parts, 0};
        const int32_t base = L / parts, rem = L % parts;
        int32_t start = 0;
        for (int32_t p = 0; p < parts; ++p) {
            const int32_t len = base + (p < rem ? 1 : 0);
            units[nu++] = Unit{b, start, start + len, next_partial++};
            start += len;
        }
    }
    std::stable_sort(units, units + nu, [](const Unit& x, const Unit& y) {
        return (x.tok_end - x.tok_begin) > (y.tok_end - y.tok_begin);
    });
    *n_units_out = nu;
    *n_merges_out = nm;
    *chunk_out = static_cast<int>(chunk);
    return PKV_OK;
}

}  // namespace pkv
