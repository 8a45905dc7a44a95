// Oracle for paged GQA decode attention over a page-size-1 token pool.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the library path calls, links or loads this
// file; only the tests, the smoke check and the benchmark's CPU-baseline leg do.
// It shares no code, header or constant with the CUDA path.
//
// What is computed, and where it is stated:
//  * The KV cache is a token pool with page size 1: one pool row per token slot,
//    and a decode batch lists, per request, the slots of its context
//    ("Agent-Infer: 纯 Rust 编写的高性能 LLM 推理引擎", section "分页 KV 缓存"
//    (paged KV cache): SGLang's TokenToKVPool pattern with page size 1, decode
//    batched across all requests).
//  * Grouped-query attention: the query heads are split into groups that share
//    one K/V head, 32 query heads on 8 KV heads at head_dim 128, and head_dim 256
//    on the hybrid model's full-attention layers ("Pegainfer: 纯Rust+CUDA构建的
//    LLM推理引擎", sections "1. 注意力机制优化" and "2. Qwen3.5的混合架构支持").
//    Reading taken: contiguous groups, query head h uses KV head h / G.
//  * The attention itself is the plain softmax definition, evaluated in fp64
//    with every bf16 input widened exactly:
//        s_j   = scale * sum_d q[b,h,d] * K[idx_j, g, d]
//        lse   = m + ln sum_j exp(s_j - m),   m = max_j s_j
//        out   = sum_j exp(s_j - lse) * V[idx_j, g, :]
//    An empty context gives out = 0 and lse = -inf (a reading: the pages are
//    silent on it).
//  * The log-sum-exp merge of attention over disjoint parts of one context,
//    the identity that lets a context be split: lse = ln sum_c exp(lse_c) and
//    out = sum_c exp(lse_c - lse) * out_c.
//  * The append is a row copy: pool[slot_ids[i]] = rows[i].
//  * Chunked prefill over the same pool ("Agent-Infer", section "连续批处理"
//    (continuous batching): long prefills are cut into chunks of 512 tokens, 64
//    while decodes are running, so decode steps can run between chunks). Reading
//    taken: a chunk holds the request's newest C tokens, already appended, so its
//    slot list has L >= C entries and query token i of the chunk (i < C) sits at
//    position p = L - C + i; it attends causally to list entries 0 .. p, with the
//    same softmax definition as above.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

inline double widen_bf16(uint16_t bits) {
    uint32_t w = static_cast<uint32_t>(bits) << 16;
    float f;
    std::memcpy(&f, &w, sizeof f);
    return static_cast<double>(f);
}

}  // namespace

extern "C" {

// Attention for every (request b, query head h).
//   q      : [batch, n_qo_heads, head_dim] bf16 bit patterns
//   k_pool : [pool_slots, n_kv_heads, head_dim] bf16 bit patterns (v_pool alike)
//   kv_indptr [batch+1], kv_indices [kv_indptr[batch]] : CSR slot lists
//   out    : [batch, n_qo_heads, head_dim] fp64;  lse : [batch, n_qo_heads] fp64
// Returns 0, or -1 on a bad argument (shape, CSR or slot out of range).
int oracle_decode(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                  const int32_t* kv_indptr, const int32_t* kv_indices, int64_t batch,
                  int64_t n_qo_heads, int64_t n_kv_heads, int64_t head_dim,
                  int64_t pool_slots, float sm_scale, double* out, double* lse,
                  int n_threads) {
    if (batch < 0 || n_kv_heads <= 0 || n_qo_heads % n_kv_heads != 0 || head_dim <= 0)
        return -1;
    if (kv_indptr[0] != 0) return -1;
    for (int64_t b = 0; b < batch; ++b) {
        if (kv_indptr[b + 1] < kv_indptr[b]) return -1;
    }
    for (int64_t i = 0; i < kv_indptr[batch]; ++i) {
        if (kv_indices[i] < 0 || kv_indices[i] >= pool_slots) return -1;
    }
    const int64_t G = n_qo_heads / n_kv_heads;
    const double scale = static_cast<double>(sm_scale);
    const int64_t pairs = batch * n_qo_heads;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
    {
        std::vector<double> qd(head_dim), s;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t bh = 0; bh < pairs; ++bh) {
            const int64_t b = bh / n_qo_heads;
            const int64_t h = bh % n_qo_heads;
            const int64_t g = h / G;
            const int64_t begin = kv_indptr[b], L = kv_indptr[b + 1] - begin;
            double* o = out + bh * head_dim;
            for (int64_t d = 0; d < head_dim; ++d) {
                qd[d] = widen_bf16(q[bh * head_dim + d]);
                o[d] = 0.0;
            }
            if (L == 0) {
                lse[bh] = -std::numeric_limits<double>::infinity();
                continue;
            }
            s.assign(L, 0.0);
            double m = -std::numeric_limits<double>::infinity();
            for (int64_t j = 0; j < L; ++j) {
                const uint16_t* k = k_pool + (int64_t(kv_indices[begin + j]) * n_kv_heads + g) * head_dim;
                double dot = 0.0;
                for (int64_t d = 0; d < head_dim; ++d) dot += qd[d] * widen_bf16(k[d]);
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
            }
            double sum = 0.0;
            for (int64_t j = 0; j < L; ++j) sum += std::exp(s[j] - m);
            const double l = m + std::log(sum);
            lse[bh] = l;
            for (int64_t j = 0; j < L; ++j) {
                const double p = std::exp(s[j] - l);
                const uint16_t* v = v_pool + (int64_t(kv_indices[begin + j]) * n_kv_heads + g) * head_dim;
                for (int64_t d = 0; d < head_dim; ++d) o[d] += p * widen_bf16(v[d]);
            }
        }
    }
    return 0;
}

// Causal attention of prefill chunks over their requests' slot lists.
//   q      : [qo_indptr[batch], n_qo_heads, head_dim] bf16 bit patterns; request b's
//            chunk is rows qo_indptr[b] .. qo_indptr[b+1]
//   k_pool, v_pool, kv_indptr, kv_indices : as for oracle_decode; request b lists
//            L_b = kv_indptr[b+1] - kv_indptr[b] >= C_b = qo_indptr[b+1] - qo_indptr[b]
//   out    : [qo_indptr[batch], n_qo_heads, head_dim] fp64; lse : [qo_indptr[batch], n_qo_heads]
// Query row i of request b (chunk index c = i - qo_indptr[b]) is at position
// p = L_b - C_b + c and attends list entries 0 .. p.
// Returns 0, or -1 on a bad argument.
int oracle_prefill(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                   const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                   int64_t batch, int64_t n_qo_heads, int64_t n_kv_heads, int64_t head_dim,
                   int64_t pool_slots, float sm_scale, double* out, double* lse, int n_threads) {
    if (batch < 0 || n_kv_heads <= 0 || n_qo_heads % n_kv_heads != 0 || head_dim <= 0)
        return -1;
    if (kv_indptr[0] != 0 || qo_indptr[0] != 0) return -1;
    for (int64_t b = 0; b < batch; ++b) {
        if (kv_indptr[b + 1] < kv_indptr[b] || qo_indptr[b + 1] < qo_indptr[b]) return -1;
        if (qo_indptr[b + 1] - qo_indptr[b] > kv_indptr[b + 1] - kv_indptr[b]) return -1;
    }
    for (int64_t i = 0; i < kv_indptr[batch]; ++i) {
        if (kv_indices[i] < 0 || kv_indices[i] >= pool_slots) return -1;
    }
    const int64_t G = n_qo_heads / n_kv_heads;
    const double scale = static_cast<double>(sm_scale);
    const int64_t rows = int64_t(qo_indptr[batch]) * n_qo_heads;
    // request of every query row
    std::vector<int64_t> req(qo_indptr[batch]);
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t i = qo_indptr[b]; i < qo_indptr[b + 1]; ++i) req[i] = b;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
#endif
    {
        std::vector<double> qd(head_dim), s;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t ih = 0; ih < rows; ++ih) {
            const int64_t i = ih / n_qo_heads;
            const int64_t kv_head = (ih % n_qo_heads) / G;
            const int64_t b = req[i];
            const int64_t first = kv_indptr[b];
            const int64_t L = kv_indptr[b + 1] - first;
            const int64_t C = qo_indptr[b + 1] - qo_indptr[b];
            const int64_t pos = L - C + (i - qo_indptr[b]);  // position of this query
            const int64_t n_seen = pos + 1;                  // entries 0 .. pos
            double* orow = out + ih * head_dim;
            for (int64_t d = 0; d < head_dim; ++d) {
                qd[d] = widen_bf16(q[ih * head_dim + d]);
                orow[d] = 0.0;
            }
            s.assign(n_seen, 0.0);
            double smax = -std::numeric_limits<double>::infinity();
            for (int64_t j = 0; j < n_seen; ++j) {
                const int64_t row = int64_t(kv_indices[first + j]) * n_kv_heads + kv_head;
                double qk = 0.0;
                for (int64_t d = 0; d < head_dim; ++d) qk += qd[d] * widen_bf16(k_pool[row * head_dim + d]);
                s[j] = qk * scale;
                smax = std::fmax(smax, s[j]);
            }
            double denom = 0.0;
            for (int64_t j = 0; j < n_seen; ++j) denom += std::exp(s[j] - smax);
            const double log_denom = smax + std::log(denom);
            lse[ih] = log_denom;
            for (int64_t j = 0; j < n_seen; ++j) {
                const int64_t row = int64_t(kv_indices[first + j]) * n_kv_heads + kv_head;
                const double w = std::exp(s[j] - log_denom);
                for (int64_t d = 0; d < head_dim; ++d) orow[d] += w * widen_bf16(v_pool[row * head_dim + d]);
            }
        }
    }
    return 0;
}

// Row append: pool[slot_ids[i], :] = rows[i, :] for i < n, row_elems bf16 per row.
// Returns 0, or -1 if a slot is out of range (the pool is then left untouched).
int oracle_append(uint16_t* pool, const int32_t* slot_ids, const uint16_t* rows, int64_t n,
                  int64_t row_elems, int64_t pool_slots) {
    for (int64_t i = 0; i < n; ++i)
        if (slot_ids[i] < 0 || slot_ids[i] >= pool_slots) return -1;
    for (int64_t i = 0; i < n; ++i)
        std::memcpy(pool + int64_t(slot_ids[i]) * row_elems, rows + i * row_elems,
                    sizeof(uint16_t) * row_elems);
    return 0;
}

// Log-sum-exp merge of n_parts attention results over disjoint parts of the same
// contexts. outs: [n_parts, rows, head_dim], lses: [n_parts, rows] -> out, lse.
// Parts with lse = -inf (empty) contribute nothing; all parts empty gives out = 0,
// lse = -inf.
int oracle_lse_merge(const double* outs, const double* lses, int64_t n_parts, int64_t rows,
                     int64_t head_dim, double* out, double* lse) {
    const double ninf = -std::numeric_limits<double>::infinity();
    for (int64_t r = 0; r < rows; ++r) {
        double m = ninf;
        for (int64_t c = 0; c < n_parts; ++c) m = std::fmax(m, lses[c * rows + r]);
        for (int64_t d = 0; d < head_dim; ++d) out[r * head_dim + d] = 0.0;
        if (m == ninf) {
            lse[r] = ninf;
            continue;
        }
        double sum = 0.0;
        for (int64_t c = 0; c < n_parts; ++c) sum += std::exp(lses[c * rows + r] - m);
        const double l = m + std::log(sum);
        lse[r] = l;
        for (int64_t c = 0; c < n_parts; ++c) {
            const double w = std::exp(lses[c * rows + r] - l);
            if (w == 0.0) continue;
            for (int64_t d = 0; d < head_dim; ++d)
                out[r * head_dim + d] += w * outs[(c * rows + r) * head_dim + d];
        }
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

}  // extern "C"
