// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "pkv.h"

namespace pkv {

// ---- errors -------------------------------------------------------------
int fail(int code, const char* fmt, ...);  // records the message, returns code
void clear_error();
bool debug_checks();

// ---- plan ----------------------------------------------------------------
// One work unit of the split-KV kernel: tokens [tok_begin, tok_end) of request b,
// all KV heads. partial < 0: the unit covers the whole context and writes out/lse;
// otherwise it writes partial slot `partial` of the workspace.
struct Unit {
    int32_t b, tok_begin, tok_end, partial;
};
// One split request: its parts occupy partial slots [first, first + count).
struct Merge {
    int32_t b, first, count, pad;
};
static_assert(sizeof(Unit) == 16 && sizeof(Merge) == 16, "16-byte plan records");

struct PlanShape {
    int num_sms;
    int ctas_per_sm;
};

// Tokens below which a context is never split: a split costs one fp32 partial
// (n_qo_heads * head_dim * 4 bytes written and read back) and is only worth it
// when the chunk it creates reads much more than that.
constexpr int kMinChunkTokens = 256;
// Chunk lengths are multiples of this many tokens.
constexpr int kChunkQuantum = 64;
// Work units the planner aims for, per resident CTA slot of the device.
constexpr int kWavesTarget = 4;

int plan_target_units(const PlanShape& s);
// Pure host planner. Returns PKV_OK or PKV_ERR_PLAN (arrays too small) /
// PKV_ERR_INVALID_ARG (bad indptr).
int plan_compute(const int32_t* indptr, int batch, const PlanShape& shape, Unit* units,
                 int max_units, Merge* merges, int max_merges, int* n_units, int* n_merges,
                 int* chunk_tokens);

// ---- kernels -------------------------------------------------------------
struct DecodeArgs {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const int32_t* kv_indptr;
    const int32_t* kv_indices;
    const Unit* units;
    const Merge* merges;
    int n_units;
    int n_merges;
    int n_qo_heads;
    int n_kv_heads;
    int head_dim;
    float sm_scale;
    void* out;
    float* lse;
    float* ws_o;    // [max_units, n_qo_heads, head_dim] fp32 partial outputs
    float* ws_lse;  // [max_units, n_qo_heads] fp32 partial lse (base 2)
};

bool decode_shape_supported(int n_qo_heads, int n_kv_heads, int head_dim);
// Resident CTAs per SM of the split kernel for this shape (0 on error).
int decode_ctas_per_sm(int n_qo_heads, int n_kv_heads, int head_dim);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

cudaError_t launch_append(void* k_pool, void* v_pool, const int32_t* slot_ids,
                          const void* k_new, const void* v_new, int64_t n, int row_bytes,
                          cudaStream_t stream);

}  // namespace pkv

struct pkv_plan {
    int device = 0;
    pkv::PlanShape shape{};
    int max_batch = 0;
    int64_t max_tokens = 0;
    int n_qo_heads = 0, n_kv_heads = 0, head_dim = 0;
    int max_units = 0, max_merges = 0;
    void* host_staging = nullptr;  // pinned: units[max_units] then merges[max_merges]
    void* dev_meta = nullptr;      // device copy of the same
    float* ws_o = nullptr;
    float* ws_lse = nullptr;
    cudaEvent_t copy_done = nullptr;
    bool copy_pending = false;
    // the current step
    bool planned = false;
    int batch = 0, n_units = 0, n_merges = 0, chunk_tokens = 0;
    std::vector<int32_t> indptr_host;

    pkv::Unit* host_units() { return static_cast<pkv::Unit*>(host_staging); }
    pkv::Merge* host_merges() { return reinterpret_cast<pkv::Merge*>(host_units() + max_units); }
    const pkv::Unit* dev_units() const { return static_cast<const pkv::Unit*>(dev_meta); }
    const pkv::Merge* dev_merges() const {
        return reinterpret_cast<const pkv::Merge*>(dev_units() + max_units);
    }
};
