// PTX wrappers for the fifth-generation tensor cores of sm_100-family GPUs (PTX ISA:
// "Tensor Memory", "tcgen05" instructions, the shared-memory matrix descriptor and
// the instruction descriptor of tcgen05.mma kind::f16).
//
// The operands of tcgen05.mma are read by the tensor core from shared memory
// through 64-bit matrix descriptors; the accumulator lives in tensor memory (TMEM,
// 128 lanes x 512 columns of 32 bits per SM), which a CTA allocates, reads back
// with tcgen05.ld and frees before it exits. One thread issues the MMAs; their
// completion is signalled on an mbarrier by tcgen05.commit.
#pragma once

#include <cstdint>

namespace pkv {
namespace tc {

// ---- descriptors (host and device, so the encodings are plain functions)

// Shared-memory matrix descriptor of an operand stored in the 128-byte swizzled
// canonical layout: rows of 128 bytes, eight rows to a 1024-byte atom whose 16-byte
// chunks are XOR-ed with the row index within the atom.
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-48  fixed 0b001
//   bits 49-51  base offset (0: atoms start on 1024-byte boundaries)
//   bit  52     leading-dimension stride mode (0: relative)
//   bits 61-63  swizzle mode (2: 128-byte swizzle)
// For a K-major operand the stride offset is the distance between 8-row groups
// (the leading offset is unused with this swizzle); for an MN-major operand the
// leading offset is the distance between 64-element panels along M or N and the
// stride offset the distance between 8-row groups along K.
__host__ __device__ constexpr uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo_bytes,
                                                   uint32_t sbo_bytes) {
    return uint64_t((smem_addr & 0x3FFFFu) >> 4) | (uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo_bytes >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) |
           (uint64_t(2) << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B and an fp32
// accumulator, for an M x N x 16 step:
//   bits  4-5   D format (1: f32)      bits  7-9   A format (1: bf16)
//   bits 10-12  B format (1: bf16)     bit  15     A MN-major   bit 16  B MN-major
//   bits 17-22  N >> 3                 bits 24-28  M >> 4
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n, bool a_mn_major,
                                                      bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn_major) << 15) |
           (uint32_t(b_mn_major) << 16) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

#if defined(__CUDACC__)

// ---- tensor memory allocation (one warp, .sync.aligned)

// Allocates `ncols` columns (a power of two, >= 32) and writes the TMEM address to
// the shared-memory word at `dst_smem`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// ---- ordering

// tcgen05 operations before a thread synchronisation (barrier arrive) ...
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
// ... and after one (barrier wait)
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy writes to shared memory (st.shared, cp.async) before reads of the
// async proxy (the tensor core's operand fetch).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- MMA (one thread)

// D[tmem] (+)= A[smem] * B[smem]^T-ish per the descriptors, one M x N x 16 step.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], one M x N x 16 step with A in tensor memory: row
// i of A in lane i, its 16 bf16 of the step packed two to a 32-bit column (element
// 2j in the low half of column j) from the address's column on.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// The same, issued only where `issue` is true: a whole warp executes the statement
// with warp-uniform operands and one lane issues, so that no branch separates the
// operands from the instruction.
__device__ __forceinline__ void mma_bf16_ss_if(bool issue, uint32_t d_tmem, uint64_t a_desc,
                                               uint64_t b_desc, uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u), "r"(issue ? 1u : 0u)
        : "memory");
}
__device__ __forceinline__ void mma_bf16_ts_if(bool issue, uint32_t d_tmem, uint32_t a_tmem,
                                               uint64_t b_desc, uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u), "r"(issue ? 1u : 0u)
        : "memory");
}
__device__ __forceinline__ void commit_if(bool issue, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %1, 0;\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
        "r"(issue ? 1u : 0u)
        : "memory");
}

// The mbarrier at `bar` receives one arrival when every tcgen05 operation this
// thread issued before has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// ---- TMEM <-> registers (one warp, .sync.aligned): warp w % 4 reaches lanes
// 32 (w % 4) .. + 31; thread t reads / writes lane 32 (w % 4) + t, 32 consecutive
// columns from the address's column on.

#define PKV_TC_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                     "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define PKV_TC_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                     "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// Load and wait in one statement, so no use of the registers can be scheduled
// before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : PKV_TC_R8(0), PKV_TC_R8(8), PKV_TC_R8(16), PKV_TC_R8(24)
        : "r"(taddr)
        : "memory");
}

// 64 consecutive columns in one instruction (and its wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : PKV_TC_R8(0), PKV_TC_R8(8), PKV_TC_R8(16), PKV_TC_R8(24), PKV_TC_R8(32), PKV_TC_R8(40),
          PKV_TC_R8(48), PKV_TC_R8(56)
        : "r"(taddr)
        : "memory");
}

// 128 consecutive columns in one instruction (and its wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, "
        "%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
        "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, "
        "%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, "
        "%112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : PKV_TC_R8(0), PKV_TC_R8(8), PKV_TC_R8(16), PKV_TC_R8(24), PKV_TC_R8(32), PKV_TC_R8(40),
          PKV_TC_R8(48), PKV_TC_R8(56), PKV_TC_R8(64), PKV_TC_R8(72), PKV_TC_R8(80), PKV_TC_R8(88),
          PKV_TC_R8(96), PKV_TC_R8(104), PKV_TC_R8(112), PKV_TC_R8(120)
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        PKV_TC_W8(0), PKV_TC_W8(8), PKV_TC_W8(16), PKV_TC_W8(24)
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef PKV_TC_R8
#undef PKV_TC_W8

#endif  // __CUDACC__

}  // namespace tc
}  // namespace pkv
