// pa_tc.cuh -- tcgen05 (5th-generation tensor core) helpers for sm_103a:
// tensor-memory allocation, MMA issue with shared-memory and tensor-memory
// operands, commit to mbarriers, tensor-memory loads/stores, and the
// shared-memory matrix and instruction descriptors.
#pragma once

#include <stdint.h>

#include "pa_ptx.cuh"

namespace pa {
namespace tc {

// ---- tensor memory ---------------------------------------------------------------
// Allocates ncols columns (a power of two >= 32) for the CTA; the address is
// written to *dst (shared memory).  Whole warp.
__device__ inline void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ inline void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ inline void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ inline void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ inline void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---- descriptors ------------------------------------------------------------------
// Shared-memory matrix descriptor (sm_100 family) as two 32-bit words: the
// low word holds the start address and the leading byte offset (16-byte
// units), the high word the stride byte offset (16-byte units), descriptor
// version 1 and the 128-byte swizzle layout.  Advancing the start address by
// `off` bytes inside one shared-memory window adds off >> 4 to the low word
// (the 14-bit field cannot carry: shared addresses stay below 256 KB).
__device__ inline uint32_t desc_lo(uint32_t saddr, uint32_t lbo) {
    return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__device__ inline uint32_t desc_hi_sw128(uint32_t sbo) {
    return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
__device__ inline uint64_t make_desc(uint32_t lo, uint32_t hi) {
    return (uint64_t(hi) << 32) | lo;
}

// Instruction descriptor for kind::f16 with f32 accumulation.
//   ab_bf16: operands are bf16 (else f16); b_mn_major: B is MN-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool ab_bf16, bool b_mn_major) {
    return (1u << 4)                                   // D format f32
           | ((ab_bf16 ? 1u : 0u) << 7)                // A format
           | ((ab_bf16 ? 1u : 0u) << 10)               // B format
           | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
           | (uint32_t(N >> 3) << 17)                  // N / 8
           | (uint32_t(M >> 4) << 24);                 // M / 16
}

// ---- MMA ----------------------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem] (mma_ss_elect) and D[tmem] (+)= A[tmem] *
// B[smem] (mma_ts_elect), issued by one elected lane of a converged warp (the
// lowest active lane, so always the same lane while the whole warp runs): the
// operands stay warp-uniform and the issue needs no divergent branch.
__device__ inline void mma_ss_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                    bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}
__device__ inline void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                    bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}
// Arrives on the mbarrier once every tcgen05 operation issued so far by the
// elected lane (the one that issues through the *_elect forms) has completed.
__device__ inline void commit_elect(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ---- tensor-memory loads and stores (32 lanes x 32 columns of 32 bits) --------------
__device__ inline void ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ inline void st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ inline void ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
}

// Stores every other register of r (r[O], r[O + 2], ..., r[O + 30]) to 16
// consecutive columns.
template <int O>
__device__ inline void st_32x32b_x16_stride2(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(r[O]), "r"(r[O + 2]), "r"(r[O + 4]), "r"(r[O + 6]), "r"(r[O + 8]), "r"(r[O + 10]), "r"(r[O + 12]),
        "r"(r[O + 14]), "r"(r[O + 16]), "r"(r[O + 18]), "r"(r[O + 20]), "r"(r[O + 22]), "r"(r[O + 24]),
        "r"(r[O + 26]), "r"(r[O + 28]), "r"(r[O + 30])
        : "memory");
}

__device__ inline void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ inline void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Registers written by tcgen05.ld are only valid after tcgen05.wait::ld.
// The compiler sees the load's outputs as defined at the load, so each use
// is tied to the wait through an empty asm that "rewrites" the registers.
template <int N>
__device__ inline void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

}  // namespace tc
}  // namespace pa
