// Inline-PTX helpers for the sm_100-family 5th-generation tensor cores
// (tcgen05): tensor-memory (TMEM) allocation, MMA with the accumulator in TMEM,
// commit to an mbarrier, and TMEM <-> register moves.
//
// Conventions used by this library (cta_group::1, M = 128):
// * a TMEM address is (lane << 16) | column; an allocation's base has lane 0;
// * the accumulator D (M x N, fp32) occupies lanes 0..127 (row i in lane i),
//   columns base .. base + N - 1;
// * an A operand held in TMEM (kind::f16) occupies lanes 0..127 (row i in lane
//   i), two fp16 K-elements per 32-bit column (the lower K index in the low half);
// * warp w of the CTA moves data of lanes 32 (w % 4) .. 32 (w % 4) + 31 with the
//   32x32b shapes (thread t of the warp <-> lane 32 (w % 4) + t).
#pragma once

#include <cstdint>

namespace tq {

// Instruction descriptor of tcgen05.mma.kind::f16: fp16 A and B, fp32 D, both
// operands K-major, no negation / sparsity, shape M x N (M = 64 or 128, N a
// multiple of 16 up to 256). Fields: D format bits 4-5 (1 = f32), A format
// bits 7-9 and B format bits 10-12 (0 = f16), A / B major bits 15 / 16
// (0 = K-major), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t tc_idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, no swizzle, K-major "interleaved" layout:
// the operand is tiled into core matrices of 8 rows x 16 bytes (8 fp16 along
// K), each stored as 128 contiguous bytes (row r at byte 16 r). `lbo` is the
// byte distance between core matrices adjacent along K, `sbo` between core
// matrices adjacent along M / N. Fields: start >> 4 in bits 0-13, lbo >> 4 in
// bits 16-29, sbo >> 4 in bits 32-45, descriptor version 1 at bit 46, layout
// type 0 (no swizzle) in bits 61-63.
__device__ __forceinline__ uint64_t tc_sdesc_kmajor(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Allocate `ncols` TMEM columns (a power of two >= 32); the whole warp calls it;
// the base address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// Free an allocation (the warp that allocated it; no tcgen05 operation on it in flight).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (TMEM) (+)= A (TMEM) x B (shared, descriptor); issued by one thread.
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
      : "memory");
}

// Arrive (once) on the mbarrier when every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint32_t mbar_smem) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar_smem)
               : "memory");
}

// 32 consecutive columns of this thread's lane <-> 32 registers. Each move
// waits for its own completion inside the same asm statement, so the compiler
// can neither read a loaded register early nor reuse a stored one too soon.
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
      "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
      "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

}  // namespace tq
