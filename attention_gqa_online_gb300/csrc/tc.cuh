// tc.cuh -- tcgen05 (5th-generation tensor core) helpers: tensor-memory
// allocation, shared-memory matrix descriptors, instruction descriptors, MMA
// issue, commit, and tensor-memory loads/stores.  Written from the PTX ISA's
// descriptions of the tcgen05 instructions and descriptor formats.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace attn {
namespace tc {

// ---------------------------------------------------------------- tensor memory
// Allocates `ncols` (power of two, 32..512) TMEM columns; the whole warp must
// call it.  The base address is written to *smem_dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor, 128-byte swizzle.  Fields: start address
// >> 4 (bits 0-13), leading-dimension byte offset >> 4 (16-29), stride-dimension
// byte offset >> 4 (32-45), descriptor version 1 (46-47), base offset 0
// (49-51), swizzle mode 2 = 128-byte (61-63).
//   K-major operand: rows of 128 bytes, 8-row groups `sbo` bytes apart; the
//     leading offset is unused.  Successive K steps inside the 128-byte row
//     advance the start address.
//   MN-major operand: each K row holds 128 bytes of MN; `lbo` is the distance
//     between 128-byte MN chunks, `sbo` between 8-row K groups.
// Layout type 1 (128-byte swizzle of 32-byte chunks) is the form a 32-bit
// MN-major operand needs; the tensor map that fills it uses the matching TMA
// swizzle.
enum : uint32_t { kLayoutSw128 = 2, kLayoutSw128Atom32 = 1 };
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                                uint32_t layout = kLayoutSw128) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)layout << 61;
  return d;
}

// Instruction descriptor for kind::tf32 / kind::f16 with fp32 accumulation:
// D format F32 (bits 4-5 = 1), A/B formats (bits 7-9 / 10-12: 0 F16, 1 BF16,
// 2 TF32), B major (bit 16: 0 K-major, 1 MN-major), N >> 3 (bits 17-22),
// M >> 4 (bits 24-28).  A is always K-major here.
enum : uint32_t { kFmtF16 = 0, kFmtBF16 = 1, kFmtTF32 = 2 };
__host__ __device__ constexpr uint32_t idesc_f32acc(uint32_t fmt, bool b_mn_major, int M, int N) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- MMA issue (one thread)
// D[tmem] (+)= A * B^T with A, B from shared memory.
__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// A from tensor memory.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Four MMAs into one accumulator in a single block: D (+)= A_i * B_i^T for
// i = 0..3, the first accumulating iff `accumulate` != 0, the others always.
// The whole warp executes the block with warp-uniform operands and one
// elected lane issues the MMAs.  An issuing warp that shares its SM
// sub-partition with busy warps gets few issue slots, so the instructions
// around each MMA are kept to a minimum.
#define ATTN_MMA4(KIND, AFORM)                                                                              \
  asm volatile(                                                                                             \
      "{\n\t.reg .pred p, t, e;\n\telect.sync _|e, 0xffffffff;\n\t"                                          \
      "setp.ne.b32 p, %10, 0;\n\tsetp.eq.b32 t, %10, %10;\n\t"                                                 \
      "@e tcgen05.mma.cta_group::1.kind::" KIND " [%0], " AFORM(1) ", %5, %9, p;\n\t"                        \
      "@e tcgen05.mma.cta_group::1.kind::" KIND " [%0], " AFORM(2) ", %6, %9, t;\n\t"                        \
      "@e tcgen05.mma.cta_group::1.kind::" KIND " [%0], " AFORM(3) ", %7, %9, t;\n\t"                        \
      "@e tcgen05.mma.cta_group::1.kind::" KIND " [%0], " AFORM(4) ", %8, %9, t;\n\t}"
#define ATTN_A_DESC(i) "%" #i
#define ATTN_A_TMEM(i) "[%" #i "]"
__device__ __forceinline__ void mma4_f16_ss(uint32_t d, uint64_t a0, uint64_t a1, uint64_t a2, uint64_t a3, uint64_t b0,
                                            uint64_t b1, uint64_t b2, uint64_t b3, uint32_t idesc, uint32_t accumulate) {
  ATTN_MMA4("f16", ATTN_A_DESC)::"r"(d), "l"(a0), "l"(a1), "l"(a2), "l"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3),
      "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma4_f16_ts(uint32_t d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint64_t b0,
                                            uint64_t b1, uint64_t b2, uint64_t b3, uint32_t idesc, uint32_t accumulate) {
  ATTN_MMA4("f16", ATTN_A_TMEM)::"r"(d), "r"(a0), "r"(a1), "r"(a2), "r"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3),
      "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma4_tf32_ts(uint32_t d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint64_t b0,
                                             uint64_t b1, uint64_t b2, uint64_t b3, uint32_t idesc, uint32_t accumulate) {
  ATTN_MMA4("tf32", ATTN_A_TMEM)::"r"(d), "r"(a0), "r"(a1), "r"(a2), "r"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3),
      "r"(idesc), "r"(accumulate)
      : "memory");
}
#undef ATTN_A_TMEM
#undef ATTN_A_DESC
#undef ATTN_MMA4

// Warp-uniform form of commit(): one elected lane of the (converged) warp
// commits, so the barrier gets exactly one arrival.
__device__ __forceinline__ void commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------- TMEM <-> registers
// 32x32b shape: thread i of the warp reads/writes TMEM lane (lane base + i),
// 32 consecutive 32-bit columns starting at the address's column.
#define ATTN_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]), "=r"(v[i + 5]), \
                   "=r"(v[i + 6]), "=r"(v[i + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24)
      : "r"(taddr));
}
// The first 16 of v from 16 consecutive columns (v[16..31] are left as is).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : ATTN_R8(0), ATTN_R8(8)
      : "r"(taddr));
}
#undef ATTN_R8
#define ATTN_W8(i) "r"(v[i]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), "r"(v[i + 4]), "r"(v[i + 5]), \
                   "r"(v[i + 6]), "r"(v[i + 7])
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      ATTN_W8(0), ATTN_W8(8), ATTN_W8(16), ATTN_W8(24)
      : "memory");
}
// The first 16 of v into 16 consecutive columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      ATTN_W8(0), ATTN_W8(8)
      : "memory");
}
#undef ATTN_W8
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// After tmem_ld_wait(): ties the loaded registers to that point, so no use of
// them is scheduled before the wait.
#define ATTN_F8(i) "+r"(v[i]), "+r"(v[i + 1]), "+r"(v[i + 2]), "+r"(v[i + 3]), "+r"(v[i + 4]), "+r"(v[i + 5]), \
                   "+r"(v[i + 6]), "+r"(v[i + 7])
__device__ __forceinline__ void reg_fence(uint32_t (&v)[32]) {
  asm volatile("" : ATTN_F8(0), ATTN_F8(8), ATTN_F8(16), ATTN_F8(24)::"memory");
}
__device__ __forceinline__ void reg_fence16(uint32_t (&v)[32]) {
  asm volatile("" : ATTN_F8(0), ATTN_F8(8)::"memory");
}
#undef ATTN_F8
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- bf16 packing
// Two floats as round-to-nearest-even bf16 in one word: lo in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The two fp16 halves of a word as floats (lo = bits 0-15).
__device__ __forceinline__ float2 unpack_f16(uint32_t v) {
  float lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(v));
  return make_float2(lo, hi);
}

// Two floats as round-to-nearest-even fp16 in one word: lo in bits 0-15.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace tc
}  // namespace attn
