// common.cuh -- small device helpers shared by the attention kernels:
// status word, bounded mbarrier waits, bulk/async copies, exp2.
// Inline PTX is written from the PTX ISA's descriptions of each instruction.
#pragma once

#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attn_gqa.h"

namespace attn {

// Records `code` in the per-device status word (the largest code wins).
__device__ __forceinline__ void record_status(unsigned* status, unsigned code) { atomicMax(status, code); }

// Wall-clock limit of every spin-wait in the library's kernels.
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s
constexpr unsigned kWaitSliceNs = 2000;  // longest sleep of one bounded-wait step

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep for up to `hint_ns` while the
// phase is incomplete; completing the phase wakes it at once.
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t* bar, unsigned parity, unsigned hint_ns) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Non-blocking test: has phase `parity` of `bar` completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Named barrier over `count` threads (a multiple of 32) with id 1..15.
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Arrives on named barrier `id` without waiting (the other `count` - 32*k
// threads wait with named_barrier()).
__device__ __forceinline__ void named_barrier_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Waits for phase `parity` of `bar` to complete, for at most kWaitLimitNs.
// Returns false (and records ATTN_ERR_TIMEOUT in *status) if the limit ran
// out.  `abort_flag` (shared memory, optional) is set on a timeout; once it
// is set, later waits of the same CTA give up at once, so a CTA whose
// pipeline broke finishes quickly instead of timing out wait after wait.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity, unsigned* status,
                                                  volatile int* abort_flag = nullptr,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    // Sleeps until the phase completes (or 2 us pass, for the checks below).
    if (mbar_try_wait_for(bar, parity, kWaitSliceNs)) return true;
    if (abort_flag != nullptr && *abort_flag != 0) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      record_status(status, ATTN_ERR_TIMEOUT);
      if (abort_flag != nullptr) *abort_flag = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------- bulk copy (TMA, non-tensor)
// Global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) that completes `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Tiled tensor copies (TMA) global -> shared, completing on `bar`.  The
// coordinates are element indices, innermost first.
__device__ __forceinline__ void tma_load_2d(void* dst_smem, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// Hint: bring one tile of a tensor map into L2 (no shared memory, no
// completion; a tile outside the tensor reads nothing).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst_smem, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst_smem)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// Tiled tensor copy shared -> global (TMA store), in the bulk group of the
// issuing thread.  Rows of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src_smem, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(smem_u32(src_smem))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Waits until every committed bulk store of this thread has read its shared
// memory source (the global writes may still be in flight; they are done
// when the grid completes).
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- cp.async (Ampere-style)
// 16-byte async copy; when src_bytes == 0 the destination is zero-filled.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src, unsigned src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst_smem)), "l"(src), "r"(src_bytes)
               : "memory");
}
// 4-byte async copy with the same zero-fill rule.
__device__ __forceinline__ void cp_async4(void* dst_smem, const void* src, unsigned src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst_smem)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels launched with programmatic stream serialization may start while the
// previous kernel in the stream is finishing.  grid_dependency_wait() blocks
// until that kernel has completed and its memory is visible: call it before
// the first global read or write.  allow_dependent_launch() lets the next
// such kernel start launching (its CTAs then wait in their own
// grid_dependency_wait()).  Both are no-ops for an ordinary launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// ---------------------------------------------------------------- math
// 2^x with the hardware's approximate exp2 (MUFU.EX2); 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-way max (one instruction on this architecture).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a0, a1) += (b0, b1) as one paired fp32 add.
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "add.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// (a0, a1) = (a0 * b0 + c0, a1 * b1 + c1) as one paired fp32 fma.
__device__ __forceinline__ void fma2(float& a0, float& a1, float b0, float b1, float c0, float c1) {
  asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\tmov.b64 z, {%4, %5};\n\t"
      "fma.rn.f32x2 x, x, y, z;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// (a0, a1) += (x0 * y0, x1 * y1) as one paired fp32 fma (each result rounded
// once, as fmaf).
__device__ __forceinline__ void fma2_acc(float& a0, float& a1, float x0, float x1, float y0, float y1) {
  asm("{\n\t.reg .b64 a, x, y;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "fma.rn.f32x2 a, x, y, a;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}

// Power-of-two range scaling of 16-bit tensor-core operands.  For the
// largest magnitude m of a set of values, pow2_scale_exp gives E such that
// m * 2^(14 - E) lies in [2^14, 2^15) (exactly representable range of fp16,
// whose largest finite value is 65504), with E clamped to [-100, 127] so both
// 2^(14 - E) and 2^(E - 14) are normal fp32 numbers.  A zero or subnormal m
// gives -100; an infinite or NaN m gives 127 (inf and NaN then stay so).
__host__ __device__ __forceinline__ int pow2_scale_exp(float m) {
  uint32_t bits;
  memcpy(&bits, &m, 4);
  int e = (int)((bits >> 23) & 0xffu) - 127;
  return e < -100 ? -100 : (e > 127 ? 127 : e);
}
// 2^k for -126 <= k <= 127, exact.
__host__ __device__ __forceinline__ float pow2f(int k) {
  const uint32_t bits = (uint32_t)(127 + k) << 23;
  float f;
  memcpy(&f, &bits, 4);
  return f;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kEmptyLse = -1e30f;

}  // namespace attn
