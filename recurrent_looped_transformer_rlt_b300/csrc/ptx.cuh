// Inline-PTX wrappers for sm_103a: mbarriers and bulk asynchronous copies
// (the TMA engine), used by the streaming kernels.  Every wait is bounded by
// a clock budget; a wait that runs out returns false and the caller records
// a timeout status instead of spinning forever.
#pragma once

#include <stdint.h>

namespace rlt {

__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Makes mbarrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete; false after
// `budget` clock cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, long long budget) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > budget) return false;
  return true;
}

// Bulk copy global -> shared (this CTA), completion signalled on `bar` as
// transaction bytes.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Programmatic dependent launch.  pdl_wait: block until the previous kernel of
// the stream has completed and its memory is visible (immediately when the
// kernel was launched without the programmatic attribute); pdl_trigger: allow
// the next kernel to be scheduled.  Kernels here trigger after their own
// wait, so at most one kernel runs ahead: before its wait a kernel may read
// only data produced two or more kernels earlier (weights, encoder memory).
// The one exception is the RMSNorm kernel (norm_rows_kernel), which triggers
// first: every kernel that follows it reads nothing but weights before its
// wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// ~1 s at the maximum SM clock: a wait that long means the copy engine never
// delivered, which is reported as a timeout.
constexpr long long kWaitBudget = 2000000000LL;

}  // namespace rlt
