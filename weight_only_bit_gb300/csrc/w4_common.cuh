// w4_common.cuh -- device-side building blocks shared by libw4's kernels (sm_103a).
//
// Inline PTX for the Blackwell pieces: mbarrier phases, 1-D bulk async copies (the TMA unit's
// cp.async.bulk, global -> shared, completion counted on an mbarrier), programmatic dependent
// launch control (griddepcontrol), and a device error word for bounded waits.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace w4 {

// Set by a kernel whose bounded wait ran out (never by a normal run).  Values: 0 = fine, otherwise
// a site code identifying the wait.  Without relocatable device code every translation unit that
// includes this header holds its own copy of the word, so each one whose kernels wait exports a
// reader built on read_clear_error_word_here(), and w4_device_check() combines all of them.
static __device__ unsigned int g_error_word = 0;

// Host side: reads and clears this translation unit's copy of the error word on the current device
// (synchronous with respect to the device).
static inline unsigned int read_clear_error_word_here() {
  unsigned int v = 0;
  const unsigned int z = 0;
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return 0;
  if (v != 0) cudaMemcpyToSymbol(g_error_word, &z, sizeof(z));
  return v;
}

// Wall-clock limit of one mbarrier wait.  A healthy wait ends within microseconds (one DRAM
// round trip); a wait still open after a second is treated as lost.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One potentially blocking test of a phase: a thread whose phase is still open is suspended by the
// hardware (issuing nothing) until the phase completes or about kSuspendHintNs pass.
constexpr uint32_t kSuspendHintNs = 20000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs) : "memory");
  return ok != 0;
}

// Bounded wait on one phase.  Returns false (after recording `site` in the error word) if the
// phase did not complete within kWaitLimitNs of wall-clock time.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) break;
  }
  atomicCAS(&g_error_word, 0u, site);
  return false;
}

// 1-D bulk copy global -> shared (TMA unit).  dst, src 16-byte aligned; bytes a multiple of 16.
// Completion adds `bytes` to the transaction count of `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

// L2 policy: weights are read exactly once, so ask L2 to evict them first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Programmatic dependent launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

}  // namespace w4
