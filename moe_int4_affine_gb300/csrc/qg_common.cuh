// qg_common.cuh -- device helpers shared by the qg kernels (sm_103a).
//
// Inline PTX for: mbarriers, 1-D bulk async copies (TMA engine, non-multicast), programmatic
// dependent launch (griddepcontrol), and bounded waits.  Every wait in this library gives up
// after a time limit, records an error bit in the device status word and lets the kernel return.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qg.h"

namespace qg {

// Device status word: bits from enum qg_status_bits (include/qg.h).  Defined in api.cu; read and
// cleared by qg_device_status().
extern __device__ uint32_t g_status;

__device__ __forceinline__ void set_status(uint32_t bits) { atomicOr(&g_status, bits); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Non-blocking test of the phase with the given parity (no suspend-time hint: with one, the wait was
// measured to sleep far past the phase's completion).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and sets
// QG_STATUS_TIMEOUT) if it has not completed within kWaitLimitNs.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait here
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
      set_status(QG_STATUS_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- bulk copies (TMA engine)
// 1-D global -> shared copy, completion counted on `bar` in bytes.  dst, src and bytes must be
// multiples of 16.  The copy goes through the async proxy: memory that generic accesses touched
// earlier in the same kernel needs a proxy fence (fence.proxy.async) before it.
__device__ __forceinline__ void bulk_g2s_bytes(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// The line holding p into L2 (no value returned; also brings its address translation along).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---------------------------------------------------------------- programmatic dependent launch
// Wait until the preceding kernel in the stream has completed and its writes are visible.  A
// no-op when the kernel was launched without the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream (if launched with the attribute) to start launching.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- shared-memory loads (32-bit addresses)
// volatile: these read buffers filled by the async proxy after an mbarrier wait and must not be
// hoisted above it.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// ---------------------------------------------------------------- small numeric helpers
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

}  // namespace qg
