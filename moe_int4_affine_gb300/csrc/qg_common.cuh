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
// The suspend-time hint lets the hardware park the waiting thread (no instruction issue) until the
// phase completes or about a microsecond passes.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000u)
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
// 1-D global -> shared copy, completion counted on `bar` in bytes, with an L2 cache hint.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Bulk prefetch of a global range into L2 (no shared memory, no completion tracking).  `bytes` a
// multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Weights are streamed once per call: mark them evict-first so activations and outputs stay.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
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

// Pack two floats into f16x2 (round to nearest even), lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16_lo_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.f32.f16 %0, a;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}
__device__ __forceinline__ float f16_hi_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %1;\n\tcvt.f32.f16 %0, b;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

// acc += a.lo * b.lo + a.hi * b.hi with f16 operands and an fp32 accumulator (sm_100+ mixed
// precision FMA: the f16 x f16 product is exact in fp32, one rounding per add).
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float acc) {
  asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
      "mov.b32 {a0, a1}, %1;\n\t"
      "mov.b32 {b0, b1}, %2;\n\t"
      "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
      "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}

// ---------------------------------------------------------------- int4 nibble -> f16 codes
// One u32 word holds codes q0..q7 (q_i in bits 4i..4i+3).  A 16-bit half whose exponent field
// (bits 10..14) and sign are zero is an IEEE binary16 subnormal worth (bits) * 2^-24, so masking
// a nibble into bits 0..3 of a half gives exactly q * 2^-24, and into bits 4..7 gives exactly
// 16 q * 2^-24 -- no implicit leading one, nothing to subtract.  Returned pairs (low half first):
//   h[0] = (q0, q4) * 2^-24        h[1] = (q1, q5) * 16 * 2^-24
//   h[2] = (q2, q6) * 2^-24        h[3] = (q3, q7) * 16 * 2^-24
// The x operand paired with h[1] and h[3] is pre-divided by 16.
__device__ __forceinline__ void nibbles_to_f16_subnormal(uint32_t w, uint32_t h[4]) {
  const uint32_t w8 = w >> 8;
  h[0] = w & 0x000F000Fu;
  h[1] = w & 0x00F000F0u;
  h[2] = w8 & 0x000F000Fu;
  h[3] = w8 & 0x00F000F0u;
}

}  // namespace qg
