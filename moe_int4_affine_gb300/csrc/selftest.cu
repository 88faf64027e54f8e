// selftest.cu -- exercises the device-side failure path without faulting anything: a kernel waits,
// with a time limit, on an mbarrier that nothing completes; the wait gives up, records
// QG_STATUS_TIMEOUT in the device status word and the kernel returns normally.
#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

__global__ void selftest_timeout_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);  // expects one arrival; none ever comes
  mbar_fence_init();
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(&bar, 0)) return;  // (cannot happen: the phase never completes)
    if ((i & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) {
      set_status(QG_STATUS_TIMEOUT);
      return;
    }
  }
}

}  // namespace qg

extern "C" int qg_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return QG_EINVAL;
  qg::selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? QG_OK : QG_ELAUNCH;
}
