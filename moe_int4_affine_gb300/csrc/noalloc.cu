// noalloc.cu -- the MoE gather step for callers that cannot allocate device memory.
//
// moe_gather_qgemv_int4 needs scratch for the SwiGLU activations h[k][inter] and asks the caller
// for it as a workspace.  Some callers have no way to provide one: code running inside a host
// runtime that owns all device memory and forbids new allocations once serving starts (a fixed,
// pre-reserved pool), or a latency-critical decode loop where cudaMalloc's implicit device
// synchronisation is not acceptable.  For them, this file keeps the scratch in a fixed array in the
// library's own device memory: every GPU that loads the library holds it until the process exits.
#include <mutex>

#include "qg_internal.h"

namespace qg {

// Scratch for h[k][inter] (fp32).  File scope: in host code `g_noalloc_h` is only a host-side
// stand-in for the array, never a device address; host code uses the address resolved below.
static __device__ __align__(256) float g_noalloc_h[QG_NOALLOC_MOE_MAX_FLOATS];

namespace {
constexpr int kMaxDev = 64;
float* g_h_ptr[kMaxDev];  // the array's device address per device, once resolved (null before)
std::mutex g_h_mutex;

// Device address of the scratch array on the current device, resolved with that device current on
// the first call made on it.  Only a successful lookup is kept: after a failure (its error cleared
// from the runtime's last-error state) the next call tries again.
float* scratch_for_current_device(int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    (void)cudaGetLastError();
    *err = QG_EDEVICE;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_h_mutex);
  if (!g_h_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_h) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      *err = QG_EDEVICE;
      return nullptr;
    }
    g_h_ptr[dev] = static_cast<float*>(p);
  }
  *err = QG_OK;
  return g_h_ptr[dev];
}
}  // namespace

}  // namespace qg

using namespace qg;

extern "C" int moe_gather_qgemv_int4_noalloc(const qg_int4_weight* gate, const qg_int4_weight* up,
                                             const qg_int4_weight* down, const uint32_t* idx, const float* p, int k,
                                             const uint16_t* x, const uint16_t* residual, float* y, void* stream) {
  // the same argument checks as moe_gather_qgemv_int4, with the library's scratch as workspace
  if (!gate || !up || !down) return QG_EINVAL;
  if (k >= 1 && (size_t)k * (size_t)(down->in > 0 ? down->in : 0) > (size_t)QG_NOALLOC_MOE_MAX_FLOATS)
    return QG_ENOTSUP;
  int err = QG_OK;
  float* h = scratch_for_current_device(&err);
  if (err != QG_OK) return err;
  return moe_gather_qgemv_int4(gate, up, down, idx, p, k, x, residual, y, h,
                               sizeof(float) * (size_t)QG_NOALLOC_MOE_MAX_FLOATS, stream);
}
