// qg_internal.h -- host-side interface between the C ABI layer (api.cu) and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/qg.h"

namespace qg {

// Device properties the planners need (queried once per device).
struct DeviceInfo {
  int num_sms;
  int max_smem_optin;
  int id;  // the device's ordinal
};
const DeviceInfo& device_info();

bool pdl_enabled();

// Launch a kernel with the library's launch attributes (programmatic dependent launch when
// enabled).  Returns QG_OK or QG_ELAUNCH.
template <typename... KArgs, typename... Args>
int launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) return QG_ELAUNCH;
  e = cudaGetLastError();
  return e == cudaSuccess ? QG_OK : QG_ELAUNCH;
}

// The same with the kernel's CTAs grouped into clusters of `cluster` along x (1: no cluster); the
// grid must be a multiple of it.
template <typename... KArgs, typename... Args>
int launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, int cluster,
                   Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl_enabled()) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cluster > 1) {
    if (grid.x % (unsigned)cluster != 0) return QG_EINVAL;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) return QG_ELAUNCH;
  e = cudaGetLastError();
  return e == cudaSuccess ? QG_OK : QG_ELAUNCH;
}

// ---------------------------------------------------------------- GEMV family (qgemv.cu)
struct GemvMatArg {
  const uint32_t* packed;
  const uint16_t* scales;
  const uint16_t* biases;
  float* y;
  int out;
};
// Optional prologue / epilogue of a dense or pair GEMV: RMSNorm of x (gamma set), and the gated
// epilogue y = base + sigmoid(*sgate) * (W x) (sgate set) followed by + resid (resid set).
struct GemvExtras {
  const uint16_t* gamma;
  float eps;
  const void* gz;  // gated RMSNorm: z (the type of x), per head of head_dim columns (needs gamma)
  int head_dim;
  const float* sgate;
  const float* ebase;
  const uint16_t* resid;
  int bits;  // 0 or 4: Q4_64A codes; 2: Q2_64A
};
// n in 1..4 matrices sharing x (rows of each written to its y).
int gemv_dense_launch(const GemvMatArg* mats, int n, const void* x, int xt, int in, cudaStream_t stream,
                      const GemvExtras& ex = GemvExtras{});
// h = silu(gate x) * (up x)
int gemv_pair_launch(const GemvMatArg& gate, const GemvMatArg& up, const void* x, int xt, int in, float* h,
                     cudaStream_t stream, const GemvExtras& ex = GemvExtras{});
// out[i] = base[i] + sigmoid(*gate) * value[i] (+ resid[i] when set)  (moe.cu)
int sigmoid_fma_launch(const float* gate, const float* value, const float* base, const uint16_t* resid, float* out,
                       int n, cudaStream_t stream);
int gemv_tune(int ctas_per_sm);
int gemv_tune_split(int kcl);
int moe_gate_up_launch(const qg_int4_weight* gate, const qg_int4_weight* up, const uint32_t* idx, int k,
                       const uint16_t* x, float* h, cudaStream_t stream, int bits = 4);
int moe_gate_up_routed_launch(const float* logits, int n_logits, int renorm, const qg_int4_weight* gate,
                              const qg_int4_weight* up, int k, const uint16_t* x, float* h, uint32_t* idx_out,
                              float* p_out, cudaStream_t stream, int bits = 4);
// Copy `bytes` (a multiple of 16) from device-mapped host memory to device memory, in the launch
// chain (gemv_dense.cu).
int ingest_launch(const void* src_dev_mapped, void* dst, size_t bytes, cudaStream_t stream);
// Gated RMSNorm per head of head_dim elements (gemv_dense.cu): x = silu(z) * gamma * rmsnorm_head(y), fp32.
int gated_norm_launch(const void* y, const void* z, int xt, const uint16_t* gamma, int n, int head_dim, float eps,
                      float* x, cudaStream_t stream);
// Affine group-64 encode (quant.cu): bits 4 or 2, w bf16 or fp32 [out][in].
int quant_launch(const void* w, int wt, int out, int in, int bits, uint32_t* packed, uint16_t* scales,
                 uint16_t* biases, cudaStream_t stream);
int moe_down_launch(const qg_int4_weight* down, const uint32_t* idx, const float* p, int k, const float* h,
                    const uint16_t* residual, float* y, cudaStream_t stream, int bits = 4);

// ---------------------------------------------------------------- MoE (moe.cu)
int router_batch_launch(const float* logits, int T, int n_experts, int k, int renorm, uint32_t* idx, float* p,
                        cudaStream_t stream);
// Grouped (MoE prefill) tensor-core pieces (qgemm_tc.cu): token tiles of grouped rows (token t's X
// row, converted once, into rows rowpos[t k + s] for its k slots; or the SwiGLU of the grouped
// gate/up outputs, pair i into row rowpos[i]), and the GEMM over expert stacks whose token tile y
// belongs to expert tile_expert[y] (< 0: none).
int qgemm_prep_pairs_launch(const uint16_t* X, int T, int in, const int* rowpos, int npairs, int k, int n_tile,
                            uint8_t* xt, float* xs, cudaStream_t stream);
int qgemm_prep_swiglu_launch(const float* G, const float* U, int in, const int* rowpos, int npairs, int n_tile,
                             uint8_t* xt, float* xs, cudaStream_t stream);
int qgemm_tc_grouped_launch(const qg_int4_weight* w, int n, const uint8_t* xt, const float* xs, int n_tiles,
                            int n_tile, const int* tile_expert, float* const* Y, cudaStream_t stream);
// MoE prefill (moe_prefill.cu)
size_t moe_prefill_workspace_bytes(const qg_int4_weight* down, int T);
int moe_prefill_launch(const float* logits, int T, int renorm, const qg_int4_weight* gate, const qg_int4_weight* up,
                       const qg_int4_weight* down, int k, const uint16_t* X, const uint16_t* residual, float* Y,
                       uint32_t* idx, float* p, void* ws, size_t ws_bytes, cudaStream_t stream);
int router_launch(const float* logits, int n_experts, int k, int renorm, uint32_t* idx, float* p,
                  cudaStream_t stream);
int chain8_launch(const float* p, const float* v, const uint16_t* residual, float* out, int n, cudaStream_t stream);

// ---------------------------------------------------------------- GEMM (qgemm.cu)
size_t qgemm_workspace_bytes(const qg_int4_weight* w, int T);
int qgemm_launch(const qg_int4_weight* w, const uint16_t* X, int T, float* Y, void* ws, size_t ws_bytes,
                 cudaStream_t stream);
int qgemm_tune(int tc_min_T);
// tensor-core path (qgemm_tc.cu)
size_t qgemm_tc_workspace_bytes(const qg_int4_weight* w, int T);
int qgemm_tc_launch(const qg_int4_weight* w, const uint16_t* X, int T, float* Y, void* ws, size_t ws_bytes,
                    cudaStream_t stream);
// n in 1..4 weights sharing X (same in): Y[i] = X W_i^T, one launch over all their row tiles.
int qgemm_tc_launch_multi(const qg_int4_weight* w, int n, const uint16_t* X, int T, float* const* Y, void* ws,
                          size_t ws_bytes, cudaStream_t stream);
int qgemm_multi_launch(const qg_int4_weight* w, int n, const uint16_t* X, int T, float* const* Y, void* ws,
                       size_t ws_bytes, cudaStream_t stream);

}  // namespace qg
