// qgemm.cu -- dequant-GEMM for T token rows ([FFAI#9] "Ops.dequantGemmDynamicM"):
//   Y[t][r] = sum_j w[r][j] * X[t][j]
// Dispatch: T >= the tensor-core threshold (3 unless tuned) runs the tcgen05 kernel of qgemm_tc.cu
// (the tokens padded to a multiple of 16 inside the kernel's tiles); smaller T runs the streaming
// CUDA-core GEMV once per token row.
#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

// The tensor-core path from this many tokens on: its one 16-token tile (30 us at 17408 x 5120)
// beats the per-token GEMV launches (about 12 us each) from T = 3 (measured on the GB300).
constexpr int kTcMinTDefault = 3;
static int g_tc_min_T = kTcMinTDefault;

int qgemm_tune(int tc_min_T) {
  if (tc_min_T < 0 || tc_min_T > 4096) return QG_EINVAL;
  g_tc_min_T = tc_min_T ? tc_min_T : kTcMinTDefault;
  return QG_OK;
}

size_t qgemm_workspace_bytes(const qg_int4_weight* w, int T) {
  return T >= g_tc_min_T ? qgemm_tc_workspace_bytes(w, T) : 0;
}

int qgemm_launch(const qg_int4_weight* w, const uint16_t* X, int T, float* Y, void* ws, size_t ws_bytes,
                 cudaStream_t stream) {
  if (T >= g_tc_min_T) return qgemm_tc_launch(w, X, T, Y, ws, ws_bytes, stream);
  for (int t = 0; t < T; ++t) {
    GemvMatArg m{w->packed, w->scales, w->biases, Y + (size_t)t * w->out, w->out};
    const int rc = gemv_dense_launch(&m, 1, X + (size_t)t * w->in, QG_X_BF16, w->in, stream);
    if (rc != QG_OK) return rc;
  }
  return QG_OK;
}

// Projections sharing X: one tensor-core launch over all row tiles, or per token one GEMV launch
// over all n matrices.
int qgemm_multi_launch(const qg_int4_weight* w, int n, const uint16_t* X, int T, float* const* Y, void* ws,
                       size_t ws_bytes, cudaStream_t stream) {
  if (n < 1 || n > 4) return QG_EINVAL;
  if (T >= g_tc_min_T) return qgemm_tc_launch_multi(w, n, X, T, Y, ws, ws_bytes, stream);
  for (int t = 0; t < T; ++t) {
    GemvMatArg m[4];
    for (int i = 0; i < n; ++i) m[i] = GemvMatArg{w[i].packed, w[i].scales, w[i].biases, Y[i] + (size_t)t * w[i].out, w[i].out};
    const int rc = gemv_dense_launch(m, n, X + (size_t)t * w[0].in, QG_X_BF16, w[0].in, stream);
    if (rc != QG_OK) return rc;
  }
  return QG_OK;
}

}  // namespace qg
