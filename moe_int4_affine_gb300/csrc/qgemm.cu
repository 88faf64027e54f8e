// qgemm.cu -- dequant-GEMM for T token rows ([FFAI#9] "Ops.dequantGemmDynamicM").
//   Y[t][r] = sum_j w[r][j] * X[t][j]
// CUDA-core path: one streaming GEMV pass per token row (the weights are re-read per row).
#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

size_t qgemm_workspace_bytes(const qg_int4_weight* w, int T) {
  (void)w;
  (void)T;
  return 0;
}

int qgemm_launch(const qg_int4_weight* w, const uint16_t* X, int T, float* Y, void* ws, size_t ws_bytes,
                 cudaStream_t stream) {
  (void)ws;
  (void)ws_bytes;
  for (int t = 0; t < T; ++t) {
    GemvMatArg m{w->packed, w->scales, w->biases, Y + (size_t)t * w->out, w->out};
    const int rc = gemv_dense_launch(&m, 1, X + (size_t)t * w->in, QG_X_BF16, w->in, stream);
    if (rc != QG_OK) return rc;
  }
  return QG_OK;
}

}  // namespace qg
