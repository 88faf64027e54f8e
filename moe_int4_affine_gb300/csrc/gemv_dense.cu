// gemv_dense.cu -- dense dequant-GEMV launches: one matrix, or n in {2,3,4} matrices sharing x
// ([FFAI#14] "dequant_gemv_int4_*", "dequantGemvInt4Two/Three/Four", "ffai_batched_4_qgemv_fast").
#include "gemv_kernel.cuh"

namespace qg {

GemvTune g_gemv_tune = {0};

int gemv_tune(int ctas_per_sm) {
  if (ctas_per_sm < 0 || ctas_per_sm > 4) return QG_EINVAL;
  g_gemv_tune = GemvTune{ctas_per_sm};
  return QG_OK;
}

int gemv_dense_launch(const GemvMatArg* mats, int n, const void* x, int xt, int in, cudaStream_t stream) {
  if (n < 1 || n > 4) return QG_EINVAL;
  GemvArgs a{};
  int rows = 0;
  a.nmat = n;
  for (int i = 0; i < n; ++i) {
    a.mat[i].w[0] = WRef{mats[i].packed, mats[i].scales, mats[i].biases, -1};
    a.mat[i].w[1] = a.mat[i].w[0];
    a.mat[i].y = mats[i].y;
    a.mat[i].out = mats[i].out;
    a.mat[i].row0 = rows;
    rows += mats[i].out;
  }
  a.nseg = 1;
  a.x = x;
  a.xf32 = xt == QG_X_F32;
  a.in = in;
  a.total_rows = rows;
  return plan_and_launch<kDense>(a, stream);
}

}  // namespace qg
