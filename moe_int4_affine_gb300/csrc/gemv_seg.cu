// gemv_seg.cu -- MoE down projection fused with the slot-weighted accumulate and the residual:
//   y[i] = residual[i] + sum_k p[k] * (W_down[idx[k]] h_k)[i]
// computed as one GEMV whose row i is the concatenation of the k selected experts' row i and whose
// input is the concatenation of p_k * h_k ([FFAI#14] commit "ffai_moe_down_swiglu_accum_int4_chain8").
#include "gemv_kernel.cuh"

namespace qg {

int moe_down_launch(const qg_int4_weight* down, const uint32_t* idx, const float* p, int k, const float* h,
                    const uint16_t* residual, float* y, cudaStream_t stream, int bits) {
  if (k < 1 || k > kMaxMats) return QG_EINVAL;
  GemvArgs a = moe_down_args(down, idx, p, k, h, residual, y, bits);
  return plan_and_launch<kSeg>(a, stream);
}

}  // namespace qg
