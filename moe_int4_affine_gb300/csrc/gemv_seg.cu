// gemv_seg.cu -- MoE down projection fused with the slot-weighted accumulate and the residual:
//   y[i] = residual[i] + sum_k p[k] * (W_down[idx[k]] h_k)[i]
// computed as one GEMV whose row i is the concatenation of the k selected experts' row i and whose
// input is the concatenation of p_k * h_k ([FFAI#14] commit "ffai_moe_down_swiglu_accum_int4_chain8").
#include "gemv_kernel.cuh"

namespace qg {

int moe_down_launch(const qg_int4_weight* down, const uint32_t* idx, const float* p, int k, const float* h,
                    const uint16_t* residual, float* y, cudaStream_t stream) {
  if (k < 1 || k > kMaxMats) return QG_EINVAL;
  GemvArgs a{};
  a.nmat = 1;
  a.mat[0].w[0] = WRef{down->packed, down->scales, down->biases, -1};
  a.mat[0].w[1] = a.mat[0].w[0];
  a.mat[0].y = y;
  a.mat[0].out = down->out;
  a.mat[0].row0 = 0;
  a.seg = WRef{down->packed, down->scales, down->biases, 0};
  a.nseg = k;
  a.x = h;
  a.xf32 = 1;
  a.idx = idx;
  a.p = p;
  a.resid = residual;
  a.n_experts = down->n_mat;
  a.slab_words = (long long)down->out * (down->in / 8);
  a.slab_groups = (long long)down->out * (down->in / 64);
  a.in = down->in;
  a.total_rows = down->out;
  return plan_and_launch<kSeg>(a, stream);
}

}  // namespace qg
