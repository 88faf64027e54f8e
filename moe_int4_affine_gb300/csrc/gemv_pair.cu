// gemv_pair.cu -- gate/up pairs reduced with SwiGLU, h = silu(W_g x) * (W_u x): a dense pair, or the
// k router-selected experts' gate/up slabs of stacked weights ([FFAI#14] "dequantGemvInt4Two --
// per-expert MoE gate + up projections", commit "moeRouterTopK / dequantGemvInt4ExpertIndexed";
// SwiGLU unclamped as in [ds4#844]).
#include "gemv_kernel.cuh"

namespace qg {

int gemv_pair_launch(const GemvMatArg& gate, const GemvMatArg& up, const void* x, int xt, int in, float* h,
                     cudaStream_t stream) {
  GemvArgs a{};
  a.nmat = 1;
  a.mat[0].w[0] = WRef{gate.packed, gate.scales, gate.biases, -1};
  a.mat[0].w[1] = WRef{up.packed, up.scales, up.biases, -1};
  a.mat[0].y = h;
  a.mat[0].out = gate.out;
  a.mat[0].row0 = 0;
  a.nseg = 1;
  a.x = x;
  a.xf32 = xt == QG_X_F32;
  a.in = in;
  a.total_rows = gate.out;
  return plan_and_launch<kPair>(a, stream);
}

int moe_gate_up_launch(const qg_int4_weight* gate, const qg_int4_weight* up, const uint32_t* idx, int k,
                       const uint16_t* x, float* h, cudaStream_t stream) {
  if (k < 1 || k > kMaxMats) return QG_EINVAL;
  GemvArgs a{};
  a.nmat = k;
  for (int m = 0; m < k; ++m) {
    a.mat[m].w[0] = WRef{gate->packed, gate->scales, gate->biases, m};
    a.mat[m].w[1] = WRef{up->packed, up->scales, up->biases, m};
    a.mat[m].y = h + (size_t)m * gate->out;
    a.mat[m].out = gate->out;
    a.mat[m].row0 = m * gate->out;
  }
  a.nseg = 1;
  a.x = x;
  a.xf32 = 0;
  a.idx = idx;
  a.n_experts = gate->n_mat;
  a.slab_words = (long long)gate->out * (gate->in / 8);
  a.slab_groups = (long long)gate->out * (gate->in / 64);
  a.in = gate->in;
  a.total_rows = k * gate->out;
  return plan_and_launch<kPair>(a, stream);
}

// The same with the router in the kernel: every CTA selects the top k of n_logits logits itself;
// CTA 0 writes the selection to idx_out / p_out for the down kernel.
int moe_gate_up_routed_launch(const float* logits, int n_logits, int renorm, const qg_int4_weight* gate,
                              const qg_int4_weight* up, int k, const uint16_t* x, float* h, uint32_t* idx_out,
                              float* p_out, cudaStream_t stream) {
  if (k < 1 || k > kMaxMats) return QG_EINVAL;
  GemvArgs a{};
  a.nmat = k;
  for (int m = 0; m < k; ++m) {
    a.mat[m].w[0] = WRef{gate->packed, gate->scales, gate->biases, m};
    a.mat[m].w[1] = WRef{up->packed, up->scales, up->biases, m};
    a.mat[m].y = h + (size_t)m * gate->out;
    a.mat[m].out = gate->out;
    a.mat[m].row0 = m * gate->out;
  }
  a.nseg = 1;
  a.x = x;
  a.xf32 = 0;
  a.logits = logits;
  a.n_logits = n_logits;
  a.renorm = renorm;
  a.idx_out = idx_out;
  a.p_out = p_out;
  a.n_experts = gate->n_mat;
  a.slab_words = (long long)gate->out * (gate->in / 8);
  a.slab_groups = (long long)gate->out * (gate->in / 64);
  a.in = gate->in;
  a.total_rows = k * gate->out;
  return plan_and_launch<kPair>(a, stream);
}

}  // namespace qg
