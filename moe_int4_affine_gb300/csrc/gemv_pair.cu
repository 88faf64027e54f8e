// gemv_pair.cu -- gate/up pairs reduced with SwiGLU, h = silu(W_g x) * (W_u x): a dense pair, or the
// k router-selected experts' gate/up slabs of stacked weights ([FFAI#14]: dequantGemvInt4Two
// serves the gate and up projections of each selected expert; commit moeRouterTopK /
// dequantGemvInt4ExpertIndexed; SwiGLU without a clamp, as in [ds4#844]).
#include "gemv_kernel.cuh"

namespace qg {

int gemv_pair_launch(const GemvMatArg& gate, const GemvMatArg& up, const void* x, int xt, int in, float* h,
                     cudaStream_t stream, const GemvExtras& ex) {
  GemvArgs a = pair_args(gate, up, x, xt, in, h);
  apply_extras(a, ex);
  return plan_and_launch<kPair>(a, stream);
}

int moe_gate_up_launch(const qg_int4_weight* gate, const qg_int4_weight* up, const uint32_t* idx, int k,
                       const uint16_t* x, float* h, cudaStream_t stream, int bits) {
  if (k < 1 || k > kMaxMats) return QG_EINVAL;
  GemvArgs a = moe_gate_up_args(gate, up, idx, k, x, h, bits);
  return plan_and_launch<kPair>(a, stream);
}

// The same with the router in the kernel: every CTA selects the top k of n_logits logits itself;
// CTA 0 writes the selection to idx_out / p_out for the down kernel.
int moe_gate_up_routed_launch(const float* logits, int n_logits, int renorm, const qg_int4_weight* gate,
                              const qg_int4_weight* up, int k, const uint16_t* x, float* h, uint32_t* idx_out,
                              float* p_out, cudaStream_t stream, int bits) {
  if (k < 1 || k > kMaxMats) return QG_EINVAL;
  GemvArgs a = moe_gate_up_args(gate, up, nullptr, k, x, h, bits);
  a.logits = logits;
  a.n_logits = n_logits;
  a.renorm = renorm;
  a.idx_out = idx_out;
  a.p_out = p_out;
  return plan_and_launch<kPairRouted>(a, stream);
}

}  // namespace qg
