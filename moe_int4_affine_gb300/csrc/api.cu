// api.cu -- the C ABI (include/qg.h): argument validation, workspace sizing, status word, and
// dispatch to the kernel launchers.  No call allocates device memory.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

__device__ uint32_t g_status = 0;

namespace {
std::atomic<int> g_pdl{0};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round16(size_t n) { return (n + 15) & ~(size_t)15; }

// The device address of page-locked host memory, or null when `p` is not such memory.
void* mapped_host_pointer(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

int check_weight(const qg_int4_weight* w, bool stacked_ok) {
  if (!w || !w->packed || !w->scales || !w->biases) return QG_EINVAL;
  if (w->group_size != 64 || w->in < 64 || w->in % 64 != 0 || w->out < 1 || w->n_mat < 1) return QG_EINVAL;
  if (!stacked_ok && w->n_mat != 1) return QG_EINVAL;
  if (w->in > 32768) return QG_ENOTSUP;
  if (!aligned16(w->packed) || !aligned16(w->scales) || !aligned16(w->biases)) return QG_EALIGN;
  return QG_OK;
}
// Validation and dispatch shared by the multi-projection calls (ex: prologue / epilogue / bits).
int multi_call(int n, const qg_int4_weight* ws, const void* x, int xt, float* const* ys, int epi,
               const GemvExtras& ex, cudaStream_t s) {
  if (n < 2 || n > 4 || !ws || !ys || !x) return QG_EINVAL;
  if (xt != QG_X_BF16 && xt != QG_X_F32) return QG_EINVAL;
  if (epi != QG_EPI_NONE && epi != QG_EPI_SWIGLU) return QG_EINVAL;
  if (epi == QG_EPI_SWIGLU && (n != 2 || ws[0].out != ws[1].out)) return QG_EINVAL;
  GemvMatArg m[4];
  for (int i = 0; i < n; ++i) {
    int rc = check_weight(&ws[i], false);
    if (rc) return rc;
    if (ws[i].in != ws[0].in) return QG_EINVAL;  // all packed widths must match
    const bool need_y = !(epi == QG_EPI_SWIGLU && i == 1);
    if (need_y && !ys[i]) return QG_EINVAL;
    if (need_y && !aligned16(ys[i])) return QG_EALIGN;
    m[i] = GemvMatArg{ws[i].packed, ws[i].scales, ws[i].biases, need_y ? ys[i] : nullptr, ws[i].out};
  }
  if (!aligned16(x)) return QG_EALIGN;
  if (epi == QG_EPI_SWIGLU) return gemv_pair_launch(m[0], m[1], x, xt, ws[0].in, ys[0], s, ex);
  return gemv_dense_launch(m, n, x, xt, ws[0].in, s, ex);
}
}  // namespace

const DeviceInfo& device_info() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  std::call_once(g_dev_once[dev], [dev]() {
    DeviceInfo d{};
    cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (d.num_sms <= 0) d.num_sms = 1;
    d.id = dev;
    g_dev[dev] = d;
  });
  return g_dev[dev];
}

bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }

}  // namespace qg

using namespace qg;

extern "C" {

int qgemv_int4(const qg_int4_weight* w, const void* x, int xt, float* y, void* stream) {
  int rc = check_weight(w, false);
  if (rc) return rc;
  if (!x || !y || (xt != QG_X_BF16 && xt != QG_X_F32)) return QG_EINVAL;
  if (!aligned16(x) || !aligned16(y)) return QG_EALIGN;
  GemvMatArg m{w->packed, w->scales, w->biases, y, w->out};
  return gemv_dense_launch(&m, 1, x, xt, w->in, static_cast<cudaStream_t>(stream));
}

int qgemv_int4_multi(int n, const qg_int4_weight* ws, const void* x, int xt, float* const* ys, int epi, void* stream) {
  return multi_call(n, ws, x, xt, ys, epi, GemvExtras{}, static_cast<cudaStream_t>(stream));
}

int qgemv_q2(const qg_int4_weight* w, const void* x, int xt, float* y, void* stream) {
  int rc = check_weight(w, false);
  if (rc) return rc;
  if (!x || !y || (xt != QG_X_BF16 && xt != QG_X_F32)) return QG_EINVAL;
  if (!aligned16(x) || !aligned16(y)) return QG_EALIGN;
  GemvMatArg m{w->packed, w->scales, w->biases, y, w->out};
  GemvExtras ex{};
  ex.bits = 2;
  return gemv_dense_launch(&m, 1, x, xt, w->in, static_cast<cudaStream_t>(stream), ex);
}

int qgemv_q2_multi(int n, const qg_int4_weight* ws, const void* x, int xt, float* const* ys, int epi, void* stream) {
  GemvExtras ex{};
  ex.bits = 2;
  return multi_call(n, ws, x, xt, ys, epi, ex, static_cast<cudaStream_t>(stream));
}

int rmsnorm_qgemv_int4(const qg_int4_weight* w, const void* x, int xt, const uint16_t* gamma, float eps, float* y,
                       void* stream) {
  int rc = check_weight(w, false);
  if (rc) return rc;
  if (!x || !gamma || !y || (xt != QG_X_BF16 && xt != QG_X_F32) || !(eps >= 0.f)) return QG_EINVAL;
  if (!aligned16(x) || !aligned16(gamma) || !aligned16(y)) return QG_EALIGN;
  GemvMatArg m{w->packed, w->scales, w->biases, y, w->out};
  GemvExtras ex{};
  ex.gamma = gamma;
  ex.eps = eps;
  return gemv_dense_launch(&m, 1, x, xt, w->in, static_cast<cudaStream_t>(stream), ex);
}

int gated_rmsnorm_qgemv_int4(const qg_int4_weight* w, const void* y, const void* z, int xt, const uint16_t* gamma,
                             float eps, int head_dim, float* out, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_weight(w, false);
  if (rc) return rc;
  if (!y || !z || !gamma || !out || (xt != QG_X_BF16 && xt != QG_X_F32) || !(eps >= 0.f) || !(eps < INFINITY))
    return QG_EINVAL;
  if (head_dim < 1 || w->in % head_dim != 0) return QG_EINVAL;
  if (!aligned16(y) || !aligned16(z) || !aligned16(gamma) || !aligned16(out)) return QG_EALIGN;
  const size_t need = qg_workspace_bytes(QG_OP_GATED_NORM, w, 0);
  if (!workspace || ws_bytes < need) return QG_EWORKSPACE;
  if (!aligned16(workspace)) return QG_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GemvMatArg m{w->packed, w->scales, w->biases, out, w->out};
  if (head_dim % 64 == 0) {  // heads of whole groups: the norm inside the GEMV's prologue, one launch
    GemvExtras ex{};
    ex.gamma = gamma;
    ex.eps = eps;
    ex.gz = z;
    ex.head_dim = head_dim;
    return gemv_dense_launch(&m, 1, y, xt, w->in, s, ex);
  }
  float* x = static_cast<float*>(workspace);  // otherwise: the norm kernel, then the GEMV of its x
  rc = gated_norm_launch(y, z, xt, gamma, w->in, head_dim, eps, x, s);
  if (rc) return rc;
  return gemv_dense_launch(&m, 1, x, QG_X_F32, w->in, s);
}

int rmsnorm_qgemv_int4_multi(int n, const qg_int4_weight* ws, const void* x, int xt, const uint16_t* gamma, float eps,
                             float* const* ys, int epi, void* stream) {
  if (!gamma || !(eps >= 0.f)) return QG_EINVAL;
  if (!aligned16(gamma)) return QG_EALIGN;
  GemvExtras ex{};
  ex.gamma = gamma;
  ex.eps = eps;
  return multi_call(n, ws, x, xt, ys, epi, ex, static_cast<cudaStream_t>(stream));
}

int qgemv_int4_sigmoid_fma(const qg_int4_weight* w, const void* x, int xt, const float* gate, const float* base,
                           const uint16_t* residual, float* y, void* stream) {
  int rc = check_weight(w, false);
  if (rc) return rc;
  if (!x || !gate || !base || !y || (xt != QG_X_BF16 && xt != QG_X_F32)) return QG_EINVAL;
  if (!aligned16(x) || !aligned16(base) || !aligned16(y) || (residual && !aligned16(residual))) return QG_EALIGN;
  GemvMatArg m{w->packed, w->scales, w->biases, y, w->out};
  GemvExtras ex{};
  ex.sgate = gate;
  ex.ebase = base;
  ex.resid = residual;
  return gemv_dense_launch(&m, 1, x, xt, w->in, static_cast<cudaStream_t>(stream), ex);
}

int sigmoid_scalar_fma_residual(const float* gate, const float* value, const float* base, const uint16_t* residual,
                                float* out, int n, void* stream) {
  if (!gate || !value || !base || !out || n < 1) return QG_EINVAL;
  if (!aligned16(value) || !aligned16(base) || !aligned16(out) || (residual && !aligned16(residual))) return QG_EALIGN;
  return sigmoid_fma_launch(gate, value, base, residual, out, n, static_cast<cudaStream_t>(stream));
}

int moe_router_topk(const float* logits, int n_experts, int k, int renorm, uint32_t* idx, float* p, void* stream) {
  if (!logits || !idx || !p) return QG_EINVAL;
  if (k < 1 || k > 32 || n_experts < k || (renorm != 0 && renorm != 1)) return QG_EINVAL;
  if (n_experts > 1024) return QG_ENOTSUP;
  if (!aligned16(logits) || !aligned16(idx) || !aligned16(p)) return QG_EALIGN;
  return router_launch(logits, n_experts, k, renorm, idx, p, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {
// The MoE calls for both code widths (bits 4: Q4_64A, 2: Q2_64A).
int moe_gather_call(const qg_int4_weight* gate, const qg_int4_weight* up, const qg_int4_weight* down,
                    const uint32_t* idx, const float* p, int k, const uint16_t* x, const uint16_t* residual, float* y,
                    void* workspace, size_t ws_bytes, void* stream, int bits) {
  int rc;
  if ((rc = check_weight(gate, true)) || (rc = check_weight(up, true)) || (rc = check_weight(down, true))) return rc;
  if (!idx || !p || !x || !residual || !y) return QG_EINVAL;
  if (k < 1 || k > 8) return QG_EINVAL;
  if (gate->out != up->out || gate->in != up->in || gate->n_mat != up->n_mat || down->n_mat != gate->n_mat ||
      down->in != gate->out || down->out != gate->in)
    return QG_EINVAL;
  if (!aligned16(idx) || !aligned16(p) || !aligned16(x) || !aligned16(residual) || !aligned16(y)) return QG_EALIGN;
  const size_t need = qg_workspace_bytes(QG_OP_MOE, down, k);
  if (!workspace || ws_bytes < need) return QG_EWORKSPACE;
  if (!aligned16(workspace)) return QG_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* h = static_cast<float*>(workspace);
  rc = moe_gate_up_launch(gate, up, idx, k, x, h, s, bits);
  if (rc) return rc;
  return moe_down_launch(down, idx, p, k, h, residual, y, s, bits);
}

int moe_layer_call(const float* logits, int renorm, const qg_int4_weight* gate, const qg_int4_weight* up,
                   const qg_int4_weight* down, int k, const uint16_t* x, const uint16_t* residual, float* y,
                   uint32_t* idx, float* p, void* workspace, size_t ws_bytes, void* stream, int bits) {
  int rc;
  if ((rc = check_weight(gate, true)) || (rc = check_weight(up, true)) || (rc = check_weight(down, true))) return rc;
  if (!logits || !idx || !p || !x || !residual || !y) return QG_EINVAL;
  if (k < 1 || k > 8 || (renorm != 0 && renorm != 1) || gate->n_mat < k) return QG_EINVAL;
  if (gate->n_mat > 1024) return QG_ENOTSUP;
  if (gate->out != up->out || gate->in != up->in || gate->n_mat != up->n_mat || down->n_mat != gate->n_mat ||
      down->in != gate->out || down->out != gate->in)
    return QG_EINVAL;
  if (!aligned16(logits) || !aligned16(idx) || !aligned16(p) || !aligned16(x) || !aligned16(residual) ||
      !aligned16(y))
    return QG_EALIGN;
  const size_t need = qg_workspace_bytes(QG_OP_MOE, down, k);
  if (!workspace || ws_bytes < need) return QG_EWORKSPACE;
  if (!aligned16(workspace)) return QG_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* h = static_cast<float*>(workspace);
  rc = moe_gate_up_routed_launch(logits, gate->n_mat, renorm, gate, up, k, x, h, idx, p, s, bits);
  if (rc) return rc;
  return moe_down_launch(down, idx, p, k, h, residual, y, s, bits);
}
}  // namespace

extern "C" {

int moe_gather_qgemv_int4(const qg_int4_weight* gate, const qg_int4_weight* up, const qg_int4_weight* down,
                          const uint32_t* idx, const float* p, int k, const uint16_t* x, const uint16_t* residual,
                          float* y, void* workspace, size_t ws_bytes, void* stream) {
  return moe_gather_call(gate, up, down, idx, p, k, x, residual, y, workspace, ws_bytes, stream, 4);
}

int moe_gather_qgemv_q2(const qg_int4_weight* gate, const qg_int4_weight* up, const qg_int4_weight* down,
                        const uint32_t* idx, const float* p, int k, const uint16_t* x, const uint16_t* residual,
                        float* y, void* workspace, size_t ws_bytes, void* stream) {
  return moe_gather_call(gate, up, down, idx, p, k, x, residual, y, workspace, ws_bytes, stream, 2);
}

int moe_layer_int4(const float* logits, int renorm, const qg_int4_weight* gate, const qg_int4_weight* up,
                   const qg_int4_weight* down, int k, const uint16_t* x, const uint16_t* residual, float* y,
                   uint32_t* idx, float* p, void* workspace, size_t ws_bytes, void* stream) {
  return moe_layer_call(logits, renorm, gate, up, down, k, x, residual, y, idx, p, workspace, ws_bytes, stream, 4);
}

int moe_layer_q2(const float* logits, int renorm, const qg_int4_weight* gate, const qg_int4_weight* up,
                 const qg_int4_weight* down, int k, const uint16_t* x, const uint16_t* residual, float* y,
                 uint32_t* idx, float* p, void* workspace, size_t ws_bytes, void* stream) {
  return moe_layer_call(logits, renorm, gate, up, down, k, x, residual, y, idx, p, workspace, ws_bytes, stream, 2);
}

int moe_prefill_int4(const float* logits, int T, int renorm, const qg_int4_weight* gate, const qg_int4_weight* up,
                     const qg_int4_weight* down, int k, const uint16_t* X, const uint16_t* residual, float* Y,
                     uint32_t* idx, float* p, void* workspace, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_weight(gate, true)) || (rc = check_weight(up, true)) || (rc = check_weight(down, true))) return rc;
  if (!logits || !idx || !p || !X || !Y) return QG_EINVAL;
  if (T < 1 || T > 65535 || k < 1 || k > 8 || (renorm != 0 && renorm != 1) || gate->n_mat < k) return QG_EINVAL;
  if (gate->n_mat > 1024) return QG_ENOTSUP;
  if (gate->out != up->out || gate->in != up->in || gate->n_mat != up->n_mat || down->n_mat != gate->n_mat ||
      down->in != gate->out || down->out != gate->in)
    return QG_EINVAL;
  if (!aligned16(logits) || !aligned16(idx) || !aligned16(p) || !aligned16(X) || (residual && !aligned16(residual)) ||
      !aligned16(Y))
    return QG_EALIGN;
  const size_t need = qg_workspace_bytes(QG_OP_MOE_PREFILL, down, T);
  if (!workspace || ws_bytes < need) return QG_EWORKSPACE;
  if (!aligned16(workspace)) return QG_EALIGN;
  return moe_prefill_launch(logits, T, renorm, gate, up, down, k, X, residual, Y, idx, p, workspace, ws_bytes,
                            static_cast<cudaStream_t>(stream));
}

int dense_layer_int4(const qg_int4_weight* gate, const qg_int4_weight* up, const qg_int4_weight* down, const void* x,
                     int xt, float* y, void* workspace, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_weight(gate, false)) || (rc = check_weight(up, false)) || (rc = check_weight(down, false)))
    return rc;
  if (!x || !y || (xt != QG_X_BF16 && xt != QG_X_F32)) return QG_EINVAL;
  if (gate->out != up->out || gate->in != up->in || down->in != gate->out) return QG_EINVAL;
  if (!aligned16(x) || !aligned16(y)) return QG_EALIGN;
  const size_t need = qg_workspace_bytes(QG_OP_LAYER, down, 0);
  if (!workspace || ws_bytes < need) return QG_EWORKSPACE;
  if (!aligned16(workspace)) return QG_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* h = static_cast<float*>(workspace);
  const GemvMatArg g{gate->packed, gate->scales, gate->biases, h, gate->out};
  const GemvMatArg u{up->packed, up->scales, up->biases, nullptr, up->out};
  const GemvMatArg d{down->packed, down->scales, down->biases, y, down->out};
  rc = gemv_pair_launch(g, u, x, xt, gate->in, h, s);
  if (rc) return rc;
  return gemv_dense_launch(&d, 1, h, QG_X_F32, down->in, s);
}

int dense_layer_int4_host(const qg_int4_weight* gate, const qg_int4_weight* up, const qg_int4_weight* down,
                          const void* x_host, int xt, float* y_host, void* workspace, size_t ws_bytes, void* stream) {
  int rc;
  if ((rc = check_weight(gate, false)) || (rc = check_weight(up, false)) || (rc = check_weight(down, false)))
    return rc;
  if (!x_host || !y_host || (xt != QG_X_BF16 && xt != QG_X_F32)) return QG_EINVAL;
  if (gate->out != up->out || gate->in != up->in || down->in != gate->out) return QG_EINVAL;
  void* xd = mapped_host_pointer(x_host);
  void* yd = mapped_host_pointer(y_host);
  if (!xd || !yd) return QG_EINVAL;
  if (!aligned16(x_host) || !aligned16(y_host) || !aligned16(xd) || !aligned16(yd)) return QG_EALIGN;
  const size_t need = qg_workspace_bytes(QG_OP_LAYER_HOST, down, gate->in);
  if (!workspace || ws_bytes < need) return QG_EWORKSPACE;
  if (!aligned16(workspace)) return QG_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* h = static_cast<float*>(workspace);
  void* x_dev = static_cast<uint8_t*>(workspace) + round16((size_t)down->in * sizeof(float));
  const size_t xbytes = (size_t)gate->in * (xt == QG_X_F32 ? 4 : 2);
  if ((rc = ingest_launch(xd, x_dev, xbytes, s))) return rc;
  const GemvMatArg g{gate->packed, gate->scales, gate->biases, h, gate->out};
  const GemvMatArg u{up->packed, up->scales, up->biases, nullptr, up->out};
  const GemvMatArg d{down->packed, down->scales, down->biases, static_cast<float*>(yd), down->out};
  if ((rc = gemv_pair_launch(g, u, x_dev, xt, gate->in, h, s))) return rc;
  return gemv_dense_launch(&d, 1, h, QG_X_F32, down->in, s);
}

int scalar_fma_chain8_residual(const float* p, const float* v, const uint16_t* residual, float* out, int n,
                               void* stream) {
  if (!p || !v || !residual || !out || n < 1) return QG_EINVAL;
  if (!aligned16(p) || !aligned16(v) || !aligned16(residual) || !aligned16(out)) return QG_EALIGN;
  return chain8_launch(p, v, residual, out, n, static_cast<cudaStream_t>(stream));
}

int qgemm_int4(const qg_int4_weight* w, const uint16_t* X, int T, float* Y, void* workspace, size_t ws_bytes,
               void* stream) {
  int rc = check_weight(w, false);
  if (rc) return rc;
  if (!X || !Y || T < 1 || T > 4096) return QG_EINVAL;
  if (!aligned16(X) || !aligned16(Y)) return QG_EALIGN;
  const size_t need = qgemm_workspace_bytes(w, T);
  if (need && (!workspace || ws_bytes < need)) return QG_EWORKSPACE;
  if (need && !aligned16(workspace)) return QG_EALIGN;
  return qgemm_launch(w, X, T, Y, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

int qgemm_int4_multi(int n, const qg_int4_weight* ws, const uint16_t* X, int T, float* const* Ys, void* workspace,
                     size_t ws_bytes, void* stream) {
  if (n < 2 || n > 4 || !ws || !Ys || !X || T < 1 || T > 4096) return QG_EINVAL;
  for (int i = 0; i < n; ++i) {
    int rc = check_weight(&ws[i], false);
    if (rc) return rc;
    if (ws[i].in != ws[0].in || !Ys[i]) return QG_EINVAL;
    if (!aligned16(Ys[i])) return QG_EALIGN;
  }
  if (!aligned16(X)) return QG_EALIGN;
  const size_t need = qgemm_workspace_bytes(&ws[0], T);
  if (need && (!workspace || ws_bytes < need)) return QG_EWORKSPACE;
  if (need && !aligned16(workspace)) return QG_EALIGN;
  return qgemm_multi_launch(ws, n, X, T, Ys, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

int quantize_affine_q64a(const void* w, int wt, int out, int in, int bits, uint32_t* packed, uint16_t* scales,
                         uint16_t* biases, void* stream) {
  if (!w || !packed || !scales || !biases || (wt != QG_X_BF16 && wt != QG_X_F32)) return QG_EINVAL;
  if ((bits != 4 && bits != 2) || out < 1 || in < 64 || in % 64 != 0) return QG_EINVAL;
  if (!aligned16(w) || !aligned16(packed) || !aligned16(scales) || !aligned16(biases)) return QG_EALIGN;
  return quant_launch(w, wt, out, in, bits, packed, scales, biases, static_cast<cudaStream_t>(stream));
}

size_t qg_workspace_bytes(int op, const qg_int4_weight* w, int T_or_k) {
  if (!w) return 0;
  switch (op) {
    case QG_OP_MOE:  // h[k][inter] fp32; inter = down->in
      return (size_t)(T_or_k > 0 ? T_or_k : 0) * (size_t)w->in * sizeof(float);
    case QG_OP_QGEMM:
      return qgemm_workspace_bytes(w, T_or_k);
    case QG_OP_LAYER:  // h[inter] fp32; inter = down->in
      return (size_t)w->in * sizeof(float);
    case QG_OP_LAYER_HOST:  // h[inter], then the device copy of x[hidden] (room for fp32)
      return round16((size_t)w->in * sizeof(float)) + (size_t)(T_or_k > 0 ? T_or_k : 0) * sizeof(float);
    case QG_OP_MOE_PREFILL:  // plan tables, grouped token tiles, G, U, h tiles, down outputs
      return moe_prefill_workspace_bytes(w, T_or_k);
    case QG_OP_GATED_NORM:  // the normalised, gated vector x (fp32 [in])
      return (size_t)w->in * sizeof(float);
    default:
      return 0;
  }
}

int qg_set_pdl(int enable) { return g_pdl.exchange(enable ? 1 : 0); }

int qg_tune_gemv(int ctas_per_sm) { return gemv_tune(ctas_per_sm); }

int qg_tune_gemv_split(int kcl) { return gemv_tune_split(kcl); }

int qg_tune_qgemm(int tc_min_T) { return qgemm_tune(tc_min_T); }

int qg_device_status(void* stream, uint32_t* status) {
  if (!status) return QG_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static const uint32_t zero = 0;
  if (cudaMemcpyFromSymbolAsync(status, g_status, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return QG_EDEVICE;
  if (cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return QG_EDEVICE;
  if (cudaStreamSynchronize(s) != cudaSuccess) return QG_EDEVICE;
  return QG_OK;
}

const char* qg_strerror(int code) {
  switch (code) {
    case QG_OK: return "ok";
    case QG_EINVAL: return "invalid argument";
    case QG_EALIGN: return "pointer not 16-byte aligned";
    case QG_EWORKSPACE: return "workspace missing or too small";
    case QG_ELAUNCH: return "CUDA launch failed";
    case QG_ENOTSUP: return "shape outside the supported limits";
    case QG_EDEVICE: return "CUDA runtime call failed";
    default: return "unknown error";
  }
}

int qg_version(void) { return (1 << 16) | 0; }

}  // extern "C"
