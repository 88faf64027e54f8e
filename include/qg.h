/*
 * qg.h -- C ABI of libqg: int4 affine group-quantised dequant-GEMV / MoE-gather decode path for
 * NVIDIA GB300 (sm_103a).
 *
 * Sources for what each call computes (web pages without section numbers; each citation names
 * the page and the commit or paragraph):
 *   [FFAI#14]  thewafflehaus/FFAI pull request #14, "feat(everything-bagel): clean migration of
 *              PR #9 + #10 onto updated dev"
 *   [FFAI#9]   thewafflehaus/FFAI pull request #9, "Everything Bagel"
 *   [ds4#844]  antirez/ds4 pull request #844, "Ornith 1.5 + Qwen 3.8 27B hybrid runtime + DFlash
 *              speculative decoding on Metal"
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers, owned by the caller, 16-byte aligned.  The library
 *     never allocates, frees or retains them.  Scratch space, where a call needs it, is a
 *     caller-owned device workspace whose size qg_workspace_bytes() reports ([FFAI#14], two-pass
 *     decode attention commit: the caller owns the scratch, so a decode loop reuses it across steps).
 *   - bf16 values are passed as their raw 16-bit patterns (uint16_t).
 *   - `stream` is a cudaStream_t cast to void* (NULL = the legacy default stream).  Every call is
 *     asynchronous on that stream; none synchronises the host except qg_device_status().
 *   - Return value: QG_OK (0) or a negative qg_error.  Argument errors are detected on the host
 *     before anything is launched.  Conditions only the device can see (an expert index out of
 *     range, a wait that timed out) set bits in a device status word read by qg_device_status().
 *   - Outputs of calls in flight must not alias inputs or outputs of other calls in flight.
 *
 * Weight format ([FFAI#14], commit moeRouterTopK / dequantGemvInt4ExpertIndexed: expert weights
 * stacked as u32 words [experts][out][in/8]; the GEMV operands there are the packed weight, its
 * scales and biases, the input and the output; every fast path there requires groups of 64;
 * [ds4#844], Q4_64A: one bf16 scale and one bf16 bias per group):
 *   packed  uint32 [n_mat][out][in/8]; element j of a row is the nibble at bits 4*(j%8) of word
 *           j/8 (low nibble first), an unsigned code q in 0..15.
 *   scales  bf16   [n_mat][out][in/64]
 *   biases  bf16   [n_mat][out][in/64]
 *   w[r][j] = scales[r][j/64] * q[r][j] + biases[r][j/64]       (no zero-point subtraction)
 *
 * Accuracy: every fp32 output y satisfies |y - y_exact| <= 1e-3 * sum|w*x| + 1e-6, where y_exact
 * and sum|w*x| are computed from the same stored inputs in exact arithmetic (checked against an
 * fp64 oracle); router indices and nibble decoding are exact.
 */
#ifndef QG_H
#define QG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QG_OK = 0,
  QG_EINVAL = -1,      /* null pointer, bad shape, group_size != 64, bad n/k/T, mismatched widths */
  QG_EALIGN = -2,      /* a pointer is not 16-byte aligned                                        */
  QG_EWORKSPACE = -3,  /* workspace missing or smaller than qg_workspace_bytes()                  */
  QG_ELAUNCH = -4,     /* the CUDA launch failed (cudaGetLastError after the launch)              */
  QG_ENOTSUP = -5,     /* shape outside the limits stated for the call                            */
  QG_EDEVICE = -6      /* a CUDA runtime call made by qg_device_status() failed                   */
} qg_error;

/* Bits of the device status word (qg_device_status). */
enum qg_status_bits {
  QG_STATUS_BAD_EXPERT = 1u, /* an expert index >= n_experts was skipped (its slot added nothing) */
  QG_STATUS_TIMEOUT = 2u     /* a device-side wait gave up after its time limit (result invalid)  */
};

typedef enum { QG_X_BF16 = 0, QG_X_F32 = 1 } qg_xtype;
typedef enum { QG_EPI_NONE = 0, QG_EPI_SWIGLU = 1 } qg_epilogue;

typedef struct {
  const uint32_t *packed; /* [n_mat][out][in/8] */
  const uint16_t *scales; /* bf16 [n_mat][out][in/group_size] */
  const uint16_t *biases; /* bf16 [n_mat][out][in/group_size] */
  int32_t out;            /* rows per matrix, >= 1 */
  int32_t in;             /* columns, a multiple of 64 */
  int32_t group_size;     /* must be 64 */
  int32_t n_mat;          /* 1, or the number of stacked experts */
} qg_int4_weight;

/*
 * qgemv_int4 -- dequant-GEMV, M = 1 ([FFAI#14] "dequant_gemv_int4_*"):
 *   y[r] = sum_j w[r][j] * x[j],  0 <= r < w->out  (fp32 accumulate).
 * x: [w->in], bf16 bits (xt = QG_X_BF16) or fp32 (QG_X_F32).  y: fp32 [w->out].
 * w->n_mat must be 1.  Limits: 64 <= in <= 32768, in % 64 == 0, out >= 1.
 */
int qgemv_int4(const qg_int4_weight *w, const void *x, int xt, float *y, void *stream);

/*
 * qgemv_int4_multi -- n in {2,3,4} projections sharing one input vector, one launch ([FFAI#14]
 * dequantGemvInt4Two/Three/Four, ffai_batched_qkv_qgemv_fast, ffai_batched_4_qgemv_fast: x is
 * read once for all projections, and the projections must all have the same packed width).
 *   epi = QG_EPI_NONE:   ys[i][r] = sum_j w_i[r][j] x[j]   for each i < n.
 *   epi = QG_EPI_SWIGLU: n must be 2 with ws[0].out == ws[1].out; ws[0] = gate, ws[1] = up and
 *                        ys[0][r] = silu(g[r]) * u[r], silu(g) = g / (1 + exp(-g)) (unclamped,
 *                        [ds4#844]: no clamp); ys[1] is unused (may be NULL).
 * ws: host array of n weights, all with the same `in`, n_mat == 1.  ys: host array of n device
 * pointers.  Limits as qgemv_int4.
 */
int qgemv_int4_multi(int n, const qg_int4_weight *ws, const void *x, int xt, float *const *ys, int epi,
                     void *stream);

/*
 * qgemv_q2, qgemv_q2_multi -- the 2-bit affine variant (Q2_64A, [ds4#844]) of qgemv_int4 and
 * qgemv_int4_multi: w[r][j] = s * q + b with 2-bit codes q in 0..3, sixteen per u32 (element
 * 16k + i at bits 2i of word k: `packed` is [out][in / 16]); scales and biases bf16 [out][in / 64]
 * as for 4 bits (the qg_int4_weight struct carries them unchanged).  quantize_affine_q64a with
 * bits = 2 writes this layout.  Arguments, epilogues and limits otherwise as the 4-bit calls.
 */
int qgemv_q2(const qg_int4_weight *w, const void *x, int x_type, float *y, void *stream);
int qgemv_q2_multi(int n, const qg_int4_weight *ws, const void *x, int x_type, float *const *ys, int epi,
                   void *stream);

/*
 * moe_gather_qgemv_q2, moe_layer_q2 -- moe_gather_qgemv_int4 and moe_layer_int4 for 2-bit experts
 * (Q2_64A layout as qgemv_q2: stacked gate/up packed [n_mat][inter][hidden / 16], down
 * [n_mat][hidden][inter / 16]; scales and biases as for 4 bits).  Arguments, workspace
 * (qg_workspace_bytes(QG_OP_MOE, down, k)), results and limits as the 4-bit calls.
 */
int moe_gather_qgemv_q2(const qg_int4_weight *gate, const qg_int4_weight *up, const qg_int4_weight *down,
                        const uint32_t *idx, const float *p, int k, const uint16_t *x, const uint16_t *residual,
                        float *y, void *workspace, size_t ws_bytes, void *stream);
int moe_layer_q2(const float *logits, int renorm, const qg_int4_weight *gate, const qg_int4_weight *up,
                 const qg_int4_weight *down, int k, const uint16_t *x, const uint16_t *residual, float *y,
                 uint32_t *idx, float *p, void *workspace, size_t ws_bytes, void *stream);

/*
 * rmsnorm_qgemv_int4 -- RMSNorm fused into the GEMV prologue ([FFAI#14], the commit that wraps
 * ffai_rms_norm_qgemv_fast: the normalised activation feeds the int4 dequant-GEMV directly, and
 * the normalised vector is never written to memory):
 *   y[r] = sum_j w[r][j] * x[j] * gamma[j] / sqrt( (1/in) sum_i x[i]^2 + eps )
 * (the page names the norm without writing it out; this is the usual RMSNorm with an epsilon
 * inside the root).  x: bf16 or fp32 [in]; gamma: bf16 [in] (device, 16-byte aligned); eps >= 0.
 * Every CTA reads x anyway: it also sums x^2, quantizes x * gamma, and scales its outputs by the
 * root.  Other arguments and limits as qgemv_int4.  An all-zero x with eps = 0 gives non-finite y.
 */
int rmsnorm_qgemv_int4(const qg_int4_weight *w, const void *x, int x_type, const uint16_t *gamma, float eps, float *y,
                       void *stream);

/*
 * rmsnorm_qgemv_int4_multi -- the same prologue for n in {2, 3, 4} projections sharing x, with the
 * epilogues of qgemv_int4_multi (QG_EPI_SWIGLU: h = silu(W_g xn) * (W_u xn) for the FFN after a
 * norm).  Arguments and limits as qgemv_int4_multi plus gamma and eps as above.
 */
int rmsnorm_qgemv_int4_multi(int n, const qg_int4_weight *ws, const void *x, int x_type, const uint16_t *gamma,
                             float eps, float *const *ys, int epi, void *stream);

/*
 * qgemv_int4_sigmoid_fma -- the shared-expert step fused into its GEMV ([FFAI#14], scalar-FMA
 * commit: sigmoidScalarFMAResidual adds a sigmoid-gated value and the residual to a base in one
 * pass after the MoE; here the value is this GEMV's output):
 *   y[r] = base[r] + sigmoid(gate[0]) * sum_j w[r][j] x[j]  (+ residual[r] when not NULL)
 * gate: fp32 [1]; base: fp32 [out]; residual: bf16 [out] or NULL; y: fp32 [out] (may equal
 * base); all device, 16-byte aligned.  Other arguments as qgemv_int4.
 */
int qgemv_int4_sigmoid_fma(const qg_int4_weight *w, const void *x, int x_type, const float *gate, const float *base,
                           const uint16_t *residual, float *y, void *stream);

/*
 * sigmoid_scalar_fma_residual -- the same step on its own ([FFAI#14] sigmoidScalarFMAResidual;
 * with residual NULL, sigmoidScalarFMA):
 *   out[i] = base[i] + sigmoid(gate[0]) * value[i]  (+ residual[i])
 * gate: fp32 [1]; value, base, out: fp32 [n]; residual: bf16 [n] or NULL (all device). n >= 1.
 */
int sigmoid_scalar_fma_residual(const float *gate, const float *value, const float *base, const uint16_t *residual,
                                float *out, int n, void *stream);

/*
 * moe_router_topk -- GPU router ([FFAI#14], commit moeRouterTopK: the logits of all experts in,
 * k u32 indices and k weights out, nothing read back by the host; [FFAI#9], partial-sort commit:
 * larger logits first, equal logits by smaller index).
 * Selects the k largest logits, ties to the lower index; slot s holds the s-th selected expert.
 *   renorm = 1: p = softmax over the k selected logits (sums to 1).
 *   renorm = 0: p = softmax over all n_experts logits, read at the selected experts.
 * logits: fp32 [n_experts] (device, finite); idx: uint32 [k] (device); p: fp32 [k] (device).
 * Limits: 1 <= k <= 32, k <= n_experts <= 1024.
 */
int moe_router_topk(const float *logits, int n_experts, int k, int renorm, uint32_t *idx, float *p, void *stream);

/*
 * moe_gather_qgemv_int4 -- MoE top-K gather decode step ([FFAI#14], commits moeRouterTopK /
 * dequantGemvInt4ExpertIndexed and ffai_moe_down_swiglu_accum_int4_chain8):
 *   for slot k: e = idx[k]; g = Wg[e] x; u = Wu[e] x; h_k = silu(g) * u; d_k = Wd[e] h_k
 *   y[i] = residual[i] + sum_k p[k] * d_k[i]
 * gate, up: n_mat = n_experts stacked [inter][hidden] weights; down: n_experts stacked
 * [hidden][inter].  idx (uint32 [k]) and p (fp32 [k]) are device arrays, normally the outputs
 * of moe_router_topk.  An index >= n_experts is skipped (that slot adds nothing) and sets
 * QG_STATUS_BAD_EXPERT.  x, residual: bf16 [hidden]; y: fp32 [hidden].
 * workspace: device scratch of at least qg_workspace_bytes(QG_OP_MOE, down, k) bytes (holds the
 * fp32 SwiGLU activations h[k][inter]).
 * Limits: 1 <= k <= 8; inter and hidden multiples of 64, at most 32768.
 */
int moe_gather_qgemv_int4(const qg_int4_weight *gate, const qg_int4_weight *up, const qg_int4_weight *down,
                          const uint32_t *idx, const float *p, int k, const uint16_t *x, const uint16_t *residual,
                          float *y, void *workspace, size_t ws_bytes, void *stream);

/*
 * moe_layer_int4 -- the whole MoE decode step in two launches: moe_router_topk followed by
 * moe_gather_qgemv_int4, with the router computed inside the expert gate/up kernel (every CTA
 * selects the top k itself, so no separate router launch and no index round trip through global
 * memory before the expert weights are read).  Same results as the two calls.
 * logits: fp32 [gate->n_mat] (device, finite); renorm as in moe_router_topk.
 * idx (uint32 [k]) and p (fp32 [k]): device outputs, the router's selection (also read by the
 * down projection).  Other arguments, workspace and limits as moe_gather_qgemv_int4 (1 <= k <= 8),
 * and n_experts = gate->n_mat <= 1024.
 * (The pages run the router and the expert kernels as separate dispatches; this fusion is this
 * library's.)
 */
int moe_layer_int4(const float *logits, int renorm, const qg_int4_weight *gate, const qg_int4_weight *up,
                   const qg_int4_weight *down, int k, const uint16_t *x, const uint16_t *residual, float *y,
                   uint32_t *idx, float *p, void *workspace, size_t ws_bytes, void *stream);

/*
 * gated_rmsnorm_qgemv_int4 -- the gated RMSNorm before a projection ([FFAI#14]
 * gatedRmsNormQgemvInt4Fast: a Mamba2-style gated norm, silu(z) * w * rmsnorm(y), on the GDN
 * mixer's output ahead of its out-projection), per head of head_dim consecutive elements:
 *   x[j] = silu(z[j]) * gamma[j] * y[j] / sqrt(mean over j's head of y^2 + eps),   out = W x
 * head_dim = w->in normalises over the whole vector.  y, z: bf16 or fp32 [in] (x_type, both);
 * gamma: bf16 [in]; out: fp32 [w->out].  workspace: at least qg_workspace_bytes(QG_OP_GATED_NORM, w, 0)
 * bytes.  head_dim a multiple of 64: one launch, the norm in the GEMV's prologue (per-head roots
 * applied to each 64-column group's x factors); otherwise two (a norm kernel, one block per head,
 * writes x as fp32 into the workspace, then the GEMV).  Limits as qgemv_int4; head_dim >= 1
 * divides in; eps >= 0, finite.
 */
int gated_rmsnorm_qgemv_int4(const qg_int4_weight *w, const void *y, const void *z, int x_type,
                             const uint16_t *gamma, float eps, int head_dim, float *out, void *workspace,
                             size_t ws_bytes, void *stream);

/*
 * moe_prefill_int4 -- the MoE layer for T tokens at once (prefill; [FFAI#9] "moeGatherDequantGemmInt4",
 * "mt_moe_gather_qmm_int4": rows sorted by expert with CSR expert offsets, for prefill):
 *   for token t: (idx[t], p[t]) = moe_router_topk(logits[t], renorm);
 *     for slot s: e = idx[t][s]; h = silu(Wg[e] X[t]) * (Wu[e] X[t]); d_s = Wd[e] h
 *     Y[t][i] = residual[t][i] + sum_s p[t][s] d_s[i]            (slot order)
 * i.e. moe_layer_int4 applied to every token.  On the device the (token, slot) pairs are grouped by
 * expert (counts, tile offsets, a row map), every expert's weights are read once per tile of its
 * tokens, and the gate/up and down projections run on the tensor cores (fp16 operands, fp32
 * accumulation, the numerics of qgemm_int4), seven launches in all.
 * logits: fp32 [T][n_experts]; X: bf16 [T][hidden]; residual: bf16 [T][hidden] or NULL (zero);
 * Y: fp32 [T][hidden]; idx (uint32) and p (fp32): device outputs [T][k].  gate, up, down: expert
 * stacks as for moe_gather_qgemv_int4 (n_mat = n_experts).
 * workspace: at least qg_workspace_bytes(QG_OP_MOE_PREFILL, down, T) bytes.
 * Limits: 1 <= T <= 65535, 1 <= k <= 8, k <= n_experts <= 1024; hidden and inter multiples of 64,
 * hidden <= 32768; scales and biases within fp16's range (as qgemm_int4).
 */
int moe_prefill_int4(const float *logits, int T, int renorm, const qg_int4_weight *gate, const qg_int4_weight *up,
                     const qg_int4_weight *down, int k, const uint16_t *X, const uint16_t *residual, float *Y,
                     uint32_t *idx, float *p, void *workspace, size_t ws_bytes, void *stream);

/*
 * dense_layer_int4 -- a dense decode FFN layer in one call: the SwiGLU gate/up pair, then the down
 * projection ([FFAI#14] "dequantGemvInt4Two" for gate + up, then the down dequant-GEMV):
 *   h = silu(W_g x) * (W_u x),   y = W_down h
 * gate, up: out = inter, in = hidden; down: in = inter (any out); single matrices (n_mat = 1).
 * x: bf16 or fp32 [hidden] (x_type); y: fp32 [down->out] (device).
 * workspace: at least qg_workspace_bytes(QG_OP_LAYER, down, 0) bytes; holds h (fp32 [inter]),
 * readable after the call.  Two launches (the second programmatically dependent when qg_set_pdl is
 * on); results equal qgemv_int4_multi(SWIGLU) followed by qgemv_int4 on h.  Limits as qgemv_int4.
 */
int dense_layer_int4(const qg_int4_weight *gate, const qg_int4_weight *up, const qg_int4_weight *down,
                     const void *x, int x_type, float *y, void *workspace, size_t ws_bytes, void *stream);

/*
 * dense_layer_int4_host -- dense_layer_int4 with x and y in page-locked HOST memory (cudaHostAlloc
 * or cudaHostRegister; the GPU reaches it through the CPU-GPU link).  A one-block kernel copies x
 * into the workspace, then the two GEMV launches run, and the down projection writes y straight
 * into y_host: three launches in one dependent chain (with qg_set_pdl on), no DMA copies.  y_host
 * holds the result once the stream has passed the call (synchronise before reading it).
 * x_host: bf16 or fp32 [hidden]; y_host: fp32 [down->out]; both 16-byte aligned.  Returns
 * QG_EINVAL when either is not page-locked host memory with a device mapping.
 * workspace (device): at least qg_workspace_bytes(QG_OP_LAYER_HOST, down, hidden) bytes; h comes
 * first, as in dense_layer_int4.  Results equal dense_layer_int4 on device copies of x.
 */
int dense_layer_int4_host(const qg_int4_weight *gate, const qg_int4_weight *up, const qg_int4_weight *down,
                          const void *x_host, int x_type, float *y_host, void *workspace, size_t ws_bytes,
                          void *stream);

/*
 * moe_gather_qgemv_int4_noalloc -- the same computation, arguments and limits as
 * moe_gather_qgemv_int4, without a workspace argument.  The pages have no counterpart: this entry
 * point exists for callers that cannot hand over device scratch, such as a host runtime that owns
 * all device memory and allows no new allocation once it serves requests, or a decode loop that
 * cannot afford the device-wide synchronisation that allocating and freeing memory implies.
 *
 * The activations h[k][inter] go to a fixed array compiled into the library (one per device,
 * QG_NOALLOC_MOE_MAX_FLOATS fp32 values = 128 KB, kept until the process exits).  No call allocates
 * or frees device memory.  The first call on a device looks up that array's device address (with
 * the device current) and caches it: make it before any stream capture on that device.
 * Every element of h the call reads is written earlier in the same call, so nothing needs clearing.
 * Returns QG_ENOTSUP when k * down->in exceeds QG_NOALLOC_MOE_MAX_FLOATS (inter up to 4096 at
 * k = 8), QG_EDEVICE if the address lookup fails, otherwise what moe_gather_qgemv_int4 returns.
 * All calls on a device share the one array: two calls that may overlap in time (on different
 * streams, or from different host threads without ordering) race on it and give wrong results.
 */
#define QG_NOALLOC_MOE_MAX_FLOATS 32768
int moe_gather_qgemv_int4_noalloc(const qg_int4_weight *gate, const qg_int4_weight *up,
                                  const qg_int4_weight *down, const uint32_t *idx, const float *p, int k,
                                  const uint16_t *x, const uint16_t *residual, float *y, void *stream);

/*
 * scalar_fma_chain8_residual -- eight (scalar, vector) pairs accumulated in one pass with the
 * residual folded in ([FFAI#14], scalar-FMA commit: scalarFMAChain8 does the eight
 * scalar-times-vector accumulations of a top-8 MoE in one dispatch, each a base plus a device
 * scalar times a vector; the residual add after the MoE is fused into the same pass):
 *   out[i] = residual[i] + sum_{k<8} p[k] * v[k][i]
 * p: fp32 [8]; v: fp32 [8][n]; residual: bf16 [n]; out: fp32 [n] (all device).  n >= 1.
 */
int scalar_fma_chain8_residual(const float *p, const float *v, const uint16_t *residual, float *out, int n,
                               void *stream);

/*
 * qgemm_int4 -- dequant-GEMM for T >= 1 token rows ([FFAI#9], Ops.dequantGemmDynamicM: the
 * token count is rounded up to a multiple of 32 with zero rows for the MMA kernel and only the
 * first T output rows are kept):
 *   Y[t][r] = sum_j w[r][j] * X[t][j],  0 <= t < T.
 * X: bf16 [T][in]; Y: fp32 [T][out].  The caller passes exactly T rows; padding is internal and
 * only the T real rows are written.  w->n_mat must be 1.
 * T >= 3 (see qg_tune_qgemm) runs on the tensor cores (tcgen05): the weights are dequantized to
 * fp16 in tensor memory, each token row is scaled by a power of two into fp16's range, products
 * accumulate in fp32.  Error: a bf16 token element within 2^31 of its row's largest converts to
 * fp16 exactly; a weight rounds once to fp16 (relative 2^-11 when |w| >= 2^-14, else 2^-25
 * absolute); the tensor cores add 16 exact products per MMA and round the running fp32 sum once
 * per MMA (assumed: relative 2^-23 of the magnitudes involved; undocumented hardware behaviour,
 * checked by the tests at K = 5120, 17408 and 32768).  So |Y - Y_exact| <= (2^-11 + (K/16 + 1)
 * 2^-23) sum |w x| (+ the 2^-25 and out-of-range terms): 6.2e-4 at K = 17408 and 7.3e-4 at
 * K = 32768, inside the 1e-3 bound.  That path needs every scale and bias within fp16's normal
 * range (2^-14 <= |s|, |b| < 65504, or zero; typical models are far inside it).  T < 3 runs the
 * CUDA-core GEMV once per token row.
 * workspace: at least qg_workspace_bytes(QG_OP_QGEMM, w, T) bytes (0 means none is needed): the
 * tensor-core path stages the converted tokens there.  With in a multiple of 512 and T outside
 * 65..112 the weights are read by tensor-map copies (encoded on the host for each call through the
 * driver entry point the CUDA runtime provides); QG_ELAUNCH if that encoding fails.
 * Limits: 1 <= T <= 4096; in % 64 == 0, 64 <= in <= 32768.
 */
int qgemm_int4(const qg_int4_weight *w, const uint16_t *X, int T, float *Y, void *workspace, size_t ws_bytes,
               void *stream);

/*
 * qgemm_int4_multi -- n in {2, 3, 4} projections of the same T tokens ([FFAI#14]
 * ffai_batched_qkv_qmm_fast / ffai_batched_4_qmm_fast: the M > 1 prefill form of the fused
 * QKV / GDN-input projections, x read once for all of them):
 *   Ys[i][t][r] = sum_j w_i[r][j] * X[t][j]
 * ws[i]: single matrices with the same in; X: bf16 [T][in]; Ys[i]: fp32 [T][ws[i].out] (device).
 * For T >= 3 (see qg_tune_qgemm) one tensor-core launch covers the row tiles of all n matrices
 * (the tokens staged once); below that, one GEMV launch per token covers all n.  workspace: at least
 * qg_workspace_bytes(QG_OP_QGEMM, &ws[0], T) bytes.  Limits as qgemm_int4.
 */
int qgemm_int4_multi(int n, const qg_int4_weight *ws, const uint16_t *X, int T, float *const *Ys, void *workspace,
                     size_t ws_bytes, void *stream);

/*
 * quantize_affine_q64a -- the affine group-64 encoder that makes this library's weights (Q4_64A,
 * bits = 4) and the 2-bit variant (Q2_64A, bits = 2) ([ds4#844]: "Q4_64A and Q2_64A codes are
 * derived from the serialized BF16 scale/bias").  Per row r and group g of 64 columns:
 *   lo = min, hi = max (-0 taken as +0);  s = bf16((hi - lo) / (2^bits - 1));  b = bf16(lo)
 *   q_j = clamp(rint((w_j - b) / s), 0, 2^bits - 1), 0 when s = 0
 * (bf16 rounding: nearest, ties to even; the code arithmetic in binary32 with correctly rounded
 * subtract and divide).  The pages give only the bf16 rule; the min/max affine form is the plain
 * reading.  w: bf16 or fp32 [out][in] (w_type QG_X_BF16 / QG_X_F32), finite; packed: u32
 * [out][in * bits / 32], low bits first (4 bits: element 8k + i at bits 4i of word k; 2 bits:
 * element 16k + i at bits 2i); scales, biases: bf16 [out][in / 64].  All device, 16-byte
 * aligned.  in % 64 == 0; out * in / 64 < 2^31 (QG_ENOTSUP beyond).  With bits = 4 the outputs
 * form a qg_int4_weight for every GEMV call.
 */
int quantize_affine_q64a(const void *w, int w_type, int out, int in, int bits, uint32_t *packed, uint16_t *scales,
                         uint16_t *biases, void *stream);

typedef enum {
  QG_OP_QGEMV = 0,
  QG_OP_MULTI = 1,
  QG_OP_MOE = 2,
  QG_OP_QGEMM = 3,
  QG_OP_LAYER = 4,     /* dense_layer_int4 */
  QG_OP_LAYER_HOST = 5, /* dense_layer_int4_host (T_or_k = hidden) */
  QG_OP_MOE_PREFILL = 6, /* moe_prefill_int4 (the down weight, T_or_k = T; room for any k <= 8) */
  QG_OP_GATED_NORM = 7   /* gated_rmsnorm_qgemv_int4 (T_or_k ignored) */
} qg_op;

/* Workspace bytes the call `op` needs for weight `w` and T (QG_OP_QGEMM) or k (QG_OP_MOE; pass
 * the down weight; QG_OP_LAYER: the down weight, T_or_k ignored).  Returns 0 when the call needs
 * none. */
size_t qg_workspace_bytes(int op, const qg_int4_weight *w, int T_or_k);

/*
 * qg_set_pdl -- enable (1) or disable (0, the default) programmatic dependent launch for the
 * kernels launched by this library in this process.  When enabled, a kernel may begin before
 * the preceding kernel in the stream has finished and streams its weights, scales and biases
 * into shared memory before waiting for it; activations, indices and outputs are only touched
 * after the wait.  Enable it only when no kernel immediately preceding a qg call writes that
 * call's weights (the normal case: weights are loaded once and reused every decode step).
 * Returns the previous setting.
 */
int qg_set_pdl(int enable);


/*
 * qg_tune_gemv -- CTAs per SM of the streaming GEMV kernels (1..4; 0 restores the default, 1), for
 * sweeps.  Process-wide, not thread-safe.  Returns QG_EINVAL outside that range.
 */
int qg_tune_gemv(int ctas_per_sm);

/*
 * qg_tune_gemv_split -- the GEMV planner's split of K across a thread-block cluster: 0 (default)
 * lets the planner choose per shape, 1 never splits, 2..4 splits K across clusters of that many CTAs
 * wherever a split is allowed (no norm prologue, at least one 32-group chunk of K per CTA).  The
 * CTAs of a cluster share one row range, each converts and streams its own slice of K, and their
 * row sums are added through distributed shared memory in rank order (deterministic).  Process-wide,
 * not thread-safe; for tests and sweeps.  Returns QG_EINVAL outside 0..4.  QG_DEBUG_PLAN=1 in the
 * environment prints each distinct shape's plan (grid, split, shared memory) once, on stderr.
 */
int qg_tune_gemv_split(int kcl);

/*
 * qg_tune_qgemm -- smallest T that qgemm_int4 runs on the tensor cores (1..4096; 0 restores the
 * default, 3); smaller T runs the CUDA-core GEMV once per token row.  Process-wide, not thread-safe;
 * query qg_workspace_bytes(QG_OP_QGEMM, ...) after changing it.  Returns QG_EINVAL outside that range.
 */
int qg_tune_qgemm(int tc_min_T);

/* Reads the device status word (qg_status_bits) of the current device into *status and clears
 * it.  Synchronises `stream`.  Returns QG_OK or QG_EDEVICE. */
int qg_device_status(void *stream, uint32_t *status);

/*
 * qg_selftest_wait_timeout -- exercises the device-side failure path: launches one kernel whose
 * single wait (on an mbarrier that nothing completes) gives up after limit_us microseconds
 * (1 .. 1000000), sets QG_STATUS_TIMEOUT in the device status word and returns normally.  The
 * context stays usable; qg_device_status() then reports (and clears) the bit.  Every wait in the
 * library's kernels ends the same way.  Returns QG_EINVAL outside the range, QG_ELAUNCH on a
 * launch error.  (No counterpart in the pages: a test hook for the status mechanism.)
 */
int qg_selftest_wait_timeout(int limit_us, void *stream);

/* Static description of an error code. */
const char *qg_strerror(int code);

/* Library version, (major << 16) | minor. */
int qg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QG_H */
