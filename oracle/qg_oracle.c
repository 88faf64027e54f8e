/*
 * qg_oracle.c -- plain fp64 CPU oracle for the int4 affine dequant-GEMV decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA library is compared with.
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load it.  It shares
 * no code, header, table or constant with the CUDA library (moe_int4_affine_gb300/csrc), and
 * neither side includes or links the other.
 *
 * Everything here is the plain definition, written out: decode the stored values exactly into
 * double, unpack each nibble, dequantise each weight on its own, multiply, and sum in index
 * order.  No blocking, no factoring of the group sum, no fusion.
 *
 * Sources (web pages; they carry no section numbers, so each citation names the page and the
 * commit or paragraph that states the fact):
 *   [FFAI#14]  thewafflehaus/FFAI pull request #14, "feat(everything-bagel): clean migration
 *              of PR #9 + #10 onto updated dev"
 *   [FFAI#9]   thewafflehaus/FFAI pull request #9, "Everything Bagel"
 *   [ds4#844]  antirez/ds4 pull request #844, "Ornith 1.5 + Qwen 3.8 27B hybrid runtime +
 *              DFlash speculative decoding on Metal"
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)

/* x / activation element types accepted by the oracle */
#define ORC_X_BF16 0
#define ORC_X_F32 1

/* ---------------------------------------------------------------------------------------
 * Stored-value decode.
 * bf16 is the upper 16 bits of an IEEE-754 binary32; widening to binary32 is exact, and
 * binary32 -> binary64 is exact.  Scales and biases are bf16 ([FFAI#9], loader commit: the
 * affine-quantized weights are u32-packed and their float type is taken from the scales;
 * [ds4#844], Q4_64A commit: bf16 scale and bias).
 * ------------------------------------------------------------------------------------- */
double orc_bf16_to_f64(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double load_x(const void *x, int xtype, int64_t j) {
  if (xtype == ORC_X_BF16) return orc_bf16_to_f64(((const uint16_t *)x)[j]);
  return (double)((const float *)x)[j];
}

/* ---------------------------------------------------------------------------------------
 * Nibble unpack.
 * Weight tensor is u32 words, [out][in/8] ([FFAI#14], commit moeRouterTopK /
 * dequantGemvInt4ExpertIndexed: experts stacked as u32 [experts][out][in/8]; [FFAI#14], the
 * batched-projection wrappers take the input width as eight times the packed width).  Within a word, element
 * 8*w + i sits in bits 4i..4i+3 (low nibble first).
 * ------------------------------------------------------------------------------------- */
unsigned orc_nibble(const uint32_t *packed, int64_t in, int64_t row, int64_t j) {
  uint32_t word = packed[row * (in / 8) + j / 8];
  return (unsigned)((word >> (4 * (j % 8))) & 0xFu);
}

void orc_unpack_rows(const uint32_t *packed, int64_t in, int64_t r0, int64_t r1, uint8_t *q) {
  for (int64_t r = r0; r < r1; ++r)
    for (int64_t j = 0; j < in; ++j) q[(r - r0) * in + j] = (uint8_t)orc_nibble(packed, in, r, j);
}

/* ---------------------------------------------------------------------------------------
 * Affine group dequantisation: w[r][j] = scale[r][j/gs] * q[r][j] + bias[r][j/gs].
 * Scales and biases are [out][in/gs] ([FFAI#14]: the GEMV operands are the packed weight, its
 * scales and biases, the input and the output; every fast path there requires groups of 64).  No
 * zero-point is subtracted: the bias carries the offset ([ds4#844], Q4_64A: a scale and a bias).
 * ------------------------------------------------------------------------------------- */
double orc_dequant(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases, int64_t in,
                   int64_t gs, int64_t row, int64_t j) {
  int64_t g = j / gs, ng = in / gs;
  double s = orc_bf16_to_f64(scales[row * ng + g]);
  double b = orc_bf16_to_f64(biases[row * ng + g]);
  return s * (double)orc_nibble(packed, in, row, j) + b;
}

/* ---------------------------------------------------------------------------------------
 * Dequant-GEMV, M = 1:  y[r] = sum_j w[r][j] * x[j]  for rows r0 <= r < r1, summed in j
 * order in double ([FFAI#14] dequant_gemv_int4_*; its tests check every wrapper against a
 * CPU reference built from the packed weights, scales and biases).
 * absref[r] = sum_j |w[r][j] * x[j]| is the scale of the acceptance bound.
 * y and absref are indexed r - r0.  absref may be NULL.
 * ------------------------------------------------------------------------------------- */
int orc_qgemv_rows(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases, int64_t out,
                   int64_t in, int64_t gs, const void *x, int xtype, int64_t r0, int64_t r1, double *y,
                   double *absref) {
  if (gs <= 0 || in <= 0 || in % gs != 0 || in % 8 != 0 || r0 < 0 || r1 > out || r0 > r1) return ORC_EINVAL;
  if (xtype != ORC_X_BF16 && xtype != ORC_X_F32) return ORC_EINVAL;
  for (int64_t r = r0; r < r1; ++r) {
    double acc = 0.0, aacc = 0.0;
    for (int64_t j = 0; j < in; ++j) {
      double t = orc_dequant(packed, scales, biases, in, gs, r, j) * load_x(x, xtype, j);
      acc += t;
      aacc += fabs(t);
    }
    y[r - r0] = acc;
    if (absref) absref[r - r0] = aacc;
  }
  return ORC_OK;
}

/* Same product with a double-precision input vector (used for the MoE down projection, whose
 * input h is kept in double by the oracle). */
int orc_qgemv_rows_f64x(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases, int64_t out,
                        int64_t in, int64_t gs, const double *x, int64_t r0, int64_t r1, double *y,
                        double *absref) {
  if (gs <= 0 || in <= 0 || in % gs != 0 || in % 8 != 0 || r0 < 0 || r1 > out || r0 > r1) return ORC_EINVAL;
  for (int64_t r = r0; r < r1; ++r) {
    double acc = 0.0, aacc = 0.0;
    for (int64_t j = 0; j < in; ++j) {
      double t = orc_dequant(packed, scales, biases, in, gs, r, j) * x[j];
      acc += t;
      aacc += fabs(t);
    }
    y[r - r0] = acc;
    if (absref) absref[r - r0] = aacc;
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------------------------
 * SwiGLU: h = silu(g) * u = g / (1 + exp(-g)) * u, unclamped ([FFAI#14], fused MoE down
 * commit: each slot's inner activation is silu of its gate times its up; [ds4#844]: no clamp).
 * ------------------------------------------------------------------------------------- */
double orc_silu(double g) { return g / (1.0 + exp(-g)); }

void orc_swiglu(const double *g, const double *u, int64_t n, double *h) {
  for (int64_t i = 0; i < n; ++i) h[i] = orc_silu(g[i]) * u[i];
}

/* ---------------------------------------------------------------------------------------
 * Router top-K ([FFAI#14], commit moeRouterTopK: the logits of all experts in, k u32 indices
 * and k weights out; its test takes logits (1, 5, 3, 4) with k = 2, expects experts 1 and 3 and
 * weights that add up to one; [FFAI#9], partial-sort commit: larger value first, ties by index).
 * Selection: k rounds of "take the not-yet-taken expert with the largest logit; on equal
 * logits the smaller index".  Weights: renorm=1 -> softmax over the k selected logits
 * (sums to 1); renorm=0 -> the full softmax over all n experts, read at the selected ones.
 * The slot order of the output is the selection order.
 * ------------------------------------------------------------------------------------- */
int orc_router_topk(const float *logits, int n, int k, int renorm, uint32_t *idx, double *p) {
  if (n <= 0 || k <= 0 || k > n) return ORC_EINVAL;
  char *taken = (char *)calloc((size_t)n, 1);
  if (!taken) return ORC_EINVAL;
  for (int s = 0; s < k; ++s) {
    int best = -1;
    for (int e = 0; e < n; ++e) {
      if (taken[e]) continue;
      if (best < 0 || logits[e] > logits[best]) best = e; /* strict '>' keeps the lower index on ties */
    }
    taken[best] = 1;
    idx[s] = (uint32_t)best;
  }
  free(taken);
  double m = (double)logits[idx[0]];
  if (renorm) {
    double z = 0.0;
    for (int s = 0; s < k; ++s) z += exp((double)logits[idx[s]] - m);
    for (int s = 0; s < k; ++s) p[s] = exp((double)logits[idx[s]] - m) / z;
  } else {
    double z = 0.0;
    for (int e = 0; e < n; ++e) z += exp((double)logits[e] - m); /* idx[0] holds the global max */
    for (int s = 0; s < k; ++s) p[s] = exp((double)logits[idx[s]] - m) / z;
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------------------------
 * Scalar-weighted chain accumulate with residual:
 *   y[i] = r[i] + sum_{k<K} p[k] * v[k][i]
 * ([FFAI#14], scalar-FMA commit: scalarFMAChain8 fuses the eight base-plus-scalar-times-vector
 * updates of a top-8 MoE into one dispatch; the residual is added in the same pass, as
 * sigmoidScalarFMAResidual does after the MoE).
 * absref[i] = |r[i]| + sum_k |p[k] * v[k][i]|.  Indices i0 <= i < i1; outputs indexed i - i0.
 * r is bf16; v is fp32 [K][n].
 * ------------------------------------------------------------------------------------- */
void orc_chain_residual(const double *p, int K, const float *v, const uint16_t *r, int64_t n, int64_t i0,
                        int64_t i1, double *y, double *absref) {
  for (int64_t i = i0; i < i1; ++i) {
    double rv = orc_bf16_to_f64(r[i]);
    double acc = rv, aacc = fabs(rv);
    for (int k = 0; k < K; ++k) {
      double t = p[k] * (double)v[(int64_t)k * n + i];
      acc += t;
      aacc += fabs(t);
    }
    y[i - i0] = acc;
    if (absref) absref[i - i0] = aacc;
  }
}

/* ---------------------------------------------------------------------------------------
 * MoE top-K gather decode step ([FFAI#14], commits moeRouterTopK / dequantGemvInt4ExpertIndexed
 * and ffai_moe_down_swiglu_accum_int4_chain8):
 *   for each slot k:  e = idx[k];  g = Wg[e] x;  u = Wu[e] x;  h = silu(g) * u;  d = Wd[e] h
 *   y[i] = r[i] + sum_k p[k] * d_k[i]
 * The expert slab e of a stacked weight is the e-th [rows][in/8] block (and the e-th
 * [rows][in/gs] block of its scales and biases).  h stays in double.  A slot whose index is
 * >= n_experts contributes nothing and sets the returned flag bit (1 << k).
 * absref[i] = |r[i]| + sum_k |p[k]| * sum_j |Wd[e][i][j] * h_k[j]|.
 * Shapes: gate/up [n_experts][inter][hidden/8], down [n_experts][hidden][inter/8].
 * ------------------------------------------------------------------------------------- */
int orc_moe(const uint32_t *gq, const uint16_t *gs_, const uint16_t *gb, const uint32_t *uq, const uint16_t *us,
            const uint16_t *ub, const uint32_t *dq, const uint16_t *ds, const uint16_t *db, int64_t n_experts,
            int64_t hidden, int64_t inter, int64_t gsz, const uint32_t *idx, const double *p, int K,
            const uint16_t *x, const uint16_t *resid, double *y, double *absref) {
  if (hidden % gsz || inter % gsz || hidden % 8 || inter % 8) return ORC_EINVAL;
  double *g = (double *)malloc(sizeof(double) * (size_t)inter);
  double *u = (double *)malloc(sizeof(double) * (size_t)inter);
  double *h = (double *)malloc(sizeof(double) * (size_t)inter);
  double *d = (double *)malloc(sizeof(double) * (size_t)hidden);
  double *da = (double *)malloc(sizeof(double) * (size_t)hidden);
  if (!g || !u || !h || !d || !da) return ORC_EINVAL;
  int flags = 0;
  for (int64_t i = 0; i < hidden; ++i) {
    y[i] = orc_bf16_to_f64(resid[i]);
    if (absref) absref[i] = fabs(y[i]);
  }
  const int64_t gu_words = inter * (hidden / 8), gu_groups = inter * (hidden / gsz);
  const int64_t d_words = hidden * (inter / 8), d_groups = hidden * (inter / gsz);
  for (int k = 0; k < K; ++k) {
    int64_t e = (int64_t)idx[k];
    if (e < 0 || e >= n_experts) {
      flags |= 1 << k;
      continue;
    }
    orc_qgemv_rows(gq + e * gu_words, gs_ + e * gu_groups, gb + e * gu_groups, inter, hidden, gsz, x, ORC_X_BF16,
                   0, inter, g, NULL);
    orc_qgemv_rows(uq + e * gu_words, us + e * gu_groups, ub + e * gu_groups, inter, hidden, gsz, x, ORC_X_BF16,
                   0, inter, u, NULL);
    orc_swiglu(g, u, inter, h);
    orc_qgemv_rows_f64x(dq + e * d_words, ds + e * d_groups, db + e * d_groups, hidden, inter, gsz, h, 0, hidden, d,
                        da);
    for (int64_t i = 0; i < hidden; ++i) {
      y[i] += p[k] * d[i];
      if (absref) absref[i] += fabs(p[k]) * da[i];
    }
  }
  free(g);
  free(u);
  free(h);
  free(d);
  free(da);
  return flags;
}

/* ---------------------------------------------------------------------------------------
 * Dequant-GEMM for T > 1:  Y[t][r] = sum_j w[r][j] * X[t][j]  ([FFAI#9] "Ops.dequantGemmDynamicM:
 * host-side T-padding driver ... Pads T -> ceil(T/32)*32 with zero rows, dispatches, slices the
 * first T rows back").  Padding rows contribute nothing to the first T rows, so the oracle
 * computes exactly T rows.  X is bf16 [T][in].  Rows r0 <= r < r1; Y and absref are
 * [T][r1 - r0].
 * ------------------------------------------------------------------------------------- */
int orc_qgemm_rows(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases, int64_t out, int64_t in,
                   int64_t gs, const uint16_t *X, int64_t T, int64_t r0, int64_t r1, double *Y, double *absref) {
  if (T <= 0) return ORC_EINVAL;
  int64_t w = r1 - r0;
  for (int64_t t = 0; t < T; ++t) {
    int rc = orc_qgemv_rows(packed, scales, biases, out, in, gs, X + t * in, ORC_X_BF16, r0, r1, Y + t * w,
                            absref ? absref + t * w : NULL);
    if (rc) return rc;
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------------------------
 * RMSNorm ([FFAI#14] commit wrapping "ffai_rms_norm_qgemv_fast": the norm's output is fed
 * straight into the int4 dequant-GEMV; the page names the norm without writing it out, and
 * the plain reading is the usual root-mean-square norm with a per-element weight gamma and an
 * epsilon inside the root):
 *   out[j] = x[j] * gamma[j] / sqrt( (1/n) sum_i x[i]^2 + eps )
 * x bf16 or fp32 [n]; gamma bf16 [n]; out double [n].  The sum of squares runs in index order.
 * ------------------------------------------------------------------------------------- */
int orc_rmsnorm(const void *x, int xtype, const uint16_t *gamma, int64_t n, double eps, double *out) {
  if (n <= 0 || eps < 0.0) return ORC_EINVAL;
  double ss = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double v = load_x(x, xtype, i);
    ss += v * v;
  }
  double denom = sqrt(ss / (double)n + eps);
  if (!(denom > 0.0)) return ORC_EINVAL; /* all-zero x with eps = 0 has no norm */
  for (int64_t j = 0; j < n; ++j) out[j] = load_x(x, xtype, j) * orc_bf16_to_f64(gamma[j]) / denom;
  return ORC_OK;
}

/* ---------------------------------------------------------------------------------------
 * Gated RMSNorm ([FFAI#14] "gatedRmsNormQgemvInt4Fast": the Mamba2-style gated norm of the GDN
 * mixer's output, silu(z) * w * rmsnorm(y), before its out-projection; heads of head_dim
 * consecutive elements, "Hv*Dv" of them in all):
 *   for head h (elements j = h*head_dim .. (h+1)*head_dim - 1):
 *     r_h = sqrt( (1/head_dim) sum_{i in h} y[i]^2 + eps )
 *     out[j] = silu(z[j]) * gamma[j] * y[j] / r_h,      silu(t) = t / (1 + exp(-t))
 * head_dim = n is the norm over the whole vector.  y, z bf16 or fp32 (the same type) [n]; gamma
 * bf16 [n]; out double [n].  Sums in index order.
 * ------------------------------------------------------------------------------------- */
int orc_gated_rmsnorm(const void *y, const void *z, int xtype, const uint16_t *gamma, int64_t n, int64_t head_dim,
                      double eps, double *out) {
  if (n <= 0 || head_dim <= 0 || n % head_dim != 0 || eps < 0.0) return ORC_EINVAL;
  for (int64_t h0 = 0; h0 < n; h0 += head_dim) {
    double ss = 0.0;
    for (int64_t i = h0; i < h0 + head_dim; ++i) {
      double v = load_x(y, xtype, i);
      ss += v * v;
    }
    double r = sqrt(ss / (double)head_dim + eps);
    if (!(r > 0.0)) return ORC_EINVAL; /* an all-zero head with eps = 0 has no norm */
    for (int64_t j = h0; j < h0 + head_dim; ++j) {
      double t = load_x(z, xtype, j);
      double silu = t / (1.0 + exp(-t));
      out[j] = silu * orc_bf16_to_f64(gamma[j]) * (load_x(y, xtype, j) / r);
    }
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------------------------
 * Sigmoid-gated scalar FMA with the residual folded in ([FFAI#14], scalar-FMA commit:
 * sigmoidScalarFMAResidual takes a gate, a value, a base and a residual and adds the sigmoid-gated
 * value and the residual to the base in one pass; the shared-expert step of a decode layer:
 * y = routed + sigmoid(shared_gate . x) * shared_expert(x) + r):
 *   out[i] = base[i] + sigmoid(gate) * value[i] + residual[i]      (residual may be NULL)
 * sigmoid(g) = 1 / (1 + exp(-g)).  gate: one value; value, base fp32 [n]; residual bf16 [n].
 * absref[i] = |base[i]| + |sigmoid(gate) * value[i]| + |residual[i]|.
 * ------------------------------------------------------------------------------------- */
double orc_sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

void orc_sigmoid_scalar_fma(double gate, const float *value, const float *base, const uint16_t *residual, int64_t n,
                            double *out, double *absref) {
  double s = orc_sigmoid(gate);
  for (int64_t i = 0; i < n; ++i) {
    double b = (double)base[i];
    double t = s * (double)value[i];
    double r = residual ? orc_bf16_to_f64(residual[i]) : 0.0;
    out[i] = b + t + r;
    if (absref) absref[i] = fabs(b) + fabs(t) + fabs(r);
  }
}

/* ---------------------------------------------------------------------------------------
 * Affine group-64 quantizer (encode) for the Q4_64A / Q2_64A formats ([ds4#844], Q4_64A /
 * Q2_64A commit: the codes come from the scale and bias as stored, after their rounding to bf16;
 * the page gives no formula for the scale and bias themselves -- the plain reading is min/max
 * affine):
 *   lo = min of the group (-0 taken as +0), hi = max;  scale = (hi - lo) / (2^bits - 1);  bias = lo
 *   s = bf16(scale), b = bf16(bias)            (round to nearest, ties to even)
 *   q_j = clamp(round_to_nearest_even((w_j - b) / s), 0, 2^bits - 1);   q_j = 0 when s == 0
 * The codes are an integer decided by floating point, so they are computed here in the precision
 * the GPU kernel uses, IEEE binary32 with correctly rounded subtract, divide and
 * round-to-integer (the pages fix no precision).  Packing: bits = 4 -> 8 codes per u32, element
 * 8w + i at bits 4i; bits = 2 -> 16 codes per u32, element 16w + i at bits 2i (low first).
 * w bf16 or fp32 [out][in]; packed [out][in * bits / 32]; scales, biases bf16 [out][in / 64].
 * ------------------------------------------------------------------------------------- */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16); /* inf / nan: not expected */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t orc_bf16_round(float f) { return f32_to_bf16_rne(f); }

int orc_quantize_rows(const void *w, int wtype, int64_t out, int64_t in, int bits, int64_t r0, int64_t r1,
                      uint32_t *packed, uint16_t *scales, uint16_t *biases) {
  if ((bits != 4 && bits != 2) || in % 64 != 0 || in <= 0 || r0 < 0 || r1 > out || r0 > r1) return ORC_EINVAL;
  const int per_word = 32 / bits;
  const unsigned qmax = (1u << bits) - 1u;
  const int64_t ngs = in / 64, nwords = in / per_word;
  for (int64_t r = r0; r < r1; ++r) {
    for (int64_t g = 0; g < ngs; ++g) {
      float lo = 0.f, hi = 0.f;
      for (int64_t j = 0; j < 64; ++j) {
        float v = (float)load_x(w, wtype, r * in + g * 64 + j); /* bf16 / fp32: exact in binary32 */
        if (j == 0 || v < lo) lo = v;
        if (j == 0 || v > hi) hi = v;
      }
      volatile float lz = lo + 0.0f, hz = hi + 0.0f; /* a zero of either sign taken as +0 */
      lo = lz;
      hi = hz;
      volatile float range = hi - lo;                 /* binary32 operations, one rounding each */
      volatile float scale = range / (float)qmax;
      uint16_t sb = f32_to_bf16_rne(scale), bb = f32_to_bf16_rne(lo);
      scales[r * ngs + g] = sb;
      biases[r * ngs + g] = bb;
      float s = bf16_to_f32(sb), b = bf16_to_f32(bb);
      for (int64_t j = 0; j < 64; j += per_word) {
        uint32_t word = 0;
        for (int i = 0; i < per_word; ++i) {
          unsigned q = 0;
          if (s != 0.f) {
            volatile float d = (float)load_x(w, wtype, r * in + g * 64 + j + i) - b;
            volatile float t = d / s;
            float qf = rintf(t); /* round to nearest, ties to even (default rounding mode) */
            if (qf < 0.f) qf = 0.f;
            if (qf > (float)qmax) qf = (float)qmax;
            q = (unsigned)qf;
          }
          word |= (uint32_t)q << (bits * i);
        }
        packed[r * nwords + (g * 64 + j) / per_word] = word;
      }
    }
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------------------------
 * 2-bit affine variant (Q2_64A, [ds4#844]): 16 codes per u32, element 16w + i at bits 2i of word
 * w (low first), codes 0..3; w = s * q + b per group of 64 with bf16 s, b; y = W x in double, as
 * orc_qgemv_rows.  packed [out][in / 16].
 * ------------------------------------------------------------------------------------- */
unsigned orc_code2(const uint32_t *packed, int64_t in, int64_t row, int64_t j) {
  uint32_t word = packed[row * (in / 16) + j / 16];
  return (unsigned)((word >> (2 * (j % 16))) & 0x3u);
}

int orc_qgemv2_rows(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases, int64_t out, int64_t in,
                    const void *x, int xtype, int64_t r0, int64_t r1, double *y, double *absref) {
  if (in <= 0 || in % 64 != 0 || r0 < 0 || r1 > out || r0 > r1) return ORC_EINVAL;
  if (xtype != ORC_X_BF16 && xtype != ORC_X_F32) return ORC_EINVAL;
  const int64_t ng = in / 64;
  for (int64_t r = r0; r < r1; ++r) {
    double acc = 0.0, aacc = 0.0;
    for (int64_t j = 0; j < in; ++j) {
      double s = orc_bf16_to_f64(scales[r * ng + j / 64]);
      double b = orc_bf16_to_f64(biases[r * ng + j / 64]);
      double t = (s * (double)orc_code2(packed, in, r, j) + b) * load_x(x, xtype, j);
      acc += t;
      aacc += fabs(t);
    }
    y[r - r0] = acc;
    if (absref) absref[r - r0] = aacc;
  }
  return ORC_OK;
}

/* 2-bit GEMV with a double-precision input vector (the 2-bit MoE down projection's h). */
int orc_qgemv2_rows_f64x(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases, int64_t out,
                         int64_t in, const double *x, int64_t r0, int64_t r1, double *y, double *absref) {
  if (in <= 0 || in % 64 != 0 || r0 < 0 || r1 > out || r0 > r1) return ORC_EINVAL;
  const int64_t ng = in / 64;
  for (int64_t r = r0; r < r1; ++r) {
    double acc = 0.0, aacc = 0.0;
    for (int64_t j = 0; j < in; ++j) {
      double s = orc_bf16_to_f64(scales[r * ng + j / 64]);
      double b = orc_bf16_to_f64(biases[r * ng + j / 64]);
      double t = (s * (double)orc_code2(packed, in, r, j) + b) * x[j];
      acc += t;
      aacc += fabs(t);
    }
    y[r - r0] = acc;
    if (absref) absref[r - r0] = aacc;
  }
  return ORC_OK;
}

/* The MoE decode step of orc_moe with 2-bit experts (Q2_64A): stacked gate/up packed
 * [E][inter][hidden / 16], down [E][hidden][inter / 16]; the same steps in the same order. */
int orc_moe2(const uint32_t *gq, const uint16_t *gs_, const uint16_t *gb, const uint32_t *uq, const uint16_t *us,
             const uint16_t *ub, const uint32_t *dq, const uint16_t *ds, const uint16_t *db, int64_t n_experts,
             int64_t hidden, int64_t inter, const uint32_t *idx, const double *p, int K, const uint16_t *x,
             const uint16_t *resid, double *y, double *absref) {
  if (hidden % 64 || inter % 64) return ORC_EINVAL;
  double *g = (double *)malloc(sizeof(double) * (size_t)inter);
  double *u = (double *)malloc(sizeof(double) * (size_t)inter);
  double *h = (double *)malloc(sizeof(double) * (size_t)inter);
  double *d = (double *)malloc(sizeof(double) * (size_t)hidden);
  double *da = (double *)malloc(sizeof(double) * (size_t)hidden);
  if (!g || !u || !h || !d || !da) return ORC_EINVAL;
  int flags = 0;
  for (int64_t i = 0; i < hidden; ++i) {
    y[i] = orc_bf16_to_f64(resid[i]);
    if (absref) absref[i] = fabs(y[i]);
  }
  const int64_t gu_words = inter * (hidden / 16), gu_groups = inter * (hidden / 64);
  const int64_t d_words = hidden * (inter / 16), d_groups = hidden * (inter / 64);
  for (int k = 0; k < K; ++k) {
    int64_t e = (int64_t)idx[k];
    if (e < 0 || e >= n_experts) {
      flags |= 1 << k;
      continue;
    }
    orc_qgemv2_rows(gq + e * gu_words, gs_ + e * gu_groups, gb + e * gu_groups, inter, hidden, x, ORC_X_BF16, 0,
                    inter, g, NULL);
    orc_qgemv2_rows(uq + e * gu_words, us + e * gu_groups, ub + e * gu_groups, inter, hidden, x, ORC_X_BF16, 0,
                    inter, u, NULL);
    orc_swiglu(g, u, inter, h);
    orc_qgemv2_rows_f64x(dq + e * d_words, ds + e * d_groups, db + e * d_groups, hidden, inter, h, 0, hidden, d, da);
    for (int64_t i = 0; i < hidden; ++i) {
      y[i] += p[k] * d[i];
      if (absref) absref[i] += fabs(p[k]) * da[i];
    }
  }
  free(g);
  free(u);
  free(h);
  free(d);
  free(da);
  return flags;
}
