// gemv_kernel.cuh -- the streaming int4 affine dequant-GEMV kernel (M = 1), shared by three uses:
//   * dense: one matrix, or n in {2,3,4} matrices sharing one input vector ([FFAI#14]
//     "dequant_gemv_int4_*", "dequantGemvInt4Two/Three/Four", "ffai_batched_qkv_qgemv_fast",
//     "ffai_batched_4_qgemv_fast");
//   * pair: gate/up matrices reduced with SwiGLU, h = silu(W_g x) * (W_u x) -- a dense gate/up
//     pair, or the k selected experts' gate/up slabs picked on the device from the router's index
//     array ([FFAI#14], commit moeRouterTopK / dequantGemvInt4ExpertIndexed);
//   * seg (MoE down): one output row is the concatenation of the k selected experts' down rows,
//     the input the concatenation of p_k * h_k, and the residual is added on the way out
//     ([FFAI#14] commit "ffai_moe_down_swiglu_accum_int4_chain8").
//
// Each weight is  w[r][j] = scale[r][j/64] * q[r][j] + bias[r][j/64]  (q = nibble j of row r, low
// nibble first), and each output an fp32 dot product with x.
//
// Design (GB300, sm_103a)
//   * Persistent grid, one CTA of 16 warps per SM.  A CTA owns a contiguous range of rows (one contiguous
//     byte range of codes per matrix).  (An L2 bulk prefetch of the CTA's whole range at kernel start
//     was measured slower: the flood of prefetch requests queued the x and code loads behind it.)
//   * x is read once per CTA and stored in shared memory as fixed point per 64-column group g, in two
//     16-bit passes: X_j = round(x_j 2^k_g), 2^k_g putting the group's largest |x| in [2^14, 2^15),
//     and L_j = round((x_j 2^k_g - X_j) 2^15).  The represented value is x~_j = X_j 2^-k_g (first
//     pass) or (X_j + L_j 2^-15) 2^-k_g (both); |x~_j - x_j| <= 2^(E_g - 15) or 2^(E_g - 30) with
//     2^E_g <= max|x_g| < 2^(E_g + 1), and bf16 x is exact for every element within 2^7 (2^22) of
//     its group's largest.  A group takes the second pass when its largest |x| is above 32 times its
//     mean |x| (outlier channels), else the first alone.  The bias term uses the group's sum of the
//     same x~, so a row is the fp32-rounded dot product of W with x~:
//       |y - W x| <= sum_g eps_g sum_{j in g} |w_j|  (+ fp32 rounding, ~1e-6 relative),
//     eps_g the pass's bound above.
//   * Warps are independent.  A work unit is 4 rows (2 for gate/up pairs) x 32 consecutive groups
//     (2048 columns): lane l handles group 32 c + l of each row, keeps that group of x in registers
//     for the unit, and reads its 32 bytes of codes per row straight from global memory with two
//     128-bit loads (a warp reads 1 KB contiguous per row) plus the group's scale and bias.  The
//     next unit's loads are issued before the current unit is computed (two register buffers in
//     turn); a warp walks its units u = warp, warp + 16, ... without divisions.
//   * Unpack + dot: two ANDs split a u32 word into the byte codes of its even and sixteen times its
//     odd nibbles; integer dp2a instructions accumulate q_j * X_j (and q_j * L_j) exactly in int32,
//     two products per instruction.  Per group and row the scale and bias are applied once in fp32:
//     y += s * (acc * 2^-k_g) + b * sum_g x~.
//   * Each unit's row sums go to shared memory; after a CTA barrier they are added in a fixed
//     order (deterministic), the epilogue (SwiGLU / residual) applied and the outputs written.
//   * Programmatic dependent launch: the first unit's codes are loaded before griddepcontrol.wait;
//     x, router outputs and all outputs are touched only after it.
#pragma once
#include <algorithm>
#include <atomic>
#include <type_traits>
#include <utility>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int kMaxMats = 8;
constexpr int kMaxXGroups = 512;  // groups of x: in <= 32768
enum GemvMode { kDense = 0, kPair = 1, kSeg = 2 };
constexpr int kThreads = 512;       // 16 warps per CTA, one CTA per SM
constexpr int kGroupsPerUnit = 32;  // groups of one work unit (one per lane)
constexpr int kXBytesPerGroup = 265;  // shared memory per group of x: X (128), L (128), factors (8), flag (1)
// A group of x takes the second fixed-point pass when its largest |x| exceeds 32 times its mean |x|
// (sum |x| < 2 max |x|): outlier channels, where the first pass alone would leave the group's small
// entries with a few bits.  Below the ratio the first pass's error, 2^-15 max|x_g| sum |w| at most,
// is under 32 2^-15 = 0.98e-3 times mean|x_g| sum |w|.  (The SwiGLU output of the dense layer here
// peaks at 25 times its group mean, so it never takes the second pass; N(0, 1) inputs at 7.)
constexpr float kLoSumOverMax = 2.0f;

// A weight operand: base pointers of a (possibly stacked) weight, and the expert slot whose slab to
// use (-1: the base itself).
struct WRef {
  const uint32_t* packed;
  const uint16_t* scales;
  const uint16_t* biases;
  int slot;
};

struct GemvMat {
  WRef w[2];  // [0] main / gate, [1] up (pair mode)
  float* y;
  int out;
  int row0;  // first flattened row of this matrix
};

struct GemvArgs {
  GemvMat mat[kMaxMats];
  int nmat;
  WRef seg;               // seg mode: the stacked weight whose slabs form the segments
  int nseg;               // segments per row (1 unless seg mode)
  const void* x;          // [nseg][in] (bf16 or fp32)
  int xf32;               // x is fp32
  const uint32_t* idx;    // expert indices (device) or null
  const float* p;         // per-slot weights (seg mode)
  const uint16_t* resid;  // residual added by the finisher (seg mode) or null
  int n_experts;
  long long slab_words, slab_groups;  // per-expert strides of stacked weights
  int in;                             // columns of one segment (multiple of 64)
  int groups;                         // nseg * in / 64
  int total_rows;
  int rows_per_cta;  // upper bound of a CTA's row count (sizes the partial-sum buffer)
  // Router in the kernel (pair mode, MoE gate/up): with `logits` set, every CTA selects the top
  // nmat of n_logits logits itself (instead of reading idx), and CTA 0 writes the selection to
  // idx_out / p_out for the kernels that follow.
  const float* logits;
  int n_logits, renorm;
  uint32_t* idx_out;
  float* p_out;
  // x staging: with `stage` set, x arrives in shared memory (at byte offset stage_off) through one
  // bulk copy, which the TMA engine serves beside the weight loads already in flight; otherwise the
  // threads load it into registers.
  int stage, stage_off;
  // RMSNorm prologue (NORM kernels): the product is taken with x * gamma / sqrt(mean(x^2) + eps):
  // x * gamma is what gets quantized, and the finisher multiplies by the root (y is linear in x).
  const uint16_t* gamma;  // bf16 [in]
  float eps;
  // Gated RMSNorm (NORM kernels, dense, gz set): x * gamma * silu(z) is quantized, and every group's
  // x factors are scaled by its head's 1 / sqrt(mean over the head of x^2 + eps) before the main
  // loop (heads of head_dim columns, a multiple of 64).
  const void* gz;  // z, the type of x [in]
  int head_dim;
  // Gated epilogue (dense): y = ebase + sigmoid(*sgate) * (W x), then + resid when set.
  const float* sgate;
  const float* ebase;
  int bits;  // code width: 4 (Q4_64A, 8 codes per u32) or 2 (Q2_64A, 16 per u32)
};

struct WPtr {
  const uint32_t* packed;
  const uint16_t* scales;
  const uint16_t* biases;
};

// Resolve a weight reference to this call's slab, expert indices from `idx` (global or shared
// memory).  `ok` is false for an out-of-range index.
__device__ __forceinline__ WPtr resolve(const GemvArgs& a, const uint32_t* idx, const WRef& r, bool& ok) {
  ok = true;
  if (r.slot < 0) return WPtr{r.packed, r.scales, r.biases};
  const uint32_t e = idx[r.slot];
  if (e >= (uint32_t)a.n_experts) {
    ok = false;
    return WPtr{r.packed, r.scales, r.biases};
  }
  return WPtr{r.packed + (size_t)e * a.slab_words, r.scales + (size_t)e * a.slab_groups,
              r.biases + (size_t)e * a.slab_groups};
}

// d = c + a.lo16 * b.byte0 + a.hi16 * b.byte1 (lo) or b.byte2, b.byte3 (hi); a signed 16-bit,
// b unsigned bytes, exact int32 arithmetic.
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 16-bit fixed point by the magic-number rule: for |t| < 2^22, t + 1.5 * 2^23 rounded to float
// has the nearest integer to t (ties to even) in its low mantissa bits: the float's bit pattern is
// 0x4B400000 + round(t), whose low 16 bits are round(t) as a 16-bit two's-complement value when
// |round(t)| < 2^15.

// Row sums of RN per-lane values; lane l returns the total of value (l * RN) / 32.
template <int RN>
__device__ __forceinline__ float warp_sum_rows(const float (&v)[RN], int lane) {
  if constexpr (RN == 1) {
    float c = v[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    return c;
  } else if constexpr (RN == 2) {
    const bool b4 = lane & 16;
    float c = (b4 ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, b4 ? v[0] : v[1], 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    return c;
  } else {
    static_assert(RN == 4, "RN in {1, 2, 4}");
    const bool b4 = lane & 16, b3 = lane & 8;
    const float a0 = (b4 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, b4 ? v[0] : v[2], 16);
    const float a1 = (b4 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, b4 ? v[1] : v[3], 16);
    float c = (b3 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, b3 ? a0 : a1, 8);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    return c;
  }
}

// One lane's loads of one work unit: RN entries (row, component), each the group's 32 bytes of
// codes (8 words) plus its scale and bias bits.
template <int RN>
struct UnitLoads {
  uint4 a[RN], b[RN];
  uint32_t s[RN], t[RN];
};

// A warp's position in its sequence of work units u = warp, warp + NW, ...: row block u / nkc and
// K chunk u % nkc, advanced without a division.
struct UnitCursor {
  int blk, kc;
};

// Row block b of a CTA's rows [vb, ve): blocks of RB rows formed per matrix.  Returns false past
// the last block.
template <int RB>
__device__ __forceinline__ bool block_rows(const GemvArgs& a, int vb, int ve, int b, int& m, int& r_first,
                                           int& nr, int& local0) {
  int bb = b;
  for (int mi = 0; mi < a.nmat; ++mi) {
    const int lo = max(vb, a.mat[mi].row0), hi = min(ve, a.mat[mi].row0 + a.mat[mi].out);
    if (lo >= hi) continue;
    const int nb = (hi - lo + RB - 1) / RB;
    if (bb < nb) {
      m = mi;
      r_first = lo - a.mat[mi].row0 + bb * RB;
      nr = min(RB, hi - (lo + bb * RB));
      local0 = lo + bb * RB - vb;
      return true;
    }
    bb -= nb;
  }
  return false;
}

// ------------------------------------------------------------------ router top-k (one warp)
// Order-preserving key of a finite float: larger floats give larger unsigned keys; -0 and +0 get
// the same key (they compare equal, so the index decides between them).
__device__ __forceinline__ uint32_t router_float_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of n logits by one warp ([FFAI#14] commit "moeRouterTopK"; order (value desc, index asc)
// as in [FFAI#9]): a candidate is the 64-bit key (float key << 32) | ~index, unique per expert, so
// round s takes the warp's largest key below round s - 1's.  Weights: softmax over the k selected
// logits (renorm) or over all n read at the selected ones.  Results for slot s go to idx[s] / p[s]
// (shared memory) and, when given, to gidx[s] / gp[s] (global).  k <= 32, n <= 1024.
__device__ __forceinline__ void route_topk_warp(const float* logits, int n, int k, int renorm, uint32_t* idx,
                                                float* p, uint32_t* gidx, float* gp) {
  const int lane = threadIdx.x & 31;
  // up to 128 experts: the lane's keys stay in registers; beyond, they are re-read each round
  unsigned long long kr[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = lane + 32 * j;
    kr[j] = e < n ? ((unsigned long long)router_float_key(__ldg(logits + e)) << 32) | (uint32_t)~(uint32_t)e : 0ull;
  }
  unsigned long long prev = ~0ull, mine = 0;
  for (int s = 0; s < k; ++s) {
    unsigned long long best = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (kr[j] < prev && kr[j] > best) best = kr[j];
    for (int e = lane + 128; e < n; e += 32) {
      const unsigned long long key = ((unsigned long long)router_float_key(__ldg(logits + e)) << 32) | (uint32_t)~(uint32_t)e;
      if (key < prev && key > best) best = key;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
      best = o > best ? o : best;
    }
    if (lane == s) mine = best;
    prev = best;
  }
  const uint32_t my_idx = ~(uint32_t)mine;
  const uint32_t kv = (uint32_t)(mine >> 32);
  const float my_v = __uint_as_float((kv & 0x80000000u) ? (kv & 0x7FFFFFFFu) : ~kv);
  const float m = __shfl_sync(0xffffffffu, my_v, 0);  // round 0 took the largest logit
  float z = 0.f;
  if (renorm) {
    z = lane < k ? expf(my_v - m) : 0.f;
  } else {
    for (int e = lane; e < n; e += 32) z += expf(__ldg(logits + e) - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  if (lane < k) {
    const float pv = expf(my_v - m) / z;
    idx[lane] = my_idx;
    p[lane] = pv;
    if (gidx) {
      gidx[lane] = my_idx;
      gp[lane] = pv;
    }
  }
}

// Shared memory per CTA: x of group g as 32 u32 (64 int16 values paired for dp2a: per 8-column
// word w, (X0, X2), (X4, X6), (X1, X3), (X5, X7)) stored at 16-byte slot (w + g) % 8 of the group's
// 128 bytes -- the rotation keeps a warp's loads (one group per lane, 128 bytes apart) free of bank
// conflicts; then the second fixed-point pass L in the same layout (written for the groups that
// take it); then per group (2^-k_g / 16, the sum of its represented values, -, takes-the-second-pass
// flag); then the partial sums [row][NC][chunk]; then (STG) the staged copy of x.
// STG: x arrives through one bulk copy (a.stage set by the planner), else the threads load it.
// BITS: 4 or 2 (the 2-bit variant is built without NORM).
template <int MODE, int RN, bool STG, bool NORM, int BITS = 4>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float s_gss[NORM ? kMaxXGroups : 1];  // gated: each group's sum of x^2, then
  __shared__ float s_hrn[NORM ? kMaxXGroups : 1];  // each head's 1 / root
  __shared__ uint32_t s_idx[kMaxMats];  // the in-kernel router's selection
  __shared__ float s_p[kMaxMats];
  __shared__ float s_ss[kThreads / 32];  // NORM: per-warp sums of x^2
  __shared__ __align__(8) uint64_t xbar;  // the x copy's completion
  pdl_trigger();
  if (STG && threadIdx.x == 0) {
    mbar_init(&xbar, 1);
    mbar_fence_init();
  }
  constexpr bool PAIR = MODE == kPair, SEG = MODE == kSeg;
  constexpr int NC = PAIR ? 2 : 1;  // components per row
  constexpr int RB = RN / NC;       // rows per work unit
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NW = kThreads / 32;
  const int G = a.groups;
  const int ngs = a.in / 64;  // groups per segment
  uint32_t* xq = reinterpret_cast<uint32_t*>(smem);                      // [G][32] first pass X
  uint32_t* xl = reinterpret_cast<uint32_t*>(smem + (size_t)G * 128);    // [G][32] second pass L
  float2* gsx = reinterpret_cast<float2*>(smem + (size_t)G * 256);       // [G]
  uint8_t* gflag = smem + (size_t)G * 264;                                // [G] takes the second pass
  float* part = reinterpret_cast<float*>(smem + (((size_t)G * 265 + 15) & ~(size_t)15));  // [rows][NC][nkc]

  const int vb = (int)((long long)blockIdx.x * a.total_rows / gridDim.x);
  const int ve = (int)((long long)(blockIdx.x + 1) * a.total_rows / gridDim.x);
  const int nkc = (G + kGroupsPerUnit - 1) / kGroupsPerUnit;  // K chunks per row

  const bool indexed = a.idx != nullptr || a.logits != nullptr;  // slots resolved through indices
  const uint32_t* idxp = a.logits ? s_idx : a.idx;

  int nblocks = 0;
  for (int mi = 0; mi < a.nmat; ++mi) {
    const int lo = max(vb, a.mat[mi].row0), hi = min(ve, a.mat[mi].row0 + a.mat[mi].out);
    if (lo < hi) nblocks += (hi - lo + RB - 1) / RB;
  }
  const int nunits = nblocks * nkc;

  // The loads of a unit for this lane.
  auto issue = [&](const UnitCursor& uc, UnitLoads<RN>& L) {
    int m = 0, rf = 0, nr = 0, l0 = 0;
    block_rows<RB>(a, vb, ve, uc.blk, m, rf, nr, l0);
    const int g = uc.kc * kGroupsPerUnit + lane;  // this lane's group (across segments)
    const bool gv = g < G;
    const int gl = gv ? g : G - 1;  // (a valid group to load from; its terms are zeroed below)
    const int sg = SEG ? gl / ngs : 0;
    const int lg = SEG ? gl - sg * ngs : gl;
#pragma unroll
    for (int e = 0; e < RN; ++e) {
      const int r = e / NC, c = e % NC;
      bool ok;
      const WPtr w = resolve(a, idxp, SEG ? WRef{a.seg.packed, a.seg.scales, a.seg.biases, sg} : a.mat[m].w[c], ok);
      const size_t row = (size_t)(rf + min(r, nr - 1));
      // Every load is in bounds (clamped row and group, the base slab for a bad expert); entries
      // past the block, past the last group or of a bad expert get scale and bias 0, so add 0.
      if constexpr (BITS == 4) {
        const uint4* src = reinterpret_cast<const uint4*>(w.packed + row * (size_t)(a.in / 8)) + lg * 2;
        L.a[e] = __ldg(src);
        L.b[e] = __ldg(src + 1);
      } else {  // a group's 64 2-bit codes: one 16-byte word
        L.a[e] = __ldg(reinterpret_cast<const uint4*>(w.packed + row * (size_t)(a.in / 16)) + lg);
      }
      const bool live = ok && gv && r < nr;
      L.s[e] = live ? (uint32_t)__ldg(w.scales + row * (size_t)ngs + lg) : 0u;
      L.t[e] = live ? (uint32_t)__ldg(w.biases + row * (size_t)ngs + lg) : 0u;
    }
  };
  // u -> u + NW: NW = bstep * nkc + kstep
  const int bstep = NW / nkc, kstep = NW % nkc;
  auto advance = [&](UnitCursor uc) {
    uc.blk += bstep;
    uc.kc += kstep;
    if (uc.kc >= nkc) {
      uc.kc -= nkc;
      ++uc.blk;
    }
    return uc;
  };

  UnitLoads<RN> b0, b1;
  int u = warp;
  UnitCursor uc{warp / nkc, warp % nkc};
  if (u < nunits && !indexed) issue(uc, b0);  // before the dependency wait: weights only

  // --- x: 16-bit fixed point per group, into shared memory ---
  pdl_wait();
  uint8_t* stage = smem + a.stage_off;
  if (STG && threadIdx.x == 0) {
    // (x was written before this kernel and shared memory is untouched so far: no proxy fence,
    // which would also wait for this thread's weight loads in flight)
    constexpr uint32_t kChunk = 32768;
    const uint32_t xbytes = (uint32_t)G * (a.xf32 ? 256u : 128u);
    const uint32_t gbytes = NORM ? (uint32_t)G * 128u : 0u;  // gamma after x
    mbar_arrive_expect_tx(&xbar, xbytes + gbytes);
    for (uint32_t off = 0; off < xbytes; off += kChunk)
      bulk_g2s_bytes(stage + off, static_cast<const uint8_t*>(a.x) + off, min(kChunk, xbytes - off), &xbar);
    if constexpr (NORM) {
      for (uint32_t off = 0; off < gbytes; off += kChunk)
        bulk_g2s_bytes(stage + xbytes + off, reinterpret_cast<const uint8_t*>(a.gamma) + off, min(kChunk, gbytes - off),
                       &xbar);
    }
  }
  if (a.logits) {  // the router, in every CTA
    if (warp == 0) route_topk_warp(a.logits, a.n_logits, a.nmat, a.renorm, s_idx, s_p, blockIdx.x == 0 ? a.idx_out : nullptr,
                                   blockIdx.x == 0 ? a.p_out : nullptr);
    __syncthreads();
  }
  if (u < nunits && indexed) issue(uc, b0);
  {
    // 8 lanes per group, 8 values (one 8-column word) per lane.  All of a thread's loads (up to 8
    // groups of bf16 or 5 of fp32: one round for every in <= 32768 bf16 / 20480 fp32) are issued
    // together and then processed: one memory latency for the whole prologue.  The loops are
    // uniform per warp (shuffles below).
    const int sub = lane & 7;
    float ss = 0.f;  // NORM: this thread's sum of x^2
    // NORM: accumulate x^2 (live groups only), then x *= gamma (eight bf16 in gw)
    auto apply_norm = [&](int g, float (&v)[8], const uint4& gw) {
      float pg = 0.f;  // this lane's part of group g's sum of x^2
      if (g < G) {
#pragma unroll
        for (int j = 0; j < 8; ++j) pg = fmaf(v[j], v[j], pg);
      }
      ss += pg;
      const uint32_t w[4] = {gw.x, gw.y, gw.z, gw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] *= __uint_as_float(w[j] << 16);
        v[2 * j + 1] *= __uint_as_float(w[j] & 0xFFFF0000u);
      }
      if (a.gz) {  // gated (uniform): times silu(z), and the group's sum of x^2 for its head
        float zf[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (g < G) {
          if (a.xf32) {
            const float4* zp = reinterpret_cast<const float4*>(static_cast<const float*>(a.gz) + (size_t)g * 64) + 2 * sub;
            const float4 z0 = __ldg(zp), z1 = __ldg(zp + 1);
            zf[0] = z0.x; zf[1] = z0.y; zf[2] = z0.z; zf[3] = z0.w;
            zf[4] = z1.x; zf[5] = z1.y; zf[6] = z1.z; zf[7] = z1.w;
          } else {
            const uint4 zr = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.gz) + (size_t)g * 64) + sub);
            const uint32_t zw[4] = {zr.x, zr.y, zr.z, zr.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              zf[2 * j] = __uint_as_float(zw[j] << 16);
              zf[2 * j + 1] = __uint_as_float(zw[j] & 0xFFFF0000u);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] *= zf[j] / (1.f + expf(-zf[j]));
        pg += __shfl_xor_sync(0xffffffffu, pg, 1);
        pg += __shfl_xor_sync(0xffffffffu, pg, 2);
        pg += __shfl_xor_sync(0xffffffffu, pg, 4);
        if (sub == 0 && g < G) s_gss[g] = pg;
      }
    };
    // Group g of x (eight values per lane, eight lanes) to fixed point: the first pass
    // X_j = round(x_j 2^k) with 2^k putting the group's largest |x| in [2^14, 2^15), the second pass
    // L_j = round((x_j 2^k - X_j) 2^15); x~_j = (X_j + L_j 2^-15) 2^-k.  The per-group sums of the
    // represented values (first pass alone, and both passes) carry the bias term, so that the code
    // and bias terms see the same x~ and the whole product is the exact W x~ up to fp32 rounding.
    auto quant = [&](int g, const float (&v)[8]) {
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      // E = floor(log2 max|x|), k = 14 - E: |x| 2^k < 2^15.  Groups whose largest |x| is below
      // 2^-60 add less than 64 |w| 2^-60 to a row and are dropped (X = L = 0).
      const bool live = m >= 8.673617e-19f;  // 2^-60
      int E = max((int)((__float_as_uint(m) >> 23) & 0xFF) - 127, -60);
      // When max|x| 2^k would round up to 2^15 (fp32 x only: a bf16 max is at most
      // (2 - 2^-7) 2^14 after scaling), one bit less for this group, so every |X_j| <= 32767.
      if (live && m * exp2i(14 - E) >= 32767.5f) ++E;
      const float scale = live ? exp2i(14 - E) : 0.f;  // 14 - E in [-113, 74]
      // X_j = the low 16 bits of the float x_j 2^k + 1.5 2^23 (the magic-number rule above)
      uint32_t b[8];
      float sa = 0.f;  // sum of |x_j|
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        b[j] = __float_as_uint(fmaf(v[j], scale, 12582912.0f));
        sa += fabsf(v[j]);
      }
      // sum of X_j, exact: dp2a of the packed int16 pairs with byte weights (1, 1)
      int hsi = 0;
#pragma unroll
      for (int j = 0; j < 8; j += 2) hsi = dp2a_lo(__byte_perm(b[j], b[j + 1], 0x5410), 0x0101u, hsi);
      float hs = (float)hsi;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {
        hs += __shfl_xor_sync(0xffffffffu, hs, o);
        sa += __shfl_xor_sync(0xffffffffu, sa, o);
      }
      const bool need = sa < kLoSumOverMax * m;  // (false for an all-zero group)
      float ls = 0.f;                            // sum of L_j (exact integers)
      uint32_t l[8];
      if (__any_sync(0xffffffffu, need)) {  // (uniform per warp) the second pass: the remainder
        // x_j 2^k - X_j (exact, |.| <= 1/2) scaled by 2^15, rounded by the same rule
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float u = fmaf(fmaf(v[j], scale, 12582912.0f - __uint_as_float(b[j])), 32768.0f, 12582912.0f);
          l[j] = __float_as_uint(u);
          ls += u - 12582912.0f;
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
      }
      if (g < G) {
        // paired for dp2a as (X0, X2), (X4, X6), (X1, X3), (X5, X7); 2-bit: (X0, X4), (X1, X5), ...
        constexpr int P0 = BITS == 4 ? 0 : 0, P1 = BITS == 4 ? 2 : 4, P2 = BITS == 4 ? 4 : 1, P3 = BITS == 4 ? 6 : 5;
        constexpr int P4 = BITS == 4 ? 1 : 2, P5 = BITS == 4 ? 3 : 6, P6 = BITS == 4 ? 5 : 3, P7 = BITS == 4 ? 7 : 7;
        reinterpret_cast<uint4*>(xq + (size_t)g * 32)[(sub + g) & 7] =
            make_uint4(__byte_perm(b[P0], b[P1], 0x5410), __byte_perm(b[P2], b[P3], 0x5410),
                       __byte_perm(b[P4], b[P5], 0x5410), __byte_perm(b[P6], b[P7], 0x5410));
        if (need)
          reinterpret_cast<uint4*>(xl + (size_t)g * 32)[(sub + g) & 7] =
              make_uint4(__byte_perm(l[P0], l[P1], 0x5410), __byte_perm(l[P2], l[P3], 0x5410),
                         __byte_perm(l[P4], l[P5], 0x5410), __byte_perm(l[P6], l[P7], 0x5410));
        if (sub == 0) {
          float wgt = 1.f;
          if (SEG) {
            bool ok;
            resolve(a, idxp, WRef{a.seg.packed, a.seg.scales, a.seg.biases, g / ngs}, ok);
            wgt = ok ? __ldg(a.p + g / ngs) : 0.f;
          }
          // (2^-k / 16: the odd codes are accumulated sixteen times over, see the main loop); the
          // group's sum of its represented values x~ (both passes when it takes the second)
          const float kinv = live ? exp2i(E - 14) * wgt : 0.f;
          gsx[g] = make_float2(live ? exp2i(E - (BITS == 4 ? 18 : 20)) * wgt : 0.f,
                               (need ? fmaf(ls, 3.0517578125e-05f, hs) : hs) * kinv);
          gflag[g] = need ? 1 : 0;
        }
      }
    };
    if constexpr (STG) {
      // one group per 8 lanes, four groups per warp and step, read from the staged copy
      __syncthreads();  // (the barrier's initialisation, by thread 0, before anyone waits on it)
      if (!__syncthreads_and(mbar_wait(&xbar, 0))) return;
      const uint32_t st = smem_u32(stage);
      for (int g0 = warp * 4; g0 < G; g0 += NW * 4) {
        const int g = g0 + (lane >> 3);
        const int gs = g < G ? g : G - 1;  // (in range; its results are not stored)
        float v[8];
        if (!a.xf32) {
          const uint4 r = lds128(st + (uint32_t)gs * 128u + (uint32_t)sub * 16u);
          const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
          }
        } else {
          const uint4 r0 = lds128(st + (uint32_t)gs * 256u + (uint32_t)sub * 32u);
          const uint4 r1 = lds128(st + (uint32_t)gs * 256u + (uint32_t)sub * 32u + 16u);
          const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(w[j]);
        }
        if constexpr (NORM) {
          const uint32_t gofs = (uint32_t)G * (a.xf32 ? 256u : 128u);  // gamma after x
          apply_norm(g, v, lds128(st + gofs + (uint32_t)gs * 128u + (uint32_t)sub * 16u));
        }
        quant(g, v);
      }
    } else if (!a.xf32) {
      constexpr int XB = NORM ? 4 : 8;  // (NORM: gamma's words take the other half of the registers)
      for (int gb = warp * 4; gb < G; gb += NW * 4 * XB) {
        uint4 raw[XB], graw[NORM ? XB : 1];
#pragma unroll
        for (int i = 0; i < XB; ++i) {
          const int g = gb + i * NW * 4 + (lane >> 3);
          raw[i] = g < G ? __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + (size_t)g * 64) + sub)
                         : make_uint4(0u, 0u, 0u, 0u);
          if constexpr (NORM)
            graw[i] = g < G ? __ldg(reinterpret_cast<const uint4*>(a.gamma + (size_t)g * 64) + sub) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < XB; ++i) {
          if (gb + i * NW * 4 >= G) break;  // (uniform per warp: nothing left in this batch)
          const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
          float v[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
          }
          if constexpr (NORM) apply_norm(gb + i * NW * 4 + (lane >> 3), v, graw[i]);
          quant(gb + i * NW * 4 + (lane >> 3), v);
        }
      }
    } else {
      constexpr int XB = NORM ? 3 : 5;
      for (int gb = warp * 4; gb < G; gb += NW * 4 * XB) {
        float4 r0[XB], r1[XB];
        uint4 graw[NORM ? XB : 1];
#pragma unroll
        for (int i = 0; i < XB; ++i) {
          const int g = gb + i * NW * 4 + (lane >> 3);
          const float4* p4 = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)g * 64) + 2 * sub;
          r0[i] = g < G ? __ldg(p4) : make_float4(0.f, 0.f, 0.f, 0.f);
          r1[i] = g < G ? __ldg(p4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
          if constexpr (NORM)
            graw[i] = g < G ? __ldg(reinterpret_cast<const uint4*>(a.gamma + (size_t)g * 64) + sub) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < XB; ++i) {
          if (gb + i * NW * 4 >= G) break;  // (uniform per warp: nothing left in this batch)
          float v[8] = {r0[i].x, r0[i].y, r0[i].z, r0[i].w, r1[i].x, r1[i].y, r1[i].z, r1[i].w};
          if constexpr (NORM) apply_norm(gb + i * NW * 4 + (lane >> 3), v, graw[i]);
          quant(gb + i * NW * 4 + (lane >> 3), v);
        }
      }
    }
    if constexpr (NORM) {  // the CTA's sum of x^2, per warp (added in warp order by the finisher)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) s_ss[warp] = ss;
    }
  }
  if (a.idx && blockIdx.x == 0 && (int)threadIdx.x < (SEG ? a.nseg : a.nmat)) {
    if (idxp[threadIdx.x] >= (uint32_t)a.n_experts) set_status(QG_STATUS_BAD_EXPERT);
  }
  __syncthreads();
  if constexpr (NORM) {
    if (a.gz) {  // gated: each head's root, then every group's x factors scaled by its head's
      const int hg = a.head_dim / 64, nh = G / hg;
      for (int h = threadIdx.x; h < nh; h += kThreads) {
        float t = 0.f;
        for (int q = 0; q < hg; ++q) t += s_gss[h * hg + q];
        s_hrn[h] = 1.f / sqrtf(t / (float)a.head_dim + a.eps);
      }
      __syncthreads();
      for (int g = threadIdx.x; g < G; g += kThreads) {
        const float r = s_hrn[g / hg];
        gsx[g] = make_float2(gsx[g].x * r, gsx[g].y * r);
      }
      __syncthreads();
    }
  }

  // --- main loop: this warp's units u = warp, warp + NW, ...; two buffers in turn, the next unit's
  // codes in flight while one is computed ---
  const uint32_t xq_s = smem_u32(xq), xl_s = smem_u32(xl);
  // The unit's RN dot products in exact int32 arithmetic, word by word (word wd of this lane's group
  // of x from shared memory, the codes in registers).  LO: the second pass too (the warp takes it
  // when one of its 32 groups does; the other lanes' L reads as zero).
  auto dot = [&](const UnitLoads<RN>& L, uint32_t xo, bool own_lo, auto lo_tag, float (&acc)[RN]) {
    constexpr bool LO = decltype(lo_tag)::value;
    if constexpr (BITS == 4 && !LO) {
      int s0[RN], s1[RN];
#pragma unroll
      for (int e = 0; e < RN; ++e) s0[e] = s1[e] = 0;
#pragma unroll
      for (int wd = 0; wd < 8; ++wd) {
        const uint4 X = lds128(xq_s + xo + (uint32_t)((wd + (xo >> 7)) & 7) * 16u);
#pragma unroll
        for (int e = 0; e < RN; ++e) {
          const uint4& c4 = wd < 4 ? L.a[e] : L.b[e];
          const int k = wd & 3;
          const uint32_t w = k == 0 ? c4.x : k == 1 ? c4.y : k == 2 ? c4.z : c4.w;
          const uint32_t c0 = w & 0x0F0F0F0Fu;  // codes q0, q2, q4, q6 as bytes
          const uint32_t c1 = w & 0xF0F0F0F0u;  // 16 q1, 16 q3, 16 q5, 16 q7
          s0[e] = dp2a_hi(X.y, c0, dp2a_lo(X.x, c0, s0[e]));
          s1[e] = dp2a_hi(X.w, c1, dp2a_lo(X.z, c1, s1[e]));
        }
      }
      // |s0| <= 32 * 15 * 32767 and |s1| <= 16 times that: 16 s0 + s1 < 2^29, exact in int32
      // (rounded once to float, relative error 2^-24); the group factor carries the matching 1/16
#pragma unroll
      for (int e = 0; e < RN; ++e) acc[e] = (float)(s0[e] * 16 + s1[e]);
    } else if constexpr (BITS == 4) {
      // both passes; each pass in one accumulator, its even codes as bytes 16 q (one shift), so
      // that both sums are 16 sum q X: |.| <= 64 * 240 * 32767 < 2^31 (second pass: half that)
      int s[RN], t[RN];
#pragma unroll
      for (int e = 0; e < RN; ++e) s[e] = t[e] = 0;
#pragma unroll
      for (int wd = 0; wd < 8; ++wd) {
        const uint32_t ofs = xo + (uint32_t)((wd + (xo >> 7)) & 7) * 16u;
        const uint4 X = lds128(xq_s + ofs);
        const uint4 Lw = own_lo ? lds128(xl_s + ofs) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int e = 0; e < RN; ++e) {
          const uint4& c4 = wd < 4 ? L.a[e] : L.b[e];
          const int k = wd & 3;
          const uint32_t w = k == 0 ? c4.x : k == 1 ? c4.y : k == 2 ? c4.z : c4.w;
          const uint32_t c0 = (w & 0x0F0F0F0Fu) << 4;  // 16 q0, 16 q2, 16 q4, 16 q6
          const uint32_t c1 = w & 0xF0F0F0F0u;         // 16 q1, 16 q3, 16 q5, 16 q7
          s[e] = dp2a_hi(X.w, c1, dp2a_lo(X.z, c1, dp2a_hi(X.y, c0, dp2a_lo(X.x, c0, s[e]))));
          t[e] = dp2a_hi(Lw.w, c1, dp2a_lo(Lw.z, c1, dp2a_hi(Lw.y, c0, dp2a_lo(Lw.x, c0, t[e]))));
        }
      }
      // the second pass weighs 2^-15 (each sum rounded once to float, then one fused add)
#pragma unroll
      for (int e = 0; e < RN; ++e) acc[e] = fmaf((float)t[e], 3.0517578125e-05f, (float)s[e]);
    } else {
      // 2-bit: word k holds columns 16k .. 16k + 15 at bits 2i; masks 3 << 2m pick codes
      // m, m + 4, m + 8, m + 12 as bytes (times 4^m), paired with (X_m, X_m+4) of x's word 2k
      // and (X_m+8, X_m+12) of word 2k + 1
      int s0[RN], s1[RN], s2[RN], s3[RN], t0[RN], t1[RN], t2[RN], t3[RN];
#pragma unroll
      for (int e = 0; e < RN; ++e) s0[e] = s1[e] = s2[e] = s3[e] = t0[e] = t1[e] = t2[e] = t3[e] = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t oa = xo + (uint32_t)((2 * k + (xo >> 7)) & 7) * 16u;
        const uint32_t ob = xo + (uint32_t)((2 * k + 1 + (xo >> 7)) & 7) * 16u;
        const uint4 A = lds128(xq_s + oa), B = lds128(xq_s + ob);
        uint4 LA = make_uint4(0u, 0u, 0u, 0u), LB = LA;
        if (LO && own_lo) {
          LA = lds128(xl_s + oa);
          LB = lds128(xl_s + ob);
        }
#pragma unroll
        for (int e = 0; e < RN; ++e) {
          const uint32_t w = k == 0 ? L.a[e].x : k == 1 ? L.a[e].y : k == 2 ? L.a[e].z : L.a[e].w;
          const uint32_t c0 = w & 0x03030303u, c1 = w & 0x0C0C0C0Cu, c2 = w & 0x30303030u, c3 = w & 0xC0C0C0C0u;
          s0[e] = dp2a_hi(B.x, c0, dp2a_lo(A.x, c0, s0[e]));
          s1[e] = dp2a_hi(B.y, c1, dp2a_lo(A.y, c1, s1[e]));
          s2[e] = dp2a_hi(B.z, c2, dp2a_lo(A.z, c2, s2[e]));
          s3[e] = dp2a_hi(B.w, c3, dp2a_lo(A.w, c3, s3[e]));
          if constexpr (LO) {
            t0[e] = dp2a_hi(LB.x, c0, dp2a_lo(LA.x, c0, t0[e]));
            t1[e] = dp2a_hi(LB.y, c1, dp2a_lo(LA.y, c1, t1[e]));
            t2[e] = dp2a_hi(LB.z, c2, dp2a_lo(LA.z, c2, t2[e]));
            t3[e] = dp2a_hi(LB.w, c3, dp2a_lo(LA.w, c3, t3[e]));
          }
        }
      }
      // |s_m| <= 4^m * 16 * 3 * 32767: 64 s0 + 16 s1 + 4 s2 + s3 < 2^29, exact; gs.x carries 1/64
#pragma unroll
      for (int e = 0; e < RN; ++e) {
        acc[e] = (float)(s0[e] * 64 + s1[e] * 16 + s2[e] * 4 + s3[e]);
        if constexpr (LO)
          acc[e] = fmaf((float)(t0[e] * 64 + t1[e] * 16 + t2[e] * 4 + t3[e]), 3.0517578125e-05f, acc[e]);
      }
    }
  };
  // The unit's row sums into the partial-sum buffer.
  auto store_rows = [&](const float (&yp)[RN], const UnitCursor& c) {
    const float tot = warp_sum_rows<RN>(yp, lane);
    if ((lane & (32 / RN - 1)) == 0) {
      const int e = (lane * RN) >> 5;
      int m = 0, rf = 0, nr = 0, l0 = 0;
      block_rows<RB>(a, vb, ve, c.blk, m, rf, nr, l0);
      if (e / NC < nr) part[((l0 + e / NC) * NC + e % NC) * nkc + c.kc] = tot;
    }
  };
  auto compute = [&](const UnitLoads<RN>& L, const UnitCursor& c) {
    const int gc = min(c.kc * kGroupsPerUnit + lane, G - 1);
    // (gc past the last group: its scale and bias were loaded as zero, whatever it reads here)
    const bool own_lo = gflag[gc] != 0;
    float acc[RN];
    if (__builtin_expect(__any_sync(0xffffffffu, own_lo), 0))
      dot(L, (uint32_t)gc * 128u, own_lo, std::true_type{}, acc);
    else
      dot(L, (uint32_t)gc * 128u, false, std::false_type{}, acc);
    const float2 gs = gsx[gc];  // the bias term takes the group's sum of its represented x
    float yp[RN];
#pragma unroll
    for (int e = 0; e < RN; ++e) yp[e] = fmaf(bf16_bits_to_f32(L.s[e]), acc[e] * gs.x, bf16_bits_to_f32(L.t[e]) * gs.y);
    store_rows(yp, c);
  };
  for (; u < nunits; u += NW) {
    const UnitCursor un = advance(uc);
    if (u + NW < nunits) issue(un, b1);
    compute(b0, uc);
    b0 = b1;
    uc = un;
  }
  __syncthreads();

  // --- finish: sum each row's K chunks in order, epilogue, write ---
  float rn = 1.f;  // NORM: 1 / sqrt(mean(x^2) + eps) (gated: applied per head above)
  if constexpr (NORM) {
    if (!a.gz) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) t += s_ss[w];
    rn = 1.f / sqrtf(t / (float)a.in + a.eps);
    }
  }
  const float sig = a.sgate ? 1.f / (1.f + expf(-__ldg(a.sgate))) : 0.f;
  for (int lr = threadIdx.x; lr < ve - vb; lr += kThreads) {
    const int v = vb + lr;
    int m = 0;
    while (m + 1 < a.nmat && v >= a.mat[m + 1].row0) ++m;
    const GemvMat& mt = a.mat[m];
    const int row = v - mt.row0;
    float acc = 0.f;
    for (int kc = 0; kc < nkc; ++kc) acc += part[(lr * NC) * nkc + kc];
    if (NORM) acc *= rn;
    if (PAIR) {
      float up = 0.f;
      for (int kc = 0; kc < nkc; ++kc) up += part[(lr * NC + 1) * nkc + kc];
      if (NORM) up *= rn;
      bool ok = true;
      if (mt.w[0].slot >= 0) resolve(a, idxp, mt.w[0], ok);
      acc = ok ? acc / (1.f + expf(-acc)) * up : 0.f;
    }
    if (a.sgate) acc = fmaf(sig, acc, __ldg(a.ebase + row));
    if (a.resid) acc += bf16_bits_to_f32(a.resid[row]);
    mt.y[row] = acc;
  }
}

// ------------------------------------------------------------------ host side: arguments
// n matrices sharing x, rows of each written to its y.
inline GemvArgs dense_args(const GemvMatArg* mats, int n, const void* x, int xt, int in) {
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
  return a;
}

// A dense gate/up pair: h = silu(W_g x) * (W_u x).
inline GemvArgs pair_args(const GemvMatArg& gate, const GemvMatArg& up, const void* x, int xt, int in, float* h) {
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
  return a;
}

// The k selected experts' gate/up pairs, h[m] for slot m; experts from idx (set idx or the router
// fields before launching).
inline GemvArgs moe_gate_up_args(const qg_int4_weight* gate, const qg_int4_weight* up, const uint32_t* idx, int k,
                                 const uint16_t* x, float* h, int bits = 4) {
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
  a.slab_words = (long long)gate->out * (gate->in * bits / 32);
  a.slab_groups = (long long)gate->out * (gate->in / 64);
  a.in = gate->in;
  a.total_rows = k * gate->out;
  a.bits = bits;
  return a;
}

// MoE down with the slot-weighted accumulate and the residual (one row = k segments).
inline GemvArgs moe_down_args(const qg_int4_weight* down, const uint32_t* idx, const float* p, int k, const float* h,
                              const uint16_t* residual, float* y, int bits = 4) {
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
  a.slab_words = (long long)down->out * (down->in * bits / 32);
  a.slab_groups = (long long)down->out * (down->in / 64);
  a.in = down->in;
  a.total_rows = down->out;
  a.bits = bits;
  return a;
}

inline void apply_extras(GemvArgs& a, const GemvExtras& ex) {
  a.bits = ex.bits ? ex.bits : 4;
  a.gamma = ex.gamma;
  a.eps = ex.eps;
  a.gz = ex.gz;
  a.head_dim = ex.head_dim;
  a.sgate = ex.sgate;
  a.ebase = ex.ebase;
  a.resid = ex.resid;
}

// ------------------------------------------------------------------ host side: planning
struct GemvTune {
  int ctas_per_sm;  // 0: automatic
};
extern GemvTune g_gemv_tune;

inline size_t gemv_smem_bytes(int groups, int rows_per_cta, int nc) {
  const int nkc = (groups + kGroupsPerUnit - 1) / kGroupsPerUnit;
  return (((size_t)groups * kXBytesPerGroup + 15) & ~(size_t)15) + (size_t)rows_per_cta * nc * nkc * 4;
}

// Shared memory with the x staging area after `base` bytes, or `base` alone (staging off).  Staging
// is used for short x only: measured on the decode shapes, the bulk copy beat the threads' own loads
// for x of up to 128 groups (gate/up 5120 bf16: 20.7 -> 20.1 us; MoE 2048 bf16 and 8 x 768 fp32:
// 16.0 -> 14.9 us per layer) and lost for the 17408-wide down x (12.37 -> 12.54 us).
constexpr int kStageMaxGroups = 128;
inline size_t plan_stage(GemvArgs& a, size_t base, size_t limit) {
  const size_t off = (base + 127) & ~(size_t)127;
  const size_t total = off + (size_t)a.groups * ((a.xf32 ? 256 : 128) + (a.gamma ? 128 : 0));
  a.stage = total <= limit && a.groups <= kStageMaxGroups ? 1 : 0;
  a.stage_off = a.stage ? (int)off : 0;
  return a.stage ? total : base;
}
constexpr size_t kStaticSmemReserve = 8192;  // the kernels' static shared variables (NORM: 4.2 KB)

// The kernel's dynamic shared-memory limit is raised once per device (an attribute of the function
// in that device's context), to the largest size launched there so far.
template <int MODE, int RN, bool STG, bool NORM, int BITS = 4>
int launch_gemv_variant(const GemvArgs& a, int grid, size_t smem, cudaStream_t stream) {
  auto k = gemv_kernel<MODE, RN, STG, NORM, BITS>;
  constexpr int kDevs = 64;
  static std::atomic<int> smem_set[kDevs];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return QG_EDEVICE;
  if ((int)smem > smem_set[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return QG_ELAUNCH;
    smem_set[dev].store((int)smem, std::memory_order_relaxed);
  }
  return launch(k, dim3(grid), dim3(kThreads), smem, stream, a);
}

// Plan (grid, shared memory) and launch.
template <int MODE>
int plan_and_launch(GemvArgs& a, cudaStream_t stream) {
  const DeviceInfo& dev = device_info();
  constexpr int NC = MODE == kPair ? 2 : 1;
  a.groups = a.nseg * a.in / 64;
  const int cps = g_gemv_tune.ctas_per_sm ? g_gemv_tune.ctas_per_sm : 1;
  int grid = std::max(1, std::min(cps * dev.num_sms, a.total_rows));
  // keep x and the partial-sum buffer within the shared memory (more, smaller CTAs otherwise)
  const size_t budget = (size_t)dev.max_smem_optin - kStaticSmemReserve;
  for (;;) {
    a.rows_per_cta = (a.total_rows + grid - 1) / grid;
    if (gemv_smem_bytes(a.groups, a.rows_per_cta, NC) <= budget || grid >= a.total_rows) break;
    grid = std::min(a.total_rows, grid * 2);
  }
  const size_t limit = (size_t)dev.max_smem_optin - kStaticSmemReserve;
  const size_t smem = plan_stage(a, gemv_smem_bytes(a.groups, a.rows_per_cta, NC), limit);
  if (smem > limit) return QG_ENOTSUP;
  // rows x components per work unit: 4 (dense and seg: four rows; pair: two rows, gate and up)
  if (a.bits == 2) {
    if (a.gamma) return QG_ENOTSUP;
    return a.stage ? launch_gemv_variant<MODE, 4, true, false, 2>(a, grid, smem, stream)
                   : launch_gemv_variant<MODE, 4, false, false, 2>(a, grid, smem, stream);
  }
  if constexpr (MODE != kSeg) {
    if (a.gamma)
      return a.stage ? launch_gemv_variant<MODE, 4, true, true>(a, grid, smem, stream)
                     : launch_gemv_variant<MODE, 4, false, true>(a, grid, smem, stream);
  }
  return a.stage ? launch_gemv_variant<MODE, 4, true, false>(a, grid, smem, stream)
                 : launch_gemv_variant<MODE, 4, false, false>(a, grid, smem, stream);
}

}  // namespace qg
