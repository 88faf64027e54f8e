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
// kPairRouted: the MoE gate/up kernel that selects the experts from the logits itself (built
// apart, so that the other kernels carry none of the router's code).
enum GemvMode { kDense = 0, kPair = 1, kSeg = 2, kPairRouted = 3 };
__host__ __device__ constexpr bool mode_pair(int m) { return m == kPair || m == kPairRouted; }
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
  // Router in the kernel (the routed gate/up mode): with `logits` set, every CTA selects the top
  // nmat of n_logits logits itself instead of reading idx, and CTA 0 writes the selection to
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
  // Split K across a thread-block cluster of kcl CTAs (1: no split).  The CTAs of a cluster share
  // one row range; CTA rank r takes the r-th contiguous slice of the K chunks, converts only that
  // slice of x, and the slices' row sums are added through distributed shared memory in rank order.
  int kcl;
  int slice_groups;  // groups of x in the largest slice (sizes shared memory)
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
// round s takes the warp's largest key not yet taken.  Two steps, so that the logits' loads can be
// in flight beside other loads: router_load issues them (the first 128 experts' keys stay in
// registers, the rest are re-read each round), router_select runs the k rounds (the warp's largest
// key as the largest upper half, then the largest lower half among the lanes holding it: two warp
// reductions per round) and the weights: softmax over the k selected logits (renorm) or over all n
// read at the selected ones.  Results for slot s go to idx[s] / p[s] and, when given, to
// gidx[s] / gp[s].  k <= 32, n <= 1024.  The logits are read through L2 (ld.global.cg).
struct RouterKeys {
  unsigned long long kr[4];
};
__device__ __forceinline__ unsigned long long router_key(float f, int e) {
  return ((unsigned long long)router_float_key(f) << 32) | (uint32_t)~(uint32_t)e;
}
__device__ __forceinline__ RouterKeys router_load(const float* logits, int n) {
  const int lane = threadIdx.x & 31;
  RouterKeys r;
  float v[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) v[j] = lane + 32 * j < n ? __ldcg(logits + lane + 32 * j) : 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) r.kr[j] = lane + 32 * j < n ? router_key(v[j], lane + 32 * j) : 0ull;
  return r;
}
__device__ __forceinline__ void router_select(RouterKeys r, const float* logits, int n, int k, int renorm,
                                              uint32_t* idx, float* p, uint32_t* gidx, float* gp) {
  const int lane = threadIdx.x & 31;
  unsigned long long prev = ~0ull, mine = 0;
  for (int s = 0; s < k; ++s) {
    unsigned long long best = 0;  // (taken register keys are zeroed; no key is 0)
#pragma unroll
    for (int j = 0; j < 4; ++j) best = r.kr[j] > best ? r.kr[j] : best;
    for (int e = lane + 128; e < n; e += 32) {
      const unsigned long long key = router_key(__ldcg(logits + e), e);
      if (key < prev && key > best) best = key;
    }
    const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32));
    const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32) == hi ? (uint32_t)best : 0u);
    best = ((unsigned long long)hi << 32) | lo;
#pragma unroll
    for (int j = 0; j < 4; ++j) r.kr[j] = r.kr[j] == best ? 0ull : r.kr[j];
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
    for (int e = lane; e < n; e += 32) z += expf(__ldcg(logits + e) - m);
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
  __syncwarp();
}

// The logit a key was made from (-0 comes back as +0).
__device__ __forceinline__ float router_key_value(unsigned long long key) {
  const uint32_t kv = (uint32_t)(key >> 32);
  return __uint_as_float((kv & 0x80000000u) ? (kv & 0x7FFFFFFFu) : ~kv);
}

// CTA-wide top-k for n <= kRankExperts experts, all threads of the CTA: the expert of rank r (the
// number of keys above its own) goes to sel[r] for r < k.  Thread t counts the keys above expert
// t / 4's among every fourth expert from t % 4 (the four lanes' loads of one step fall in distinct
// banks), and the four counts are added by shuffles.  keys[0, n) (keys as in router_select) is
// complete before the call; the caller places a barrier before sel is read.
constexpr int kRankExperts = kThreads / 4;
__device__ __forceinline__ void router_rank(const unsigned long long* keys, int n, int k, uint32_t* sel) {
  const int e = threadIdx.x >> 2, q = threadIdx.x & 3;
  int c = 0;
  if (e < n) {
    const unsigned long long ke = keys[e];
#pragma unroll 8
    for (int j = q; j < n; j += 4) c += keys[j] > ke ? 1 : 0;
  }
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  if (e < n && q == 0 && c < k) sel[c] = (uint32_t)e;
}

// The weights of the selection sel[0, k) by one warp: softmax over the k selected logits (renorm)
// or over all n, from the keys; slot s's expert and weight to idx[s] / p[s] and, when given,
// gidx[s] / gp[s].
__device__ __forceinline__ void router_weights(const unsigned long long* keys, int n, int k, int renorm,
                                               const uint32_t* sel, uint32_t* idx, float* p, uint32_t* gidx,
                                               float* gp) {
  const int lane = threadIdx.x & 31;
  const uint32_t my_idx = lane < k ? sel[lane] : sel[0];
  const float my_v = router_key_value(keys[my_idx]);
  const float m = __shfl_sync(0xffffffffu, my_v, 0);  // rank 0: the largest logit
  float z = 0.f;
  if (renorm) {
    z = lane < k ? expf(my_v - m) : 0.f;
  } else {
    for (int e = lane; e < n; e += 32) z += expf(router_key_value(keys[e]) - m);
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
  __syncwarp();
}

// ------------------------------------------------------------------ thread-block cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of all CTAs of the cluster: shared-memory writes before it are visible to the
// cluster's CTAs after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// A float in CTA `rank`'s shared memory at the address this CTA's `p` has in its own.
__device__ __forceinline__ float ld_peer_f32(const float* p, uint32_t rank) {
  uint32_t ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// Shared memory per CTA: x of group g as 32 u32 (64 int16 values paired for dp2a: per 8-column
// word w, (X0, X2), (X4, X6), (X1, X3), (X5, X7)) stored at 16-byte slot (w + g) % 8 of the group's
// 128 bytes -- the rotation keeps a warp's loads (one group per lane, 128 bytes apart) free of bank
// conflicts; then the second fixed-point pass L in the same layout (written for the groups that
// take it); then per group (2^-k_g / 16, the sum of its represented values, -, takes-the-second-pass
// flag); then the partial sums [row][NC][chunk]; then (STG) the staged copy of x.
// STG: x arrives through one bulk copy (a.stage set by the planner), else the threads load it.
// BITS: 4 or 2 (the 2-bit variant is built without NORM).
template <int MODE, int RN, bool STG, bool NORM, int BITS = 4, bool KS = false>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float s_gss[NORM ? kMaxXGroups : 1];  // gated: each group's sum of x^2, then
  __shared__ float s_hrn[NORM ? kMaxXGroups : 1];  // each head's 1 / root
  constexpr bool PAIR = mode_pair(MODE), SEG = MODE == kSeg;
  constexpr bool ROUTED = MODE == kPairRouted;  // a.logits set
  constexpr int NRW = ROUTED ? kThreads / 32 : 1;
  __shared__ uint32_t s_idx[NRW][kMaxMats];  // the router's selection, per warp
  __shared__ float s_p[NRW][kMaxMats];
  __shared__ unsigned long long s_key[ROUTED ? kRankExperts : 1];  // the router's keys
  __shared__ uint32_t s_sel[kMaxMats];
  __shared__ float s_ss[kThreads / 32];  // NORM: per-warp sums of x^2
  __shared__ __align__(8) uint64_t xbar;  // the x copy's completion
  pdl_trigger();
  if (STG && threadIdx.x == 0) {
    mbar_init(&xbar, 1);
    mbar_fence_init();
  }
  constexpr int NC = PAIR ? 2 : 1;  // components per row
  constexpr int RB = RN / NC;       // rows per work unit
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NW = kThreads / 32;
  const int ngs = a.in / 64;  // groups per segment
  // This CTA's K slice: chunks [kc0, kc0 + nkc) of the row's chunks of 32 groups, i.e. groups
  // [gb0, gend) of x (all of them without a split); rows [vb, ve), its cluster's.
  // (KS: the kernel built for a K split; without it, one CTA per row range and all of K)
  const int C = KS ? a.kcl : 1;
  const int rank = KS ? (int)cluster_rank() : 0;
  const int ncl = KS ? (int)gridDim.x / C : (int)gridDim.x, cid = KS ? (int)blockIdx.x / C : (int)blockIdx.x;
  const int nkc_all = (a.groups + kGroupsPerUnit - 1) / kGroupsPerUnit;
  const int kc0 = KS ? rank * nkc_all / C : 0;
  const int nkc = KS ? (rank + 1) * nkc_all / C - kc0 : nkc_all;  // K chunks per row in this CTA
  const int gb0 = kc0 * kGroupsPerUnit;
  const int gend = KS ? min(a.groups, gb0 + nkc * kGroupsPerUnit) : a.groups;
  const int G = gend - gb0;  // groups of x in this CTA (local index g - gb0)
  const int GS = KS ? a.slice_groups : a.groups;  // (layout: every CTA of the launch uses the same offsets)
  uint32_t* xq = reinterpret_cast<uint32_t*>(smem);                      // [G][32] first pass X
  uint32_t* xl = reinterpret_cast<uint32_t*>(smem + (size_t)GS * 128);   // [G][32] second pass L
  float2* gsx = reinterpret_cast<float2*>(smem + (size_t)GS * 256);      // [G]
  uint8_t* gflag = smem + (size_t)GS * 264;                               // [G] takes the second pass
  float* part = reinterpret_cast<float*>(smem + (((size_t)GS * 265 + 15) & ~(size_t)15));  // [rows][NC][nkc]

  const int vb = (int)((long long)cid * a.total_rows / ncl);
  const int ve = (int)((long long)(cid + 1) * a.total_rows / ncl);

  const bool indexed = ROUTED || a.idx != nullptr;  // slots resolved through indices
  // Routed: the selection, made after the dependency wait, from each warp's own copy.
  const uint32_t* idxp = ROUTED ? s_idx[ROUTED ? warp : 0] : a.idx;

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
    const int g = gb0 + uc.kc * kGroupsPerUnit + lane;  // this lane's group (across segments)
    const bool gv = g < gend;
    const int gl = gv ? g : gend - 1;  // (a valid group to load from; its terms are zeroed below)
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
  // The router (logits set), every thread of the CTA (uniform; barriers inside): up to
  // kRankExperts experts ranked by the whole CTA, more by each warp on its own.  w0: the warp that
  // writes the selection to idx_out / p_out.
  auto route = [&](bool w0) {
    if constexpr (ROUTED) {
      const int k = a.nmat, n = a.n_logits;
      uint32_t* gi = w0 ? a.idx_out : nullptr;
      float* gp = w0 ? a.p_out : nullptr;
      if (n <= kRankExperts) {
        if ((int)threadIdx.x < n) s_key[threadIdx.x] = router_key(__ldcg(a.logits + threadIdx.x), (int)threadIdx.x);
        __syncthreads();
        router_rank(s_key, n, k, s_sel);
        __syncthreads();
        router_weights(s_key, n, k, a.renorm, s_sel, s_idx[warp], s_p[warp], gi, gp);
      } else {
        router_select(router_load(a.logits, n), a.logits, n, k, a.renorm, s_idx[warp], s_p[warp], gi, gp);
      }
    }
  };
  if (u < nunits && !indexed) issue(uc, b0);  // before the dependency wait: weights only
  // Before the wait, the lines that the first steps after it read (the logits, or the indices and
  // slot weights, and this CTA's slice of a staged x) are asked into L2 with their address
  // translations: the values may still change, but L2 is where the writes land, so the reads after
  // the wait see them.
  if constexpr (MODE == kPairRouted) {
    if ((int)threadIdx.x * 32 < a.n_logits) prefetch_l2(a.logits + threadIdx.x * 32);
  } else {
    if (threadIdx.x == 0 && a.idx) prefetch_l2(a.idx);
    if (threadIdx.x == 32 && a.p) prefetch_l2(a.p);
  }
  if constexpr (STG) {
    const int nl = G * (a.xf32 ? 2 : 1);
    const uint8_t* xb = static_cast<const uint8_t*>(a.x) + (size_t)gb0 * (a.xf32 ? 256u : 128u);
    for (int i = threadIdx.x; i < nl; i += kThreads) prefetch_l2(xb + (size_t)i * 128);
  }

  // --- x: 16-bit fixed point per group, into shared memory ---
  bool xok = true;   // (false: x never arrived)
  bool tlo = false;  // one of this thread's groups takes the second pass
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
      bulk_g2s_bytes(stage + off, static_cast<const uint8_t*>(a.x) + (size_t)gb0 * (a.xf32 ? 256u : 128u) + off,
                     min(kChunk, xbytes - off), &xbar);
    if constexpr (NORM) {
      for (uint32_t off = 0; off < gbytes; off += kChunk)
        bulk_g2s_bytes(stage + xbytes + off, reinterpret_cast<const uint8_t*>(a.gamma) + (size_t)gb0 * 128u + off,
                       min(kChunk, gbytes - off), &xbar);
    }
  }
  if constexpr (MODE == kPairRouted) {  // the router, then the weights, then x (staged meanwhile)
    route(blockIdx.x == 0 && warp == 0);
    if (u < nunits) issue(uc, b0);
  } else if constexpr (!ROUTED) {
    if (u < nunits && indexed) issue(uc, b0);  // indices from the previous kernel
  }
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
            const float4* zp = reinterpret_cast<const float4*>(static_cast<const float*>(a.gz) + (size_t)(gb0 + g) * 64) + 2 * sub;
            const float4 z0 = __ldg(zp), z1 = __ldg(zp + 1);
            zf[0] = z0.x; zf[1] = z0.y; zf[2] = z0.z; zf[3] = z0.w;
            zf[4] = z1.x; zf[5] = z1.y; zf[6] = z1.z; zf[7] = z1.w;
          } else {
            const uint4 zr = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.gz) + (size_t)(gb0 + g) * 64) + sub);
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
    // The first pass of group g (eight values per lane in v, eight lanes): X_j = round(x_j 2^k),
    // the group's factor and the sum of its represented values, and whether it takes the second
    // pass (computed after the prologue's barrier, only where some group takes it).
    auto quant = [&](int g, const float (&v)[8]) {
      float m = 0.f, sa = 0.f;  // largest |x_j|, sum of |x_j|
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        m = fmaxf(m, fabsf(v[j]));
        sa += fabsf(v[j]);
      }
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
      // X_j = the low 16 bits of the float x_j 2^k + 1.5 2^23 (the magic-number rule above); their
      // sum, exact, by dp2a of the packed int16 pairs with byte weights (1, 1)
      uint32_t b[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) b[j] = __float_as_uint(fmaf(v[j], scale, 12582912.0f));
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
      tlo |= need && g < G;
      if (g < G) {
        // paired for dp2a as (X0, X2), (X4, X6), (X1, X3), (X5, X7); 2-bit: (X0, X4), (X1, X5), ...
        uint4 pk;
        if constexpr (BITS == 4) {
          pk.x = __byte_perm(b[0], b[2], 0x5410);
          pk.y = __byte_perm(b[4], b[6], 0x5410);
          pk.z = __byte_perm(b[1], b[3], 0x5410);
          pk.w = __byte_perm(b[5], b[7], 0x5410);
        } else {
          pk.x = __byte_perm(b[0], b[4], 0x5410);
          pk.y = __byte_perm(b[1], b[5], 0x5410);
          pk.z = __byte_perm(b[2], b[6], 0x5410);
          pk.w = __byte_perm(b[3], b[7], 0x5410);
        }
        reinterpret_cast<uint4*>(xq + (size_t)g * 32)[(sub + g) & 7] = pk;
        if (sub == 0) {
          float wgt = 1.f;
          if (SEG) {
            bool ok;
            resolve(a, idxp, WRef{a.seg.packed, a.seg.scales, a.seg.biases, (gb0 + g) / ngs}, ok);
            wgt = ok ? __ldg(a.p + (gb0 + g) / ngs) : 0.f;
          }
          // (2^-k / 16: the odd codes are accumulated sixteen times over, see the main loop); the
          // group's sum of its represented values (the second pass adds its part later)
          gsx[g] = make_float2(live ? exp2i(E - (BITS == 4 ? 18 : 20)) * wgt : 0.f,
                               live ? hs * exp2i(E - 14) * wgt : 0.f);
          gflag[g] = need ? 1 : 0;
        }
      }
    };
    if constexpr (STG) {
      // one group per 8 lanes, four groups per warp and step, read from the staged copy
      __syncthreads();  // (the barrier's initialisation, by thread 0, before anyone waits on it)
      // a copy that never lands (bounded wait, QG_STATUS_TIMEOUT set): nothing is converted and no
      // output is written, but the CTA still reaches its cluster's barriers
      xok = __syncthreads_and(mbar_wait(&xbar, 0));
      const uint32_t st = smem_u32(stage);
      for (int g0 = warp * 4; xok && g0 < G; g0 += NW * 4) {
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
          raw[i] = g < G ? __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + (size_t)(gb0 + g) * 64) + sub)
                         : make_uint4(0u, 0u, 0u, 0u);
          if constexpr (NORM)
            graw[i] = g < G ? __ldg(reinterpret_cast<const uint4*>(a.gamma + (size_t)(gb0 + g) * 64) + sub) : make_uint4(0u, 0u, 0u, 0u);
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
          const float4* p4 = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)(gb0 + g) * 64) + 2 * sub;
          r0[i] = g < G ? __ldg(p4) : make_float4(0.f, 0.f, 0.f, 0.f);
          r1[i] = g < G ? __ldg(p4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
          if constexpr (NORM)
            graw[i] = g < G ? __ldg(reinterpret_cast<const uint4*>(a.gamma + (size_t)(gb0 + g) * 64) + sub) : make_uint4(0u, 0u, 0u, 0u);
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
  // some group of this CTA's x takes the second pass: the main loop with it, else the one without
  const bool anylo = __syncthreads_or(tlo);
  if (__builtin_expect(anylo, 0)) {
    // The second pass, for the groups that take it (rare: outlier channels), after the barrier so
    // that the common prologue stays short: each such group's eight lanes load its x again (with
    // the norm's factors), L_j = round((x_j 2^k - X_j) 2^15) with the first pass's k and X, and the
    // group's sum of represented values gains (sum L) 2^-15 2^-k.
    const int sub = lane & 7;
    const uint32_t st = smem_u32(smem + a.stage_off);
    for (int g0 = warp * 4; g0 < G; g0 += NW * 4) {
      const int g = g0 + (lane >> 3);
      if (g >= G || !gflag[g]) continue;  // (uniform per 8 lanes; the shuffles below name those 8)
      const uint32_t m8 = 0xFFu << (lane & 24);
      float v[8];
      const size_t gx = (size_t)(gb0 + g) * 64 + (size_t)sub * 8;  // this lane's first element
      if (STG && !a.xf32) {
        const uint4 r = lds128(st + (uint32_t)g * 128u + (uint32_t)sub * 16u);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[2 * j] = __uint_as_float(w[j] << 16);
          v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      } else if (STG) {
        const uint4 r0 = lds128(st + (uint32_t)g * 256u + (uint32_t)sub * 32u);
        const uint4 r1 = lds128(st + (uint32_t)g * 256u + (uint32_t)sub * 32u + 16u);
        const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(w[j]);
      } else if (!a.xf32) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + gx));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[2 * j] = __uint_as_float(w[j] << 16);
          v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      } else {
        const float4* p4 = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + gx);
        const float4 r0 = __ldg(p4), r1 = __ldg(p4 + 1);
        v[0] = r0.x; v[1] = r0.y; v[2] = r0.z; v[3] = r0.w;
        v[4] = r1.x; v[5] = r1.y; v[6] = r1.z; v[7] = r1.w;
      }
      if constexpr (NORM) {  // x * gamma (* silu(z)): the values the first pass quantized
        const uint4 gw = STG ? lds128(st + (uint32_t)G * (a.xf32 ? 256u : 128u) + (uint32_t)g * 128u + (uint32_t)sub * 16u)
                             : __ldg(reinterpret_cast<const uint4*>(a.gamma + gx));
        const uint32_t w[4] = {gw.x, gw.y, gw.z, gw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[2 * j] *= __uint_as_float(w[j] << 16);
          v[2 * j + 1] *= __uint_as_float(w[j] & 0xFFFF0000u);
        }
        if (a.gz) {
          float zf[8];
          if (a.xf32) {
            const float4* zp = reinterpret_cast<const float4*>(static_cast<const float*>(a.gz) + gx);
            const float4 z0 = __ldg(zp), z1 = __ldg(zp + 1);
            zf[0] = z0.x; zf[1] = z0.y; zf[2] = z0.z; zf[3] = z0.w;
            zf[4] = z1.x; zf[5] = z1.y; zf[6] = z1.z; zf[7] = z1.w;
          } else {
            const uint4 zr = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.gz) + gx));
            const uint32_t zw[4] = {zr.x, zr.y, zr.z, zr.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              zf[2 * j] = __uint_as_float(zw[j] << 16);
              zf[2 * j + 1] = __uint_as_float(zw[j] & 0xFFFF0000u);
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] *= zf[j] / (1.f + expf(-zf[j]));
        }
      }
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(m8, m, o));
      const bool live = m >= 8.673617e-19f;  // (the first pass's rule, step for step)
      int E = max((int)((__float_as_uint(m) >> 23) & 0xFF) - 127, -60);
      if (live && m * exp2i(14 - E) >= 32767.5f) ++E;
      const float scale = live ? exp2i(14 - E) : 0.f;
      // the remainder x_j 2^k - X_j (exact, |.| <= 1/2) scaled by 2^15, rounded by the magic rule
      uint32_t l[8];
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float t = fmaf(v[j], scale, 12582912.0f);  // (1.5 2^23 + X_j)
        const float u = fmaf(fmaf(v[j], scale, 12582912.0f - t), 32768.0f, 12582912.0f);
        l[j] = __float_as_uint(u);
        ls += u - 12582912.0f;
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) ls += __shfl_xor_sync(m8, ls, o);
      uint4 pl;
      if constexpr (BITS == 4) {
        pl = make_uint4(__byte_perm(l[0], l[2], 0x5410), __byte_perm(l[4], l[6], 0x5410),
                        __byte_perm(l[1], l[3], 0x5410), __byte_perm(l[5], l[7], 0x5410));
      } else {
        pl = make_uint4(__byte_perm(l[0], l[4], 0x5410), __byte_perm(l[1], l[5], 0x5410),
                        __byte_perm(l[2], l[6], 0x5410), __byte_perm(l[3], l[7], 0x5410));
      }
      reinterpret_cast<uint4*>(xl + (size_t)g * 32)[(sub + g) & 7] = pl;
      if (sub == 0) {  // 2^-k (times the slot weight) is the group factor times 16 (2-bit: 64)
        const float2 f = gsx[g];
        gsx[g] = make_float2(f.x, fmaf(ls * 3.0517578125e-05f, f.x * (BITS == 4 ? 16.f : 64.f), f.y));
      }
    }
    __syncthreads();
  }
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
  auto compute = [&](const UnitLoads<RN>& L, const UnitCursor& c, auto lo_tag) {
    constexpr bool LOK = decltype(lo_tag)::value;  // (the loop where some group takes the second pass)
    const int gc = min(c.kc * kGroupsPerUnit + lane, G - 1);
    // (gc past the last group: its scale and bias were loaded as zero, whatever it reads here)
    float acc[RN];
    if constexpr (LOK) {
      const bool own_lo = gflag[gc] != 0;
      if (__any_sync(0xffffffffu, own_lo))
        dot(L, (uint32_t)gc * 128u, own_lo, std::true_type{}, acc);
      else
        dot(L, (uint32_t)gc * 128u, false, std::false_type{}, acc);
    } else {
      dot(L, (uint32_t)gc * 128u, false, std::false_type{}, acc);
    }
    const float2 gs = gsx[gc];  // the bias term takes the group's sum of its represented x
    float yp[RN];
#pragma unroll
    for (int e = 0; e < RN; ++e) yp[e] = fmaf(bf16_bits_to_f32(L.s[e]), acc[e] * gs.x, bf16_bits_to_f32(L.t[e]) * gs.y);
    store_rows(yp, c);
  };
  auto main_loop = [&](auto lo_tag) {
    for (; xok && u < nunits; u += NW) {
      const UnitCursor un = advance(uc);
      if (u + NW < nunits) issue(un, b1);
      compute(b0, uc, lo_tag);
      b0 = b1;
      uc = un;
    }
  };
  if (__builtin_expect(anylo, 0))
    main_loop(std::true_type{});
  else
    main_loop(std::false_type{});
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
  // K split: each CTA's row sums over its own chunks, then (after the cluster barrier) rank r
  // finishes its share of the cluster's rows, adding the C slices' sums in rank order.
  // (at the same offset in every CTA of the cluster: after the partial sums of the widest slice)
  float* rsum = part + (size_t)a.rows_per_cta * NC * ((nkc_all + C - 1) / C);  // [rows][NC], KS only
  int lr0 = 0, lr1 = ve - vb;
  if constexpr (KS) {
    for (int i = threadIdx.x; i < (ve - vb) * NC; i += kThreads) {
      float t = 0.f;
      for (int kc = 0; kc < nkc; ++kc) t += part[i * nkc + kc];
      rsum[i] = t;
    }
    cluster_sync();
    lr0 = rank * (ve - vb) / C;
    lr1 = (rank + 1) * (ve - vb) / C;
  }
  for (int lr = lr0 + (int)threadIdx.x; xok && lr < lr1; lr += kThreads) {
    const int v = vb + lr;
    int m = 0;
    while (m + 1 < a.nmat && v >= a.mat[m + 1].row0) ++m;
    const GemvMat& mt = a.mat[m];
    const int row = v - mt.row0;
    float acc = 0.f, up = 0.f;
    if constexpr (KS) {
      for (int c = 0; c < C; ++c) {
        acc += ld_peer_f32(rsum + lr * NC, (uint32_t)c);
        if (PAIR) up += ld_peer_f32(rsum + lr * NC + 1, (uint32_t)c);
      }
    } else {
      for (int kc = 0; kc < nkc; ++kc) acc += part[(lr * NC) * nkc + kc];
      if (PAIR)
        for (int kc = 0; kc < nkc; ++kc) up += part[(lr * NC + 1) * nkc + kc];
    }
    if (NORM) acc *= rn;
    if (PAIR) {
      if (NORM) up *= rn;
      bool ok = true;
      if (mt.w[0].slot >= 0) resolve(a, idxp, mt.w[0], ok);
      acc = ok ? acc / (1.f + expf(-acc)) * up : 0.f;
    }
    if (a.sgate) acc = fmaf(sig, acc, __ldg(a.ebase + row));
    if (a.resid) acc += bf16_bits_to_f32(a.resid[row]);
    mt.y[row] = acc;
  }
  if constexpr (KS) cluster_sync();  // (no CTA leaves while a peer may still read its row sums)
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
  int kcl;          // K split (cluster size): 0 automatic, 1 none, 2..8 forced where allowed
};
extern GemvTune g_gemv_tune;

// x of GS groups (the widest K slice), the partial sums of rows x NC components x the slice's chunks,
// and (K split) the row sums the cluster's CTAs read from each other.
inline size_t gemv_smem_bytes(int GS, int rows_per_cta, int nc, int kcl) {
  const int nkc = (GS + kGroupsPerUnit - 1) / kGroupsPerUnit;
  return (((size_t)GS * kXBytesPerGroup + 15) & ~(size_t)15) + (size_t)rows_per_cta * nc * nkc * 4 +
         (kcl > 1 ? (size_t)rows_per_cta * nc * 4 : 0);
}

// Shared memory with the x staging area after `base` bytes, or `base` alone (staging off).  Staged:
// x of up to 128 groups, and fp32 x of any length (the activations a previous kernel of the chain
// produced); long bf16 x is loaded by the threads.  Measured on the decode shapes: the bulk copy beat
// the threads' own loads for short x (gate/up 5120 bf16: 20.7 -> 20.1 us; MoE 2048 bf16 and 8 x 768
// fp32: 16.0 -> 14.9 us per layer); for the 17408-wide down x it loses standalone (bf16 12.9 -> 13.3
// us) but wins in the dense layer, where x is the gate/up kernel's fresh output (36.6 -> 34.9 us).
constexpr int kStageMaxGroups = 128;
inline size_t plan_stage(GemvArgs& a, size_t base, size_t limit) {
  const size_t off = (base + 127) & ~(size_t)127;
  const size_t total = off + (size_t)a.slice_groups * ((a.xf32 ? 256 : 128) + (a.gamma ? 128 : 0));
  a.stage = total <= limit && (a.slice_groups <= kStageMaxGroups || a.xf32) ? 1 : 0;
  a.stage_off = a.stage ? (int)off : 0;
  return a.stage ? total : base;
}
constexpr size_t kStaticSmemReserve = 8192;  // the kernels' static shared variables (NORM: 4.2 KB)
constexpr int kGemvDevs = 64;

// How many clusters of C CTAs of the GEMV kernel (512 threads, one CTA per SM) can be resident at
// once on the current device (cudaOccupancyMaxActiveClusters), cached per device and C.  A K-split
// grid never asks for more, so no cluster waits for a second wave.
int gemv_max_clusters(int dev, int C);

// The kernel's dynamic shared-memory limit is raised once per device (an attribute of the function
// in that device's context), to the largest size launched there so far.
template <int MODE, int RN, bool STG, bool NORM, int BITS = 4, bool KS = false>
int launch_gemv_variant(const GemvArgs& a, int grid, size_t smem, cudaStream_t stream) {
  auto k = gemv_kernel<MODE, RN, STG, NORM, BITS, KS>;
  static std::atomic<int> smem_set[kGemvDevs];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kGemvDevs) return QG_EDEVICE;
  if ((int)smem > smem_set[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return QG_ELAUNCH;
    smem_set[dev].store((int)smem, std::memory_order_relaxed);
  }
  return launch_cluster(k, dim3(grid), dim3(kThreads), smem, stream, KS ? a.kcl : 1, a);
}

// The per-shape plan: the grid (one CTA per SM), the K split across a cluster of C CTAs and with
// it each CTA's row range and K slice, and the shared memory.  Costs, in units of the time a warp
// takes for one work unit (about 1.5 us on the decode shapes): the units of the busiest warp, the
// x conversion of the widest slice (about a quarter unit per 64 groups of x on 512 threads), and
// the cluster's start (its CTAs wait for as many free SMs of one GPC), two barriers and row-sum
// exchange (about one unit: a forced split of the 5120 x 17408 GEMV cost 1.3 us).
struct GemvPlan {
  int grid, kcl, rows_per_cta, slice_groups;
  double cost;
};
inline GemvPlan gemv_plan_for(int total_rows, int groups, int nc, int rb, int C, int num_sms, int max_cl) {
  GemvPlan p{};
  const int ncl = std::max(1, std::min(C > 1 ? max_cl : num_sms, std::min(num_sms / C, total_rows)));
  p.grid = ncl * C;
  p.kcl = C;
  p.rows_per_cta = (total_rows + ncl - 1) / ncl;
  const int nkc_all = (groups + kGroupsPerUnit - 1) / kGroupsPerUnit;
  const int nkc_max = (nkc_all + C - 1) / C;
  p.slice_groups = std::min(groups, nkc_max * kGroupsPerUnit);
  const int units = (p.rows_per_cta + rb - 1) / rb * nkc_max;
  p.cost = (double)((units + kThreads / 32 - 1) / (kThreads / 32)) + 0.25 * (p.slice_groups + 63) / 64 +
           (C > 1 ? 1.0 : 0.0);
  return p;
}

void gemv_debug_plan(int mode, const GemvArgs& a, int grid, size_t smem);

// Plan (grid, K split, shared memory) and launch.
template <int MODE>
int plan_and_launch(GemvArgs& a, cudaStream_t stream) {
  const DeviceInfo& dev = device_info();
  constexpr int NC = mode_pair(MODE) ? 2 : 1;
  constexpr int RB = 4 / NC;
  a.groups = a.nseg * a.in / 64;
  const int cps = g_gemv_tune.ctas_per_sm ? g_gemv_tune.ctas_per_sm : 1;
  const size_t limit = (size_t)dev.max_smem_optin - kStaticSmemReserve;
  // K split: not with a norm prologue (its sums of squares and per-head roots span all of x), and
  // only when every CTA of the cluster gets at least one chunk of K
  const int nkc_all = (a.groups + kGroupsPerUnit - 1) / kGroupsPerUnit;
  int best_c = 1;
  GemvPlan best = gemv_plan_for(a.total_rows, a.groups, NC, RB, 1, cps * dev.num_sms, 0);
  const int forced = g_gemv_tune.kcl;
  if (!a.gamma && cps == 1 && nkc_all >= 2 && forced != 1) {
    for (int C = 2; C <= 4; ++C) {
      if (C > nkc_all || (forced && forced != C)) continue;
      const int mc = gemv_max_clusters(dev.id, C);
      if (mc < 1) continue;
      const GemvPlan p = gemv_plan_for(a.total_rows, a.groups, NC, RB, C, dev.num_sms, mc);
      if (forced == C || p.cost < best.cost) {
        best = p;
        best_c = C;
      }
    }
  }
  int grid = best.grid;
  a.kcl = best_c;
  a.slice_groups = best.slice_groups;
  a.rows_per_cta = best.rows_per_cta;
  // keep x and the partial-sum buffer within the shared memory (more, smaller CTAs otherwise;
  // unsplit only)
  while (a.kcl == 1 && gemv_smem_bytes(a.slice_groups, a.rows_per_cta, NC, 1) > limit && grid < a.total_rows) {
    grid = std::min(a.total_rows, grid * 2);
    a.rows_per_cta = (a.total_rows + grid - 1) / grid;
  }
  const size_t smem = plan_stage(a, gemv_smem_bytes(a.slice_groups, a.rows_per_cta, NC, a.kcl), limit);
  if (smem > limit) return QG_ENOTSUP;
  gemv_debug_plan(MODE, a, grid, smem);
  // rows x components per work unit: 4 (dense and seg: four rows; pair: two rows, gate and up)
  if (a.bits == 2) {
    if (a.gamma) return QG_ENOTSUP;
    if (a.kcl > 1)
      return a.stage ? launch_gemv_variant<MODE, 4, true, false, 2, true>(a, grid, smem, stream)
                     : launch_gemv_variant<MODE, 4, false, false, 2, true>(a, grid, smem, stream);
    return a.stage ? launch_gemv_variant<MODE, 4, true, false, 2>(a, grid, smem, stream)
                   : launch_gemv_variant<MODE, 4, false, false, 2>(a, grid, smem, stream);
  }
  if (a.kcl > 1)  // (never with a norm prologue)
    return a.stage ? launch_gemv_variant<MODE, 4, true, false, 4, true>(a, grid, smem, stream)
                   : launch_gemv_variant<MODE, 4, false, false, 4, true>(a, grid, smem, stream);
  if constexpr (MODE == kDense || MODE == kPair) {
    if (a.gamma)
      return a.stage ? launch_gemv_variant<MODE, 4, true, true>(a, grid, smem, stream)
                     : launch_gemv_variant<MODE, 4, false, true>(a, grid, smem, stream);
  }
  return a.stage ? launch_gemv_variant<MODE, 4, true, false>(a, grid, smem, stream)
                 : launch_gemv_variant<MODE, 4, false, false>(a, grid, smem, stream);
}

}  // namespace qg
