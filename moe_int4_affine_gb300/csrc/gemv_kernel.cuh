// gemv_kernel.cuh -- the streaming int4 affine dequant-GEMV kernel (M = 1), shared by three uses:
//   * dense: one matrix, or n in {2,3,4} matrices sharing one input vector ([FFAI#14]
//     "dequant_gemv_int4_*", "dequantGemvInt4Two/Three/Four", "ffai_batched_qkv_qgemv_fast",
//     "ffai_batched_4_qgemv_fast");
//   * pair: gate/up matrices reduced with SwiGLU, h = silu(W_g x) * (W_u x) -- a dense gate/up
//     pair, or the k selected experts' gate/up slabs picked on the device from the router's index
//     array ([FFAI#14] commit "moeRouterTopK / dequantGemvInt4ExpertIndexed");
//   * seg (MoE down): one output row is the concatenation of the k selected experts' down rows,
//     the input the concatenation of p_k * h_k, and the residual is added on the way out
//     ([FFAI#14] commit "ffai_moe_down_swiglu_accum_int4_chain8").
//
// Each weight is  w[r][j] = scale[r][j/64] * q[r][j] + bias[r][j/64]  (q = nibble j of row r, low
// nibble first), and each output an fp32 dot product with x.
//
// Design (GB300, sm_103a)
//   * Persistent grid, one CTA per SM, sized to leave room on every SM for one CTA of the next
//     launch (registers, shared memory, threads), so that with programmatic dependent launch the
//     next GEMV streams its first weights while this one finishes.  The flattened row space is
//     split into contiguous ranges, one per CTA; a CTA's rows of one matrix are one contiguous byte
//     range of packed codes, scales and biases.
//   * Warp 0 is the producer: lane 0 streams row blocks ("stages") through a shared-memory ring
//     with 1-D bulk copies (TMA engine, L2 evict-first), several stages ahead.  Compute warps
//     hand a ring slot back as soon as its data is in registers.  Warp 1 is the finisher: it sums
//     each stage's per-warp partial sums in a fixed order (deterministic), applies the epilogue
//     (SwiGLU / residual) and writes the outputs, off the refill path.
//   * Compute lanes own fixed 64-column units of x (one quantization group each) for the whole
//     kernel.  Each unit of x is held as 16-bit fixed point: X_j = round(x_j * 2^k) with 2^k chosen so the unit's largest |x| is in
//     [2^14, 2^15) (bf16 x: exact for every element within 2^7 of the unit's largest; otherwise
//     |X_j - x_j 2^k| <= 1/2).
//   * Unpack + dot: one shift and two ANDs turn a u32 word into eight unsigned byte codes; integer
//     dp2a instructions accumulate q_j * X_j exactly in int32, two products per instruction.  Per
//     group and row the scale and bias are applied once in fp32:
//        y += s * (acc * 2^-k) + b * sum_j x_j.
//   * Programmatic dependent launch: weights are streamed before griddepcontrol.wait; x, the router
//     outputs and all outputs are touched only after it.
#pragma once
#include <algorithm>
#include <atomic>
#include <utility>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int kMaxMats = 8;
enum GemvMode { kDense = 0, kPair = 1, kSeg = 2 };

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
  int in;                             // columns of one segment
  int units;                          // nseg * in / 64
  int total_rows;
  int rt;  // rows per stage
  int nstage;
  int pf;  // stages of L2 prefetch ahead of the ring
  int ngr, wpg;
  int q;                // row alignment quantum of stage starts and sizes
  uint32_t slot_bytes;  // packed bytes per ring slot
  uint32_t sb_bytes;    // scale bytes per ring slot (same for biases); 0 when not staged
};

struct Stage {
  int m, lr, n;
};

__device__ __forceinline__ bool next_stage(const GemvArgs& a, int& v, int ve, Stage& s) {
  if (v >= ve) return false;
  int m = 0;
  while (m + 1 < a.nmat && v >= a.mat[m + 1].row0) ++m;
  const int lr = v - a.mat[m].row0;
  s.m = m;
  s.lr = lr;
  s.n = min(a.rt, min(ve - v, a.mat[m].out - lr));
  v += s.n;
  return true;
}

struct WPtr {
  const uint32_t* packed;
  const uint16_t* scales;
  const uint16_t* biases;
};

// Resolve a weight reference to this call's slab.  `ok` is false for an out-of-range index.
__device__ __forceinline__ WPtr resolve(const GemvArgs& a, const WRef& r, bool& ok) {
  ok = true;
  if (r.slot < 0) return WPtr{r.packed, r.scales, r.biases};
  const uint32_t e = __ldg(a.idx + r.slot);
  if (e >= (uint32_t)a.n_experts) {
    ok = false;
    return WPtr{r.packed, r.scales, r.biases};
  }
  return WPtr{r.packed + (size_t)e * a.slab_words, r.scales + (size_t)e * a.slab_groups,
              r.biases + (size_t)e * a.slab_groups};
}

// Sums of RB per-lane values across the warp.  RB = 4: lane l returns the total of value
// (l >> 3) & 3; RB = 2: lane l returns the total of value (l >> 4) & 1.
template <int RB>
__device__ __forceinline__ float warp_sum_rows(const float (&v)[RB], int lane) {
  if constexpr (RB == 4) {
    const bool b4 = lane & 16, b3 = lane & 8;
    const float a0 = (b4 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, b4 ? v[0] : v[2], 16);
    const float a1 = (b4 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, b4 ? v[1] : v[3], 16);
    float c = (b3 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, b3 ? a0 : a1, 8);
    c += __shfl_xor_sync(0xffffffffu, c, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    return c;
  } else {
    const bool b4 = lane & 16;
    float c = (b4 ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, b4 ? v[0] : v[1], 16);
    c += __shfl_xor_sync(0xffffffffu, c, 8);
    c += __shfl_xor_sync(0xffffffffu, c, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    return c;
  }
}
template <int RB>
__device__ __forceinline__ int row_of_lane(int lane) {
  return RB == 4 ? (lane >> 3) & 3 : (lane >> 4) & 1;
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

// One lane's 64-column unit of x (one quantization group) in 16-bit fixed point, paired for
// dot_rows: per 8-column word w, p[w][0] = (X0, X2), p[w][1] = (X4, X6), p[w][2] = (X1, X3),
// p[w][3] = (X5, X7) (low half first).  Words are stored in the lane's load order: lanes with
// bit 2 set read the unit's second 16-byte chunk first (that keeps a warp's 16-byte shared-memory
// loads free of bank conflicts), so for them p[0..3] hold words 4..7 and p[4..7] words 0..3.
struct XUnit {
  uint32_t p[8][4];
  float sc;  // 2^-k, times the slot weight in seg mode
  float sx;  // sum of the unscaled x values, times the slot weight in seg mode
};

// 16-bit fixed point by the magic-number rule: for |t| < 2^22, t + 1.5 * 2^23 rounded to float
// has the nearest integer to t in its low mantissa bits.
__device__ __forceinline__ int round_to_int(float v, float scale) {
  return __float_as_int(fmaf(v, scale, 12582912.0f)) - 0x4B400000;
}

// The 8 x values of word wd (columns 8 wd .. 8 wd + 7 of the unit), as floats.
__device__ __forceinline__ void load_x_word(const void* xp, bool xf32, int u, int wd, float (&c)[8]) {
  if (!xf32) {
    const uint4 t = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(xp) + (size_t)u * 64) + wd);
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      c[2 * i] = __uint_as_float(w[i] << 16);
      c[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(xp) + (size_t)u * 64) + 2 * wd;
    const float4 t0 = __ldg(p), t1 = __ldg(p + 1);
    c[0] = t0.x, c[1] = t0.y, c[2] = t0.z, c[3] = t0.w, c[4] = t1.x, c[5] = t1.y, c[6] = t1.z, c[7] = t1.w;
  }
}

// Two passes over the unit's 64 values (the second re-reads them from L1): the largest magnitude
// and the sum, then the 16-bit fixed-point words in the lane's load order.
__device__ __forceinline__ void load_x_unit(const void* xp, bool xf32, int u, bool swap, float wgt, XUnit& X) {
  float m = 0.f, sx = 0.f;
#pragma unroll
  for (int wd = 0; wd < 8; ++wd) {
    float c[8];
    load_x_word(xp, xf32, u, wd, c);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      m = fmaxf(m, fabsf(c[i]));
      sx += c[i];
    }
  }
  // E = floor(log2 max|x|), k = 14 - E: |x| * 2^k < 2^15.  Units whose largest |x| is below 2^-60
  // contribute less than 1e-17 per weight through the code term and are dropped from it (the bias
  // term keeps the exact sum).
  const bool live = m >= 8.673617e-19f;  // 2^-60
  const int E = max((int)((__float_as_uint(m) >> 23) & 0xFF) - 127, -60);
  const float scale = live ? exp2i(14 - E) : 0.f;  // 14 - E in [-113, 74]
#pragma unroll
  for (int wd = 0; wd < 8; ++wd) {
    float c[8];
    load_x_word(xp, xf32, u, swap ? (wd ^ 4) : wd, c);
    int q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = max(-32767, min(32767, round_to_int(c[i], scale)));
    X.p[wd][0] = (uint32_t)(q[0] & 0xFFFF) | ((uint32_t)q[2] << 16);
    X.p[wd][1] = (uint32_t)(q[4] & 0xFFFF) | ((uint32_t)q[6] << 16);
    X.p[wd][2] = (uint32_t)(q[1] & 0xFFFF) | ((uint32_t)q[3] << 16);
    X.p[wd][3] = (uint32_t)(q[5] & 0xFFFF) | ((uint32_t)q[7] << 16);
  }
  X.sc = live ? exp2i(E - 14) * wgt : 0.f;  // E - 14 in [-74, 113]
  X.sx = sx * wgt;
}

// For RB rows at once: acc[r] = sum over the 64 codes of row r's 32-byte chunk pair of q_j * X_j
// (exact in int32: |acc| <= 64 * 15 * 32767 < 2^25, and the two partial sums each < 2^24 convert
// to float exactly).
template <int RB>
__device__ __forceinline__ void dot_rows(const uint4 (&wa)[RB], const uint4 (&wb)[RB], const XUnit& X,
                                         float (&acc)[RB]) {
  int s0[RB], s1[RB];
#pragma unroll
  for (int r = 0; r < RB; ++r) s0[r] = s1[r] = 0;
#pragma unroll
  for (int wd = 0; wd < 8; ++wd) {
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const uint4& c = wd < 4 ? wa[r] : wb[r];
      const int e = wd & 3;
      const uint32_t w = e == 0 ? c.x : e == 1 ? c.y : e == 2 ? c.z : c.w;
      const uint32_t c0 = w & 0x0F0F0F0Fu;         // codes q0, q2, q4, q6 as bytes
      const uint32_t c1 = (w >> 4) & 0x0F0F0F0Fu;  // codes q1, q3, q5, q7
      s0[r] = dp2a_lo(X.p[wd][0], c0, s0[r]);
      s1[r] = dp2a_hi(X.p[wd][1], c0, s1[r]);
      s0[r] = dp2a_lo(X.p[wd][2], c1, s0[r]);
      s1[r] = dp2a_hi(X.p[wd][3], c1, s1[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < RB; ++r) acc[r] = __int2float_rn(s0[r]) + __int2float_rn(s1[r]);
}

// Threads and minimum CTAs per SM of each variant: every variant leaves room on the SM for one CTA
// of the next launch, except the 4-units-per-lane variant for very wide rows.
template <int UPL>
constexpr int max_threads() {
  return 352;
}
template <int UPL>
constexpr int min_blocks() {
  return UPL == 4 ? 1 : 2;
}

// UPL: x units per lane.  RB: rows per register batch.  SBTMA: scales/biases staged by bulk
// copies (else read from global by the compute lanes).  MODE: dense, pair or seg.
template <int UPL, int RB, bool SBTMA, int MODE>
__global__ void __launch_bounds__(max_threads<UPL>(), min_blocks<UPL>()) gemv_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool PAIR = MODE == kPair, SEG = MODE == kSeg;
  constexpr int NC = PAIR ? 2 : 1;  // weight components per row
  const int S = a.nstage;
  const int NP = SEG ? a.nseg : NC;  // copies per stage (segments or components)
  const uint32_t row_bytes = (uint32_t)a.in / 2;
  const uint32_t sb_row = (uint32_t)a.in / 32;
  const int ngroups = a.in / 64;
  const int useg = a.in / 64;  // units (64-column groups) per segment
  uint8_t* ring = smem;
  uint8_t* sring = ring + (size_t)S * a.slot_bytes;
  uint8_t* bring = sring + (size_t)S * a.sb_bytes;
  float* red = reinterpret_cast<float*>(bring + (size_t)S * a.sb_bytes);
  const int red_slot = a.rt * NC * a.wpg;  // partial sums of one stage; R = 2S buffers, round robin
  const int R = 2 * S;
  uint64_t* full = reinterpret_cast<uint64_t*>(red + (((size_t)R * red_slot + 3) & ~(size_t)3));
  uint64_t* empty = full + S;  // ring slot free again (its data has been read into registers)
  uint64_t* done = empty + S;  // stage's partial sums written (R barriers, one per buffer)
  uint64_t* freed = done + R;  // stage finished: its partial-sum buffer may be reused (R barriers)
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = a.ngr * a.wpg;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, nw);
    }
    for (int s = 0; s < R; ++s) {
      mbar_init(done + s, nw);
      mbar_init(freed + s, 1);
    }
    mbar_fence_init();
    s_abort = 0;
  }
  // every thread signals: the next kernel in the stream may launch now (its CTAs take the room each
  // SM has left beside this one and start streaming their own weights)
  pdl_trigger();
  __syncthreads();

  // CTA row range, aligned to the quantum q (every matrix's row count is a multiple of q when
  // SBTMA is set; otherwise q == 1).
  const int nq = a.total_rows / a.q;
  const int vb = (int)((long long)blockIdx.x * nq / gridDim.x) * a.q;
  const int ve =
      blockIdx.x + 1 == gridDim.x ? a.total_rows : (int)((long long)(blockIdx.x + 1) * nq / gridDim.x) * a.q;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    if (a.idx) pdl_wait();  // expert indices come from the preceding kernel
    // Byte ranges of stage st, component/segment c (false for a skipped expert).
    auto ranges = [&](const Stage& st, int c, const uint32_t*& pk, const uint16_t*& sc, const uint16_t*& bi) {
      bool ok;
      const WPtr w = resolve(a, SEG ? WRef{a.seg.packed, a.seg.scales, a.seg.biases, c} : a.mat[st.m].w[c], ok);
      pk = w.packed + (size_t)st.lr * (a.in / 8);
      sc = w.scales + (size_t)st.lr * ngroups;
      bi = w.biases + (size_t)st.lr * ngroups;
      return ok;
    };
    // L2 prefetch runs a.pf stages ahead of the shared-memory ring: the ring only has to cover the
    // L2 -> SM latency while many more bytes are in flight from HBM.
    int vp = vb, tp = 0;
    Stage sp;
    auto prefetch_to = [&](int upto) {
      while (tp < upto && next_stage(a, vp, ve, sp)) {
        if (lane < NP) {
          const uint32_t *pk;
          const uint16_t *sc, *bi;
          if (ranges(sp, lane, pk, sc, bi)) {
            bulk_prefetch_l2(pk, (uint32_t)sp.n * row_bytes);
            if (SBTMA) {
              bulk_prefetch_l2(sc, (uint32_t)sp.n * sb_row);
              bulk_prefetch_l2(bi, (uint32_t)sp.n * sb_row);
            }
          }
        }
        ++tp;
      }
    };
    prefetch_to(a.pf);
    int v = vb, t = 0;
    Stage st;
    bool ok_run = true;
    while (next_stage(a, v, ve, st)) {
      const int slot = t % S;
      if (t >= S && (!mbar_wait(empty + slot, ((t / S) - 1) & 1) || s_abort)) {
        ok_run = false;
        break;
      }
      if (t >= R && (!mbar_wait(freed + t % R, ((t / R) - 1) & 1) || s_abort)) {
        ok_run = false;
        break;
      }
      if (lane == 0) {
        const uint32_t pbytes = (uint32_t)st.n * row_bytes;
        const uint32_t sbytes = SBTMA ? (uint32_t)st.n * sb_row : 0u;
        uint32_t tx = 0;
        for (int c = 0; c < NP; ++c) {
          const uint32_t *pk;
          const uint16_t *sc, *bi;
          if (ranges(st, c, pk, sc, bi)) tx += pbytes + 2 * sbytes;
        }
        if (tx)
          mbar_arrive_expect_tx(full + slot, tx);
        else
          mbar_arrive(full + slot);
        for (int c = 0; c < NP; ++c) {
          const uint32_t *pk;
          const uint16_t *sc, *bi;
          if (!ranges(st, c, pk, sc, bi)) continue;
          bulk_g2s_hint(ring + (size_t)slot * a.slot_bytes + (size_t)c * a.rt * row_bytes, pk, pbytes, full + slot, pol);
          if (SBTMA) {
            bulk_g2s_hint(sring + (size_t)slot * a.sb_bytes + (size_t)c * a.rt * sb_row, sc, sbytes, full + slot, pol);
            bulk_g2s_hint(bring + (size_t)slot * a.sb_bytes + (size_t)c * a.rt * sb_row, bi, sbytes, full + slot, pol);
          }
        }
      }
      __syncwarp();
      ++t;
      prefetch_to(t + a.pf);
    }
    if (!ok_run) {
      s_abort = 1;
      // a wait gave up: let this CTA's bulk copies land before it exits (bounded waits)
      for (int j = max(0, t - S); j < t; ++j) mbar_wait(full + j % S, (j / S) & 1);
    }
    return;
  }
  if (warp == 1) {
    // ------------------------------------------------------------ finisher
    // Stage by stage, in order: wait for its partial sums, add them in a fixed order
    // (deterministic), apply the epilogue, write the outputs, and free the buffer.
    pdl_wait();  // outputs may be read by the preceding kernel
    int v = vb, tf = 0;
    Stage sf;
    while (next_stage(a, v, ve, sf)) {
      const int rb = tf % R;
      if (!mbar_wait(done + rb, (tf / R) & 1) || s_abort) {
        s_abort = 1;
        return;
      }
      const float* rs = red + (size_t)rb * red_slot;
      const GemvMat& mt = a.mat[sf.m];
      bool ok = true;
      if (PAIR && mt.w[0].slot >= 0) resolve(a, mt.w[0], ok);
      for (int i = lane; i < sf.n; i += 32) {
        float acc = 0.f;
        for (int w = 0; w < a.wpg; ++w) acc += rs[i * a.wpg + w];
        if (PAIR) {
          float u = 0.f;
          for (int w = 0; w < a.wpg; ++w) u += rs[(a.rt + i) * a.wpg + w];
          acc = ok ? acc / (1.f + expf(-acc)) * u : 0.f;
        }
        if (SEG && a.resid) acc += bf16_bits_to_f32(a.resid[sf.lr + i]);
        mt.y[sf.lr + i] = acc;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(freed + rb);
      ++tf;
    }
    return;
  }

  // -------------------------------------------------------------- compute warps
  const int w = warp - 2;
  const int g = w / a.wpg, wig = w % a.wpg;
  int u[UPL];
  bool uv[UPL];
  pdl_wait();
#pragma unroll
  for (int k = 0; k < UPL; ++k) {
    u[k] = wig * 32 + lane + k * a.wpg * 32;
    uv[k] = u[k] < a.units;
  }
  XUnit X[UPL];
#pragma unroll
  for (int k = 0; k < UPL; ++k) {
    if (!uv[k]) continue;
    float wgt = 1.f;
    if (SEG) {
      const int s = u[k] / useg;
      bool ok;
      resolve(a, WRef{a.seg.packed, a.seg.scales, a.seg.biases, s}, ok);
      if (!ok) {
        uv[k] = false;
        if (blockIdx.x == 0 && (u[k] % useg) == 0) set_status(QG_STATUS_BAD_EXPERT);
        continue;
      }
      wgt = __ldg(a.p + s);
    }
    load_x_unit(a.x, a.xf32 != 0, u[k], (lane >> 2) & 1, wgt, X[k]);
  }
  if (PAIR && a.idx && blockIdx.x == 0 && w == 0 && lane < a.nmat) {
    if (__ldg(a.idx + lane) >= (uint32_t)a.n_experts) set_status(QG_STATUS_BAD_EXPERT);
  }
  // per-unit offsets inside a ring slot (seg mode: the segment's block of rows); the lane's two
  // 16-byte chunks of a row are read in swizzled order (see XUnit)
  const bool swap = (lane >> 2) & 1;
  uint32_t woff[UPL], soff[UPL];
#pragma unroll
  for (int k = 0; k < UPL; ++k) {
    // lanes past the last unit read (and ignore) the last unit's bytes, so every shared-memory
    // load stays inside the ring slot
    const int uc = min(u[k], a.units - 1);
    const int sg = SEG ? uc / useg : 0;
    const int lu = SEG ? uc - sg * useg : uc;
    woff[k] = (uint32_t)sg * a.rt * row_bytes + (uint32_t)lu * 32u;
    soff[k] = 2u * ((uint32_t)sg * a.rt * ngroups + (uint32_t)lu);
  }
  const uint32_t off_a = swap ? 16u : 0u, off_b = swap ? 0u : 16u;
  const uint32_t ring_s = smem_u32(ring), sring_s = smem_u32(sring);
  const uint32_t bdelta = (uint32_t)(bring - sring);  // biases sit at a fixed offset from scales
  constexpr int JB = RB / NC;                          // rows per batch (each with NC components)
  const uint32_t srow_bytes = 2u * ngroups;

  int v = vb, slot = 0, t = 0;
  uint32_t phase = 0;
  Stage st;
  while (next_stage(a, v, ve, st)) {
    if (!mbar_wait(full + slot, phase) || s_abort) {
      s_abort = 1;
      return;
    }
    const uint32_t wbase = ring_s + (uint32_t)slot * a.slot_bytes;
    const uint32_t sbase = sring_s + (uint32_t)slot * a.sb_bytes;
    float* rs = red + (size_t)(t % R) * red_slot;
    bool released = false;
    for (int j0 = 0; g + a.ngr * j0 < st.n; j0 += JB) {
      // batch entry r: row i = g + ngr * (j0 + r / NC), component r % NC, at slot row
      // (r % NC) * rt + i.  Rows past the stage are clamped to its last row and not stored.
      uint32_t srow[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const int i = min(g + a.ngr * (j0 + r / NC), st.n - 1);
        srow[r] = (uint32_t)((r % NC) * a.rt + i);
      }
      const bool last_batch = g + a.ngr * (j0 + JB) >= st.n;
      float yp[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) yp[r] = 0.f;
#pragma unroll
      for (int k = 0; k < UPL; ++k) {
        uint4 wa[RB], wb[RB];
        float sv[RB], bv[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const uint32_t wad = wbase + srow[r] * row_bytes + woff[k];
          wa[r] = lds128(wad + off_a);  // the lane's first 16-byte chunk in load order
          wb[r] = lds128(wad + off_b);  // and the other one
          uint32_t sbits, bbits;
          if (SBTMA) {
            const uint32_t sa = sbase + srow[r] * srow_bytes + soff[k];
            sbits = lds16(sa);
            bbits = lds16(sa + bdelta);
          } else {
            const int c = r % NC;
            const int sg = SEG ? u[k] / useg : 0;
            bool ok;
            const WPtr pw = resolve(a, SEG ? WRef{a.seg.packed, a.seg.scales, a.seg.biases, sg} : a.mat[st.m].w[c], ok);
            const size_t gi = (size_t)(st.lr + (int)srow[r] - c * a.rt) * ngroups + (u[k] - sg * useg);
            sbits = ok && uv[k] ? __ldg(pw.scales + gi) : 0u;
            bbits = ok && uv[k] ? __ldg(pw.biases + gi) : 0u;
          }
          sv[r] = bf16_bits_to_f32(sbits);
          bv[r] = bf16_bits_to_f32(bbits);
        }
        if (k == UPL - 1 && last_batch) {
          // the stage's last data is in registers: hand the ring slot back to the producer
          __syncwarp();
          if (lane == 0) mbar_arrive(empty + slot);
          released = true;
        }
        if (!uv[k]) continue;
        float acc[RB];
        dot_rows<RB>(wa, wb, X[k], acc);
#pragma unroll
        for (int r = 0; r < RB; ++r) yp[r] = fmaf(sv[r], acc[r] * X[k].sc, fmaf(bv[r], X[k].sx, yp[r]));
      }
      const float tot = warp_sum_rows<RB>(yp, lane);
      if ((lane & (32 / RB - 1)) == 0) {
        const int r = row_of_lane<RB>(lane);
        const int i = g + a.ngr * (j0 + r / NC);
        if (i < st.n) rs[((r % NC) * a.rt + i) * a.wpg + wig] = tot;
      }
    }
    __syncwarp();
    if (lane == 0) {
      if (!released) mbar_arrive(empty + slot);
      mbar_arrive(done + t % R);
    }
    if (++slot == S) {
      slot = 0;
      phase ^= 1u;
    }
    ++t;
  }
}

// ------------------------------------------------------------------ host side: planning
struct GemvPlan {
  int upl, rb, ngr, wpg, rt, nstage, pf, grid, threads, q;
  bool sbtma;
  size_t smem;
  uint32_t slot_bytes, sb_bytes;
};

struct GemvTune {
  int upl, ngr, rt, nstage, cps, pf;
};
extern GemvTune g_gemv_tune;

inline int gcd_int(int x, int y) { return y ? gcd_int(y, x % y) : x; }

inline int plan_max_threads(int upl) { return 352; }

// Shared memory per CTA is kept under half an SM so one CTA of the next launch fits beside it.
constexpr size_t kSmemBudget = 104 * 1024;

inline GemvPlan plan_gemv(int in, int nseg, int total_rows, bool pair, const int* outs, int nmat) {
  const DeviceInfo& dev = device_info();
  const GemvTune tn = g_gemv_tune;
  GemvPlan p{};
  const int NC = pair ? 2 : 1;
  const int NP = nseg > 1 ? nseg : NC;
  const int units = nseg * in / 64;
  p.upl = tn.upl ? tn.upl : (units <= 11 * 32 ? 1 : (units <= 9 * 32 * 2 ? 2 : 4));
  const int lanes = (units + p.upl - 1) / p.upl;
  p.wpg = (lanes + 31) / 32;
  const int max_w = plan_max_threads(p.upl) / 32 - 2;  // minus the producer and finisher warps
  // Bulk copies of scales/biases need 16-byte multiples: stage starts and sizes are multiples of
  // q rows, which every matrix's row count must allow.
  const int sb_row = in / 32;
  p.q = 16 / gcd_int(sb_row, 16);
  p.sbtma = true;
  for (int i = 0; i < nmat; ++i) p.sbtma = p.sbtma && (outs[i] % p.q == 0);
  if (!p.sbtma) p.q = 1;
  const size_t row_bytes = (size_t)in / 2;
  const size_t vrow_bytes = NP * (row_bytes + 2 * (size_t)sb_row);
  // CTAs per SM: two when the rows allow, so each SM runs twice the warps (each CTA keeps under
  // half an SM, which also lets the next launch's CTAs start as these finish).
  int cps = tn.cps ? tn.cps : 1;
  const int ctas = cps * dev.num_sms;
  const int rows_per_cta = std::max(1, (total_rows + ctas - 1) / ctas);
  // Rows per register batch: 4, or 2 when four rows of this width make a stage above 24 KB.
  p.rb = 2;
  // Row groups: as many as the warp budget allows, no more than a stage of <= 24 KB feeds with one
  // batch each, and no more than the CTA has rows for.
  int ngr = std::max(1, std::min(8, max_w / std::max(1, p.wpg)));
  while (ngr > 1 && ((size_t)(ngr * p.rb / NC) * vrow_bytes > 24576 || ngr * p.rb / NC > 2 * rows_per_cta)) --ngr;
  if (tn.ngr) ngr = tn.ngr;
  int rt = std::max(1, ngr * p.rb / NC);  // every row group gets one batch per stage
  rt = std::min(rt, rows_per_cta);
  if (tn.rt) rt = tn.rt;
  rt = std::max(p.q, (rt + p.q - 1) / p.q * p.q);
  p.ngr = std::max(1, std::min(ngr, NC * rt));
  p.rt = rt;
  p.slot_bytes = (uint32_t)(rt * NP * row_bytes);
  p.sb_bytes = p.sbtma ? (uint32_t)(rt * NP * sb_row) : 0u;
  const size_t red_bytes = 2 * (size_t)rt * NC * p.wpg * 4;  // two partial-sum buffers per ring slot
  const size_t slot_all = p.slot_bytes + 2 * (size_t)p.sb_bytes + red_bytes;
  p.nstage = (int)std::max<size_t>(2, std::min<size_t>(8, kSmemBudget / slot_all));
  if (tn.nstage) p.nstage = tn.nstage;
  // L2 prefetch depth: about 384 KB of each CTA's stream beyond the ring (all of it for smaller
  // problems), so HBM sees several MB of outstanding reads per launch.
  p.pf = p.nstage + (int)std::max<size_t>(1, (384 * 1024) / (p.slot_bytes + 2 * (size_t)p.sb_bytes));
  if (tn.pf) p.pf = p.nstage + tn.pf;
  p.smem = p.nstage * slot_all + 16 + 6 * p.nstage * 8;
  const int nq = total_rows / p.q;
  p.grid = std::max(1, std::min(ctas, (nq * p.q + rt - 1) / rt));
  p.grid = std::min(p.grid, std::max(1, nq));
  p.threads = 32 * (2 + p.ngr * p.wpg);
  return p;
}

template <int UPL, int RB, bool SBTMA, int MODE>
int launch_gemv_variant(const GemvArgs& a, const GemvPlan& p, cudaStream_t stream) {
  auto k = gemv_kernel<UPL, RB, SBTMA, MODE>;
  static std::atomic<int> smem_set{0};
  if ((int)p.smem > smem_set.load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) != cudaSuccess)
      return QG_ELAUNCH;
    smem_set.store((int)p.smem, std::memory_order_relaxed);
  }
  return launch(k, dim3(p.grid), dim3(p.threads), p.smem, stream, a);
}

template <int MODE>
int dispatch_gemv(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
  const int key = (p.upl == 1 ? 0 : p.upl == 2 ? 1 : 2) * 2 + (p.sbtma ? 1 : 0);
  switch (key) {
    case 0: return launch_gemv_variant<1, 2, false, MODE>(a, p, s);
    case 1: return launch_gemv_variant<1, 2, true, MODE>(a, p, s);
    case 2: return launch_gemv_variant<2, 2, false, MODE>(a, p, s);
    case 3: return launch_gemv_variant<2, 2, true, MODE>(a, p, s);
    case 4: return launch_gemv_variant<4, 2, false, MODE>(a, p, s);
    default: return launch_gemv_variant<4, 2, true, MODE>(a, p, s);
  }
}

// Plan, fill in the plan fields of `a`, check limits and launch.
template <int MODE>
int plan_and_launch(GemvArgs& a, cudaStream_t stream) {
  int outs[kMaxMats];
  for (int i = 0; i < a.nmat; ++i) outs[i] = a.mat[i].out;
  const GemvPlan p = plan_gemv(a.in, a.nseg, a.total_rows, MODE == kPair, outs, a.nmat);
  if (p.threads > plan_max_threads(p.upl) || p.smem > (size_t)device_info().max_smem_optin) return QG_ENOTSUP;
  a.units = a.nseg * a.in / 64;
  a.rt = p.rt;
  a.nstage = p.nstage;
  a.pf = p.pf;
  a.ngr = p.ngr;
  a.wpg = p.wpg;
  a.q = p.q;
  a.slot_bytes = p.slot_bytes;
  a.sb_bytes = p.sb_bytes;
  return dispatch_gemv<MODE>(a, p, stream);
}

}  // namespace qg
