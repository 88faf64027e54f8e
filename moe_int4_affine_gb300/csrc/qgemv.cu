// qgemv.cu -- the streaming int4 affine dequant-GEMV kernel (M = 1) and its three uses:
//   * dense: one matrix, or n in {2,3,4} matrices sharing one input vector, optionally a
//     gate/up pair reduced with SwiGLU ([FFAI#14] "dequant_gemv_int4_*",
//     "dequantGemvInt4Two/Three/Four", "ffai_batched_qkv_qgemv_fast", "ffai_batched_4_qgemv_fast");
//   * MoE gate/up: the k selected experts' gate and up slabs, picked on the device from the
//     router's index array, reduced with SwiGLU into h[k][inter] ([FFAI#14] commit
//     "moeRouterTopK / dequantGemvInt4ExpertIndexed");
//   * MoE down: one output row is the concatenation of the k selected experts' down rows, the
//     input is the concatenation of p_k * h_k, and the residual is added on the way out
//     ([FFAI#14] commit "ffai_moe_down_swiglu_accum_int4_chain8").
//
// Each weight element is  w[r][j] = scale[r][j/64] * q[r][j] + bias[r][j/64]  (q = nibble j of
// the row, low nibble first) and each output is an fp32 dot product.
//
// Design (GB300, sm_103a)
//   * Persistent grid, at most one CTA per SM.  The flattened row space is split into contiguous
//     ranges, one per CTA; a CTA's rows of one matrix are one contiguous byte range of packed
//     codes, scales and biases.
//   * Warp 0 is the producer: lane 0 streams row blocks ("stages") through a shared-memory ring
//     with 1-D bulk copies (TMA engine, L2 evict-first), several stages ahead.  The same warp
//     finishes each stage: it sums the compute warps' partial sums in a fixed order
//     (deterministic), applies the epilogue (SwiGLU / residual) and writes the outputs.
//   * Compute lanes each own fixed 32-column units for the whole kernel, so x is read once per
//     CTA and lives in registers as f16 pairs.  Per unit the lane picks a power of two 2^e that
//     puts the unit's largest |x| in [2^14, 2^15): bf16 x is then exact in f16; fp32 x is carried
//     as an f16 hi/lo pair (about 22 significant bits).
//   * Unpack: each nibble is OR-ed into the f16 pattern of 1024.0 at bits 4..7, which reads
//     1024 + 16q exactly; the sm_100+ mixed-precision FMA (f16 x f16 product exact in fp32, fp32
//     accumulate) accumulates (1024 + 16q) * X.  Per unit and row the constant 1024 * sum(X) is
//     removed once and the group's scale and bias applied once:
//        y += s * (acc - 1024 * sum X) / (16 * 2^e) + b * sum x.
//   * Programmatic dependent launch: weights are streamed before griddepcontrol.wait; x, the
//     router outputs and all outputs are touched only after it.
#include <algorithm>
#include <atomic>
#include <utility>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int kRB = 4;  // rows per register batch
constexpr int kMaxMats = 8;

// A weight operand: base pointers of a (possibly stacked) weight, and the expert slot whose
// slab to use (-1: the base itself).
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
  WRef seg;               // segmented mode: the stacked weight whose slabs form the segments
  int nseg;               // segments per row (1 unless segmented)
  const void* x;          // [nseg][in] (bf16 or fp32)
  const uint32_t* idx;    // expert indices (device) or null
  const float* p;         // per-slot weights (segmented mode)
  const uint16_t* resid;  // residual added by the finisher (segmented mode) or null
  int n_experts;
  long long slab_words, slab_groups;  // per-expert strides of stacked weights
  int in;                             // columns of one segment
  int units;                          // nseg * in / 32
  int total_rows;
  int rt;  // rows per stage
  int nstage;
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

// Sum of four per-lane values across the warp; lane l returns the total of value (l >> 3) & 3.
__device__ __forceinline__ float warp_sum4(float v0, float v1, float v2, float v3, int lane) {
  const bool b4 = lane & 16, b3 = lane & 8;
  const float a0 = (b4 ? v2 : v0) + __shfl_xor_sync(0xffffffffu, b4 ? v0 : v2, 16);
  const float a1 = (b4 ? v3 : v1) + __shfl_xor_sync(0xffffffffu, b4 ? v1 : v3, 16);
  float c = (b3 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, b3 ? a0 : a1, 8);
  c += __shfl_xor_sync(0xffffffffu, c, 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

// One lane's 32-column unit of x: 16 f16x2 registers (pairs in the order nibbles_to_f16_magic
// produces), the fp32 low parts for fp32 x, and the unit's constants.
template <bool XF32>
struct XUnit {
  uint32_t hi[4][4];
  uint32_t lo[XF32 ? 4 : 1][XF32 ? 4 : 1];
  float sc;    // 1 / (16 * 2^e), times the slot weight in segmented mode
  float nksc;  // -1024 * sum(X) * sc
  float sx;    // sum of the unscaled x values, times the slot weight in segmented mode
};

template <bool XF32>
__device__ __forceinline__ void load_x_unit(const void* xp, int u, float wgt, XUnit<XF32>& X) {
  float v[32];
  if (!XF32) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(xp) + (size_t)u * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 t = __ldg(p + q);
      const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[q * 8 + 2 * i] = __uint_as_float(w[i] << 16);
        v[q * 8 + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(xp) + (size_t)u * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 t = __ldg(p + q);
      v[4 * q] = t.x;
      v[4 * q + 1] = t.y;
      v[4 * q + 2] = t.z;
      v[4 * q + 3] = t.w;
    }
  }
  float m = 0.f, sx = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    m = fmaxf(m, fabsf(v[i]));
    sx += v[i];
  }
  // E = floor(log2 max|x|).  Units whose largest |x| is below 2^-60 contribute less than 1e-17
  // per weight through the code term and are dropped from it (the bias term keeps the exact sum).
  const bool live = m >= 8.673617e-19f;  // 2^-60
  const int E = max((int)((__float_as_uint(m) >> 23) & 0xFF) - 127, -60);
  const int e = 14 - E;  // in [-114, 74]
  const float f1 = exp2i(e / 2), f2 = exp2i(e - e / 2);
  float ks = 0.f;
#pragma unroll
  for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = live ? (v[wd * 8 + i] * f1) * f2 : 0.f;
      const float b = live ? (v[wd * 8 + i + 4] * f1) * f2 : 0.f;
      const uint32_t h = pack_f16x2(a, b);
      X.hi[wd][i] = h;
      const float ah = f16_lo_to_f32(h), bh = f16_hi_to_f32(h);
      ks += ah + bh;
      if constexpr (XF32) {
        const uint32_t l = pack_f16x2(a - ah, b - bh);
        X.lo[wd][i] = l;
        ks += f16_lo_to_f32(l) + f16_hi_to_f32(l);
      }
    }
  }
  const float sc = live ? exp2i(E - 18) : 0.f;  // 2^(-4-e)
  X.sc = sc * wgt;
  X.nksc = -1024.f * ks * sc * wgt;
  X.sx = sx * wgt;
}

template <bool XF32>
__device__ __forceinline__ float dot_unit(const uint4& wv, const XUnit<XF32>& X) {
  float acc0 = 0.f, acc1 = 0.f;
  const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int wd = 0; wd < 4; ++wd) {
    uint32_t h[4];
    nibbles_to_f16_magic(w[wd], h);
    acc0 = fma2_f16_f32(h[0], X.hi[wd][0], acc0);
    acc1 = fma2_f16_f32(h[1], X.hi[wd][1], acc1);
    acc0 = fma2_f16_f32(h[2], X.hi[wd][2], acc0);
    acc1 = fma2_f16_f32(h[3], X.hi[wd][3], acc1);
    if constexpr (XF32) {
      acc0 = fma2_f16_f32(h[0], X.lo[wd][0], acc0);
      acc1 = fma2_f16_f32(h[1], X.lo[wd][1], acc1);
      acc0 = fma2_f16_f32(h[2], X.lo[wd][2], acc0);
      acc1 = fma2_f16_f32(h[3], X.lo[wd][3], acc1);
    }
  }
  return acc0 + acc1;
}

// UPL: x units per lane.  XF32: fp32 x.  SBTMA: scales/biases staged by bulk copies (else read
// from global by the compute lanes).  PAIR: gate/up pairs with SwiGLU.  SEG: segmented rows
// (MoE down).
// Thread cap per variant: one x unit per lane leaves room for 19 compute warps (registers capped at
// 102 per thread); more units per lane need more registers.
template <int UPL>
constexpr int max_threads() {
  return UPL == 1 ? 640 : 384;
}

template <int UPL, bool XF32, bool SBTMA, bool PAIR, bool SEG>
__global__ void __launch_bounds__(max_threads<UPL>(), 1) gemv_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NC = PAIR ? 2 : 1;  // weight components per row
  const int S = a.nstage;
  const int NP = SEG ? a.nseg : NC;  // copies per stage (segments or components)
  const uint32_t row_bytes = (uint32_t)a.in / 2;
  const uint32_t sb_row = (uint32_t)a.in / 32;
  const int ngroups = a.in / 64;
  const int useg = a.in / 32;  // units per segment
  uint8_t* ring = smem;
  uint8_t* sring = ring + (size_t)S * a.slot_bytes;
  uint8_t* bring = sring + (size_t)S * a.sb_bytes;
  float* red = reinterpret_cast<float*>(bring + (size_t)S * a.sb_bytes);
  const int red_slot = a.rt * NC * a.wpg;
  uint64_t* full = reinterpret_cast<uint64_t*>(red + (((size_t)S * red_slot + 3) & ~(size_t)3));
  uint64_t* empty = full + S;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = a.ngr * a.wpg;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, nw);
    }
    mbar_fence_init();
    s_abort = 0;
    pdl_trigger();
  }
  __syncthreads();

  // CTA row range, aligned to the quantum q (every matrix's row count is a multiple of q when
  // SBTMA is set; otherwise q == 1).
  const int nq = a.total_rows / a.q;
  const int vb = (int)((long long)blockIdx.x * nq / gridDim.x) * a.q;
  const int ve =
      blockIdx.x + 1 == gridDim.x ? a.total_rows : (int)((long long)(blockIdx.x + 1) * nq / gridDim.x) * a.q;

  if (warp == 0) {
    // ------------------------------------------------------------ producer + finisher
    const uint64_t pol = policy_evict_first();
    int v = vb, vf = vb, t = 0, tf = 0;
    bool waited = false;
    if (a.idx) {  // expert indices come from the preceding kernel: wait before resolving them
      pdl_wait();
      waited = true;
    }
    Stage st, sf;
    auto finish = [&](int slot, const Stage& s) {
      const float* rs = red + (size_t)slot * red_slot;
      const GemvMat& mt = a.mat[s.m];
      bool ok = true;
      if (PAIR && mt.w[0].slot >= 0) resolve(a, mt.w[0], ok);
      for (int i = lane; i < s.n; i += 32) {
        float acc = 0.f;
        for (int w = 0; w < a.wpg; ++w) acc += rs[i * a.wpg + w];
        if (PAIR) {
          float u = 0.f;
          for (int w = 0; w < a.wpg; ++w) u += rs[(a.rt + i) * a.wpg + w];
          acc = ok ? acc / (1.f + expf(-acc)) * u : 0.f;
        }
        if (SEG && a.resid) acc += bf16_bits_to_f32(a.resid[s.lr + i]);
        mt.y[s.lr + i] = acc;
      }
    };
    while (next_stage(a, v, ve, st)) {
      const int slot = t % S;
      if (t >= S) {
        if (!mbar_wait(empty + slot, ((t / S) - 1) & 1) || s_abort) {
          s_abort = 1;
          break;
        }
        if (!waited) {
          pdl_wait();
          waited = true;
        }
        next_stage(a, vf, ve, sf);
        finish(slot, sf);
        ++tf;
        __syncwarp();
      }
      if (lane == 0) {
        const uint32_t pbytes = (uint32_t)st.n * row_bytes;
        const uint32_t sbytes = SBTMA ? (uint32_t)st.n * sb_row : 0u;
        WPtr src[kMaxMats];
        bool ok[kMaxMats];
        uint32_t tx = 0;
        for (int c = 0; c < NP; ++c) {
          src[c] = resolve(a, SEG ? WRef{a.seg.packed, a.seg.scales, a.seg.biases, c} : a.mat[st.m].w[c], ok[c]);
          if (ok[c]) tx += pbytes + 2 * sbytes;
        }
        if (tx)
          mbar_arrive_expect_tx(full + slot, tx);
        else
          mbar_arrive(full + slot);
        for (int c = 0; c < NP; ++c) {
          if (!ok[c]) continue;
          bulk_g2s_hint(ring + (size_t)slot * a.slot_bytes + (size_t)c * a.rt * row_bytes,
                        src[c].packed + (size_t)st.lr * (a.in / 8), pbytes, full + slot, pol);
          if (SBTMA) {
            bulk_g2s_hint(sring + (size_t)slot * a.sb_bytes + (size_t)c * a.rt * sb_row,
                          src[c].scales + (size_t)st.lr * ngroups, sbytes, full + slot, pol);
            bulk_g2s_hint(bring + (size_t)slot * a.sb_bytes + (size_t)c * a.rt * sb_row,
                          src[c].biases + (size_t)st.lr * ngroups, sbytes, full + slot, pol);
          }
        }
      }
      __syncwarp();
      ++t;
    }
    if (!s_abort) {
      if (!waited) pdl_wait();
      for (; tf < t; ++tf) {
        const int slot = tf % S;
        if (!mbar_wait(empty + slot, (tf / S) & 1)) {
          s_abort = 1;
          break;
        }
        next_stage(a, vf, ve, sf);
        finish(slot, sf);
      }
    }
    return;
  }

  // -------------------------------------------------------------- compute warps
  const int w = warp - 1;
  const int g = w / a.wpg, wig = w % a.wpg;
  int u[UPL];
  bool uv[UPL];
  pdl_wait();
#pragma unroll
  for (int k = 0; k < UPL; ++k) {
    u[k] = wig * 32 + lane + k * a.wpg * 32;
    uv[k] = u[k] < a.units;
  }
  XUnit<XF32> X[UPL];
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
    load_x_unit<XF32>(a.x, u[k], wgt, X[k]);
  }
  if (PAIR && a.idx && blockIdx.x == 0 && w == 0 && lane < a.nmat) {
    if (__ldg(a.idx + lane) >= (uint32_t)a.n_experts) set_status(QG_STATUS_BAD_EXPERT);
  }

  int v = vb, t = 0;
  Stage st;
  while (next_stage(a, v, ve, st)) {
    const int slot = t % S;
    if (!mbar_wait(full + slot, (t / S) & 1) || s_abort) {
      s_abort = 1;
      return;
    }
    const uint8_t* buf = ring + (size_t)slot * a.slot_bytes;
    const uint16_t* sbuf = reinterpret_cast<const uint16_t*>(sring + (size_t)slot * a.sb_bytes);
    const uint16_t* bbuf = reinterpret_cast<const uint16_t*>(bring + (size_t)slot * a.sb_bytes);
    float* rs = red + (size_t)slot * red_slot;
    const int nwork = NC * st.n;  // work rows: component-major
    for (int i0 = 0; g + a.ngr * i0 < nwork; i0 += kRB) {
      float yp[kRB];
#pragma unroll
      for (int r = 0; r < kRB; ++r) yp[r] = 0.f;
#pragma unroll
      for (int k = 0; k < UPL; ++k) {
        if (!uv[k]) continue;
        const int sg = SEG ? u[k] / useg : 0;  // segment of this unit
        const int lu = SEG ? u[k] - sg * useg : u[k];
        uint4 wv[kRB];
        float sv[kRB], bv[kRB];
#pragma unroll
        for (int r = 0; r < kRB; ++r) {
          const int wr = g + a.ngr * (i0 + r);
          if (wr < nwork) {
            const int c = PAIR ? (wr >= st.n) : 0;
            const int i = wr - c * st.n;
            const int sr = (SEG ? sg : c) * a.rt + i;  // row index inside the ring slot
            wv[r] = *reinterpret_cast<const uint4*>(buf + (size_t)sr * row_bytes + (size_t)lu * 16);
            uint32_t sbits, bbits;
            if (SBTMA) {
              sbits = sbuf[sr * ngroups + (lu >> 1)];
              bbits = bbuf[sr * ngroups + (lu >> 1)];
            } else {
              bool ok;
              const WPtr pw =
                  resolve(a, SEG ? WRef{a.seg.packed, a.seg.scales, a.seg.biases, sg} : a.mat[st.m].w[c], ok);
              const size_t gi = (size_t)(st.lr + i) * ngroups + (lu >> 1);
              sbits = ok ? __ldg(pw.scales + gi) : 0u;
              bbits = ok ? __ldg(pw.biases + gi) : 0u;
            }
            sv[r] = bf16_bits_to_f32(sbits);
            bv[r] = bf16_bits_to_f32(bbits);
          } else {
            wv[r] = make_uint4(0u, 0u, 0u, 0u);
            sv[r] = 0.f;
            bv[r] = 0.f;
          }
        }
#pragma unroll
        for (int r = 0; r < kRB; ++r) {
          const float acc = dot_unit<XF32>(wv[r], X[k]);
          yp[r] += fmaf(sv[r], fmaf(acc, X[k].sc, X[k].nksc), bv[r] * X[k].sx);
        }
      }
      const float tot = warp_sum4(yp[0], yp[1], yp[2], yp[3], lane);
      if ((lane & 7) == 0) {
        const int wr = g + a.ngr * (i0 + (lane >> 3));
        if (wr < nwork) {
          const int c = PAIR ? (wr >= st.n) : 0;
          rs[(c * a.rt + wr - c * st.n) * a.wpg + wig] = tot;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + slot);
    ++t;
  }
}

// ------------------------------------------------------------------ host side
namespace {

struct GemvPlan {
  int upl, ngr, wpg, rt, nstage, grid, threads, q;
  bool sbtma;
  size_t smem;
  uint32_t slot_bytes, sb_bytes;
};

int gcd_int(int x, int y) { return y ? gcd_int(y, x % y) : x; }

struct Tune {
  int upl, ngr, rt, nstage;
};
Tune g_tune = {0, 0, 0, 0};

GemvPlan plan_gemv(int in, int nseg, int total_rows, bool pair, const int* outs, int nmat) {
  const DeviceInfo& dev = device_info();
  const Tune tn = g_tune;
  GemvPlan p{};
  const int NC = pair ? 2 : 1;
  const int NP = nseg > 1 ? nseg : NC;
  const int units = nseg * in / 32;
  // x units per lane: one while the row's units fit 19 warps, else two or four
  p.upl = tn.upl ? tn.upl : (units <= 19 * 32 ? 1 : (units <= 11 * 32 * 2 ? 2 : 4));
  const int lanes = (units + p.upl - 1) / p.upl;
  p.wpg = (lanes + 31) / 32;
  const int max_w = (p.upl == 1 ? 640 : 384) / 32 - 1;
  if (p.wpg > max_w) {
    p.upl = 4;
    p.wpg = (units + 127) / 128;
  }
  // Bulk copies of scales/biases need 16-byte multiples: stage starts and sizes are multiples of
  // q rows, which every matrix's row count must allow.
  const int sb_row = in / 32;
  p.q = 16 / gcd_int(sb_row, 16);
  p.sbtma = true;
  for (int i = 0; i < nmat; ++i) p.sbtma = p.sbtma && (outs[i] % p.q == 0);
  if (!p.sbtma) p.q = 1;
  const size_t row_bytes = (size_t)in / 2;
  const size_t vrow_bytes = NP * (row_bytes + 2 * (size_t)sb_row);
  const int rows_per_cta = std::max(1, (total_rows + dev.num_sms - 1) / dev.num_sms);
  // Row groups: as many as the warp budget allows, but no more than a stage of <= 48 KB can feed
  // with kRB rows each, and no more than the CTA has rows for.
  int ngr = std::max(1, std::min(8, (p.upl == 1 ? 640 : 384) / 32 / p.wpg - (p.wpg == 1 ? 1 : 0)));
  ngr = std::min(ngr, std::max(1, std::min(max_w / p.wpg, 8)));
  while (ngr > 1 && ((size_t)(ngr * kRB + NC - 1) / NC * vrow_bytes > 49152 ||
                     (ngr * kRB + NC - 1) / NC > 2 * rows_per_cta))
    --ngr;
  if (tn.ngr) ngr = tn.ngr;
  p.ngr = ngr;
  int rt = (ngr * kRB + NC - 1) / NC;  // every row group gets kRB work rows per stage
  rt = std::min(rt, rows_per_cta);
  if (tn.rt) rt = tn.rt;
  rt = std::max(p.q, (rt + p.q - 1) / p.q * p.q);
  p.rt = rt;
  p.ngr = std::max(1, std::min(p.ngr, NC * rt));
  p.slot_bytes = (uint32_t)(rt * NP * row_bytes);
  p.sb_bytes = p.sbtma ? (uint32_t)(rt * NP * sb_row) : 0u;
  const size_t red_bytes = (size_t)rt * NC * p.wpg * 4;
  const size_t slot_all = p.slot_bytes + 2 * (size_t)p.sb_bytes + red_bytes;
  const size_t budget = (size_t)std::min(dev.max_smem_optin, 200 * 1024) - 64;
  p.nstage = (int)std::max<size_t>(2, std::min<size_t>(8, budget / slot_all));
  if (tn.nstage) p.nstage = tn.nstage;
  p.smem = p.nstage * slot_all + 16 + 2 * p.nstage * 8;
  const int nq = total_rows / p.q;
  p.grid = std::max(1, std::min(dev.num_sms, (nq * p.q + rt - 1) / rt));
  p.grid = std::min(p.grid, std::max(1, nq));
  p.threads = 32 * (1 + p.ngr * p.wpg);
  return p;
}

template <int UPL, bool XF32, bool SBTMA, bool PAIR, bool SEG>
int launch_variant(const GemvArgs& a, const GemvPlan& p, cudaStream_t stream) {
  auto k = gemv_kernel<UPL, XF32, SBTMA, PAIR, SEG>;
  static std::atomic<int> smem_set{0};
  if ((int)p.smem > smem_set.load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) != cudaSuccess)
      return QG_ELAUNCH;
    smem_set.store((int)p.smem, std::memory_order_relaxed);
  }
  return launch(k, dim3(p.grid), dim3(p.threads), p.smem, stream, a);
}

template <int UPL, bool XF32, bool PAIR, bool SEG>
int dispatch_sb(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
  return p.sbtma ? launch_variant<UPL, XF32, true, PAIR, SEG>(a, p, s)
                 : launch_variant<UPL, XF32, false, PAIR, SEG>(a, p, s);
}

template <bool XF32, bool PAIR, bool SEG>
int dispatch_upl(const GemvArgs& a, const GemvPlan& p, cudaStream_t s) {
  switch (p.upl) {
    case 1: return dispatch_sb<1, XF32, PAIR, SEG>(a, p, s);
    case 2: return dispatch_sb<2, XF32, PAIR, SEG>(a, p, s);
    default: return dispatch_sb<4, XF32, PAIR, SEG>(a, p, s);
  }
}

int finish_and_launch(GemvArgs& a, bool xf32, bool pair, bool seg, cudaStream_t stream) {
  int outs[kMaxMats];
  for (int i = 0; i < a.nmat; ++i) outs[i] = a.mat[i].out;
  const GemvPlan p = plan_gemv(a.in, a.nseg, a.total_rows, pair, outs, a.nmat);
  if (p.threads > (p.upl == 1 ? 640 : 384) || p.smem > (size_t)device_info().max_smem_optin) return QG_ENOTSUP;
  a.units = a.nseg * a.in / 32;
  a.rt = p.rt;
  a.nstage = p.nstage;
  a.ngr = p.ngr;
  a.wpg = p.wpg;
  a.q = p.q;
  a.slot_bytes = p.slot_bytes;
  a.sb_bytes = p.sb_bytes;
  if (seg) return dispatch_upl<true, false, true>(a, p, stream);  // segmented mode takes fp32 x
  if (pair) return xf32 ? dispatch_upl<true, true, false>(a, p, stream) : dispatch_upl<false, true, false>(a, p, stream);
  return xf32 ? dispatch_upl<true, false, false>(a, p, stream) : dispatch_upl<false, false, false>(a, p, stream);
}

}  // namespace

int gemv_tune(int upl, int ngr, int rt, int nstage) {
  if (upl != 0 && upl != 1 && upl != 2 && upl != 4) return QG_EINVAL;
  if (ngr < 0 || ngr > 8 || rt < 0 || nstage < 0 || nstage > 8 || nstage == 1) return QG_EINVAL;
  g_tune = Tune{upl, ngr, rt, nstage};
  return QG_OK;
}

int gemv_launch(const GemvMatArg* mats, int n, int pair_swiglu, const void* x, int xt, int in, cudaStream_t stream) {
  if (n < 1 || n > 4 || (pair_swiglu && n != 2)) return QG_EINVAL;
  GemvArgs a{};
  int rows = 0;
  if (pair_swiglu) {
    a.nmat = 1;
    a.mat[0].w[0] = WRef{mats[0].packed, mats[0].scales, mats[0].biases, -1};
    a.mat[0].w[1] = WRef{mats[1].packed, mats[1].scales, mats[1].biases, -1};
    a.mat[0].y = mats[0].y;
    a.mat[0].out = mats[0].out;
    a.mat[0].row0 = 0;
    rows = mats[0].out;
  } else {
    a.nmat = n;
    for (int i = 0; i < n; ++i) {
      a.mat[i].w[0] = WRef{mats[i].packed, mats[i].scales, mats[i].biases, -1};
      a.mat[i].w[1] = a.mat[i].w[0];
      a.mat[i].y = mats[i].y;
      a.mat[i].out = mats[i].out;
      a.mat[i].row0 = rows;
      rows += mats[i].out;
    }
  }
  a.nseg = 1;
  a.x = x;
  a.in = in;
  a.total_rows = rows;
  return finish_and_launch(a, xt == QG_X_F32, pair_swiglu != 0, false, stream);
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
  a.idx = idx;
  a.n_experts = gate->n_mat;
  a.slab_words = (long long)gate->out * (gate->in / 8);
  a.slab_groups = (long long)gate->out * (gate->in / 64);
  a.in = gate->in;
  a.total_rows = k * gate->out;
  return finish_and_launch(a, false, true, false, stream);
}

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
  a.idx = idx;
  a.p = p;
  a.resid = residual;
  a.n_experts = down->n_mat;
  a.slab_words = (long long)down->out * (down->in / 8);
  a.slab_groups = (long long)down->out * (down->in / 64);
  a.in = down->in;
  a.total_rows = down->out;
  return finish_and_launch(a, true, false, true, stream);
}

}  // namespace qg
