// quant.cu -- affine group-64 quantizer (encode) for the Q4_64A / Q2_64A formats ([ds4#844],
// Q4_64A / Q2_64A commit: the codes are computed from the scale and bias after their rounding to
// bf16, the values that are stored):
//   per group of 64 weights: lo = min, hi = max (a zero of either sign taken as +0);
//   scale = (hi - lo) / (2^bits - 1); bias = lo; s = bf16(scale), b = bf16(bias) (nearest, ties to even);
//   q_j = clamp(rint((w_j - b) / s), 0, 2^bits - 1)   (0 when s = 0)
// The codes are decided as binary32 rint of the correctly rounded quotient (w - b) / s, bit for bit,
// without a division per weight.  Per group: y = RN(1/s) (correctly rounded), e0 = 1 - s y (exact
// by FMA), ye = RN(y e0).  Per weight: t = RN(d y + RN(d ye)), two operations.  The unrounded sum
// is within about 2^-45 |t| of d/s, while a quotient of a binary32 d by a bf16 s (8-bit
// significand) is never within 2^-33 |t| of a binary32 rounding midpoint (nor on one), so the
// rounding agrees with RN(d/s); checked exhaustively for every bf16 significand of s and every
// binary32 d in [2^-4, 2^7).
//
// HBM-bound: one pass over the weights (2 or 4 B each) writing bits/8 B per weight plus 4 B per
// group.  A row-major [out][in] matrix is one flat run of out*in/64 groups (group gc at element
// 64 gc, its packed words at gc * 64 bits / 32, its scale and bias at gc), so the kernel streams it
// without row arithmetic: one warp-step is 2 KB of weights, four 16-byte words per lane, loaded one
// step ahead into registers (2 KB in flight per warp while the previous step is encoded).
// Eight lanes share a group.  Per weight: d by one FMA, the quotient by a multiply and a
// saturating FMA (t/K clamped to [0, 1], K = 16 for 4 bits, 4 for 2 bits), one FMA onto 2^23
// (round to nearest even, the code in the low mantissa bits), an integer multiply-add for the
// packing, and an integer min only in steps where some group's top code could exceed 2^bits - 1:
// no branch, no conversion, and most of it on the FMA pipe (the integer pipe is the scarcer one).
// The group's division, reciprocal and bf16 rounding are done once per group by an owner lane and
// shuffled to the other lanes.
#include <algorithm>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

// bf16 bits of a binary32 (finite or infinite), round to nearest, ties to even.
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// RN(a * b + c) clamped to [0, 1] (a NaN result gives +0).
__device__ __forceinline__ float fma_sat(float a, float b, float c) {
  float r;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

constexpr uint32_t kMagic = 0x4B000000u;  // bits of 2^23: 2^23 + c has mantissa c for 0 <= c < 2^23

// Horner packing of N codes given as bits of 2^23 + c_i (low code first): sum_i c_i 2^(BITS i).
// The 2^23 exponent bits accumulate to a constant (mod 2^32) that is subtracted once.  mul is
// 2^BITS, passed at run time so that the multiply-add stays an integer multiply-add (FMA pipe)
// rather than becoming a shift-add on the integer pipe.
template <int BITS, int N>
__device__ __forceinline__ uint32_t pack_codes(const uint32_t* m, uint32_t mul) {
  constexpr uint32_t kBias = [] {
    uint32_t c = 0;
    for (int i = 0; i < N; ++i) c = c * (1u << BITS) + kMagic;
    return c;
  }();
  uint32_t acc = 0;
#pragma unroll
  for (int i = N - 1; i >= 0; --i) acc = acc * mul + m[i];
  return acc - kBias;
}

// One lane's eight weights of a group: bf16 (the eight halves of a) or fp32 (a then c).
template <bool F32>
__device__ __forceinline__ void unpack8(const uint4& a, const uint4& c, float (&v)[8]) {
  if (F32) {
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(c.x); v[5] = __uint_as_float(c.y); v[6] = __uint_as_float(c.z); v[7] = __uint_as_float(c.w);
  } else {
    const uint32_t q[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(q[i] << 16);
      v[2 * i + 1] = __uint_as_float(q[i] & 0xFFFF0000u);
    }
  }
}

// The packed codes of the eight weights: bf16, one word of 8 codes (low code first); fp32, the
// codes of a's four weights in the low 16 bits and of c's four in the high 16 (4 bits), or in the
// low and high bytes of the low half (2 bits).
template <int BITS, bool F32>
__device__ __forceinline__ uint32_t pack8(const uint32_t (&m)[8], uint32_t mul) {
  if (F32) {
    return pack_codes<BITS, 4>(m, mul) | (pack_codes<BITS, 4>(m + 4, mul) << (4 * BITS));
  } else {
    return pack_codes<BITS, 8>(m, mul);
  }
}

// What every lane of a group needs: d = FMA(v, ps, nb) = RN(v - b) ps, and yk = y/K, yek = ye/K
// for the quotient (y = RN(1/(s ps)), ye = RN(y (1 - s ps y))).  ps = 1 unless s lies outside
// [2^-100, 2^100], where it is 2^64 or 2^-64 so that s ps, y and ye stay clear of overflow and of
// the subnormal range (scaling by a power of two commutes with the rounding; the weights of such a
// group lie within 2^24 (hi - lo) of b, so nothing overflows).  s = 0: yk = yek = 0, every code 0.
struct GroupK {
  float ps, nb, yk, yek;
};

// The owner lane's work for one group: bf16 scale and bias bits, the constants above, and whether
// every code of the group is at most 2^bits - 1 before the clamp (the largest d, at w = hi, gives
// a quotient of at most 2^bits - 3/4, so no code rounds above the top).
template <int BITS>
__device__ __forceinline__ GroupK group_constants(float l, float h, uint32_t& sb, uint32_t& bb, bool& safe) {
  constexpr uint32_t kQmax = (1u << BITS) - 1u;
  constexpr float kInvK = BITS == 4 ? 0.0625f : 0.25f;
  l = __fadd_rn(l, 0.f);  // a zero of either sign -> +0
  h = __fadd_rn(h, 0.f);
  const float scale = __fdiv_rn(__fsub_rn(h, l), (float)kQmax);
  sb = f32_to_bf16_rne(scale);
  bb = f32_to_bf16_rne(l);
  const float s = __uint_as_float(sb << 16), b = __uint_as_float(bb << 16);
  GroupK g;
  if (s == 0.f) {
    g.ps = 1.f;
    g.nb = -b;
    g.yk = 0.f;
    g.yek = 0.f;
    safe = true;
  } else {
    g.ps = s < 0x1p-100f ? 0x1p64f : (s > 0x1p100f ? 0x1p-64f : 1.f);
    g.nb = -__fmul_rn(b, g.ps);
    const float sp = __fmul_rn(s, g.ps);
    const float y = __frcp_rn(sp);
    const float e0 = __fmaf_rn(-sp, y, 1.f);
    g.yk = __fmul_rn(y, kInvK);
    g.yek = __fmul_rn(__fmul_rn(y, e0), kInvK);
    safe = g.ps == 1.f && __fmul_rn(__fsub_rn(h, b), y) <= (float)kQmax + 0.25f;
  }
  return g;
}

// The packed codes of one lane's eight weights of a group: d = RN(v - b) ps, u = RN(d yk +
// RN(d yek)) = RN(d / (s ps))/K clamped to [0, 1], FMA(u, K, 2^23) rounds K u to the nearest
// integer, ties to even; CLAMP takes the integer min with 2^bits - 1.
template <int BITS, bool F32, bool CLAMP>
__device__ __forceinline__ uint32_t encode8(const uint4& a, const uint4& c, const GroupK& g, uint32_t mul) {
  constexpr float kK = BITS == 4 ? 16.f : 4.f;
  constexpr uint32_t kQmax = (1u << BITS) - 1u;
  float v[8];
  unpack8<F32>(a, c, v);
  uint32_t m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float d = __fmaf_rn(v[i], g.ps, g.nb);
    const float u = fma_sat(d, g.yk, __fmul_rn(d, g.yek));
    const uint32_t mi = __float_as_uint(__fmaf_rn(u, kK, 0x1p23f));
    m[i] = CLAMP ? min(mi, kMagic + kQmax) : mi;
  }
  return pack8<BITS, F32>(m, mul);
}

// One warp-step: kGroups = 16 (bf16) or 8 (fp32) consecutive groups, 2 KB.  Lane L (oct = L / 8,
// sub = L % 8) holds, for each of its kSlots groups 4 k + oct:
//   bf16: word k = weights 8 sub .. 8 sub + 7;
//   fp32: words 2k, 2k + 1 = weights 4 sub .. 4 sub + 3 and 32 + 4 sub .. 32 + 4 sub + 3,
// so every load instruction of the warp reads whole 128-byte lines.
template <bool F32>
struct QStep {
  static constexpr int kSlots = F32 ? 2 : 4;
  static constexpr int kGroups = 4 * kSlots;
};

template <bool F32>
__device__ __forceinline__ void load_step(const void* __restrict__ w, int step, int ngroups, int lane,
                                          uint4 (&r)[4]) {
  const int oct = lane >> 3, sub = lane & 7;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int k = F32 ? j >> 1 : j;
    const int gi = min(step * QStep<F32>::kGroups + 4 * k + oct, ngroups - 1);
    if (F32) {
      const float* p = static_cast<const float*>(w) + (size_t)gi * 64 + 32 * (j & 1) + 4 * sub;
      r[j] = __ldcs(reinterpret_cast<const uint4*>(p));
    } else {
      const uint16_t* p = static_cast<const uint16_t*>(w) + (size_t)gi * 64 + 8 * sub;
      r[j] = __ldcs(reinterpret_cast<const uint4*>(p));
    }
  }
}

// Stores one slot's packed codes: bf16, each lane holds its word (4 bits) or half-word (2 bits);
// fp32, each lane holds the codes of two quarter-groups (see pack8), combined across 2 or 4 lanes.
template <int BITS, bool F32>
__device__ __forceinline__ void store_codes(uint32_t* __restrict__ pw, bool gv, int sub, uint32_t word) {
  if (!F32) {  // word: weights 8 sub .. 8 sub + 7
    if (BITS == 4) {
      if (gv) pw[sub] = word;
    } else {
      const uint32_t other = __shfl_xor_sync(0xffffffffu, word, 1);
      if (gv && (sub & 1) == 0) pw[sub >> 1] = word | (other << 16);
    }
  } else if (BITS == 4) {  // 16 bits per quarter-group: words sub/2 and 4 + sub/2 from a lane pair
    const uint32_t other = __shfl_xor_sync(0xffffffffu, word, 1);
    if (gv) {
      if ((sub & 1) == 0)
        pw[sub >> 1] = (word & 0xFFFFu) | (other << 16);
      else
        pw[4 + (sub >> 1)] = (other >> 16) | (word & 0xFFFF0000u);
    }
  } else {  // 8 bits per quarter-group: words sub/4 and 2 + sub/4 from a lane quad
    uint32_t a = (word & 0xFFu) << (8 * (sub & 3)), c = (word >> 8) << (8 * (sub & 3));
    a |= __shfl_xor_sync(0xffffffffu, a, 1);
    c |= __shfl_xor_sync(0xffffffffu, c, 1);
    a |= __shfl_xor_sync(0xffffffffu, a, 2);
    c |= __shfl_xor_sync(0xffffffffu, c, 2);
    if (gv && (sub & 3) == 0) pw[sub >> 2] = a;
    if (gv && (sub & 3) == 1) pw[2 + (sub >> 2)] = c;
  }
}

template <int BITS, bool F32, bool CLAMP>
__device__ __forceinline__ void codes_step(const uint4 (&cur)[4], const GroupK& go, int g0, int ngroups, int lane,
                                           uint32_t mul, uint32_t* __restrict__ packed) {
  constexpr int kSlots = QStep<F32>::kSlots;
  constexpr int kWords = 64 * BITS / 32;  // packed words per group
  const int sub = lane & 7;
#pragma unroll
  for (int k = 0; k < kSlots; ++k) {
    const int src = (lane & 24) + k;
    GroupK g;
    g.ps = CLAMP ? __shfl_sync(0xffffffffu, go.ps, src) : 1.f;  // steps without the clamp have ps = 1
    g.nb = __shfl_sync(0xffffffffu, go.nb, src);
    g.yk = __shfl_sync(0xffffffffu, go.yk, src);
    g.yek = __shfl_sync(0xffffffffu, go.yek, src);
    const uint32_t word = F32 ? encode8<BITS, F32, CLAMP>(cur[2 * k], cur[2 * k + 1], g, mul)
                              : encode8<BITS, F32, CLAMP>(cur[k], cur[k], g, mul);
    const int gi = g0 + 4 * k;
    store_codes<BITS, F32>(packed + (size_t)gi * kWords, gi < ngroups, sub, word);
  }
}

// One warp-step over the words in cur (uniform per warp: shuffles and votes inside).
template <int BITS, bool F32>
__device__ __forceinline__ void quant_step(const uint4 (&cur)[4], int step, int ngroups, int lane, uint32_t mul,
                                           uint32_t* __restrict__ packed, uint16_t* __restrict__ scales,
                                           uint16_t* __restrict__ biases) {
  constexpr int kSlots = QStep<F32>::kSlots, kGroups = QStep<F32>::kGroups;
  const int oct = lane >> 3, sub = lane & 7;
  const int g0 = step * kGroups + oct;  // slot k's group: g0 + 4 k
  // 1. min and max of each slot's group over its eight lanes
  float lo[kSlots], hi[kSlots];
#pragma unroll
  for (int k = 0; k < kSlots; ++k) {
    if (F32) {
      float x[8];
      unpack8<true>(cur[2 * k], cur[2 * k + 1], x);
      float l = x[0], h = x[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) {
        l = fminf(l, x[i]);
        h = fmaxf(h, x[i]);
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        l = fminf(l, __shfl_xor_sync(0xffffffffu, l, o));
        h = fmaxf(h, __shfl_xor_sync(0xffffffffu, h, o));
      }
      lo[k] = l;
      hi[k] = h;
    } else {
      // bf16 pairs: (min, -max) in one bf16x2, so one min per step reduces both
      const uint4 q = cur[k];
      const uint32_t mn = bf16x2_min(bf16x2_min(q.x, q.y), bf16x2_min(q.z, q.w));
      const uint32_t nx = bf16x2_max(bf16x2_max(q.x, q.y), bf16x2_max(q.z, q.w)) ^ 0x80008000u;
      uint32_t p = bf16x2_min(__byte_perm(mn, nx, 0x5410), __byte_perm(mn, nx, 0x7632));
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) p = bf16x2_min(p, __shfl_xor_sync(0xffffffffu, p, o));
      lo[k] = __uint_as_float(p << 16);
      hi[k] = -__uint_as_float(p & 0xFFFF0000u);
    }
  }
  // 2. the owner lane of each group (sub = k; lanes sub >= kSlots repeat it)
  const int ko = sub & (kSlots - 1);
  float l = lo[0], h = hi[0];
#pragma unroll
  for (int k = 1; k < kSlots; ++k) {
    if (ko == k) {
      l = lo[k];
      h = hi[k];
    }
  }
  uint32_t sb, bb;
  bool safe;
  const GroupK go = group_constants<BITS>(l, h, sb, bb, safe);
  {
    const int gown = g0 + 4 * ko;
    if (sub < kSlots && gown < ngroups) {
      scales[gown] = (uint16_t)sb;
      biases[gown] = (uint16_t)bb;
    }
  }
  // 3. codes; the integer clamp only where some group of the step needs it
  if (__all_sync(0xffffffffu, safe))
    codes_step<BITS, F32, false>(cur, go, g0, ngroups, lane, mul, packed);
  else
    codes_step<BITS, F32, true>(cur, go, g0, ngroups, lane, mul, packed);
}

template <int BITS, bool F32>
__global__ void __launch_bounds__(256, 4) quant_kernel(const void* __restrict__ w, int ngroups, uint32_t mul,
                                                       uint32_t* __restrict__ packed,
                                                       uint16_t* __restrict__ scales,
                                                       uint16_t* __restrict__ biases) {
  constexpr int kGroups = QStep<F32>::kGroups;
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int nsteps = (ngroups + kGroups - 1) / kGroups;
  const int nwarps = gridDim.x * (blockDim.x / 32);
  int step = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  // two register buffers in turn: the next step's words are in flight while this step is encoded
  uint4 ba[4], bb[4];
  if (step < nsteps) load_step<F32>(w, step, ngroups, lane, ba);
  while (step < nsteps) {
    if (step + nwarps < nsteps) load_step<F32>(w, step + nwarps, ngroups, lane, bb);
    quant_step<BITS, F32>(ba, step, ngroups, lane, mul, packed, scales, biases);
    step += nwarps;
    if (step >= nsteps) break;
    if (step + nwarps < nsteps) load_step<F32>(w, step + nwarps, ngroups, lane, ba);
    quant_step<BITS, F32>(bb, step, ngroups, lane, mul, packed, scales, biases);
    step += nwarps;
  }
}

}  // namespace

int quant_launch(const void* w, int wt, int out, int in, int bits, uint32_t* packed, uint16_t* scales,
                 uint16_t* biases, cudaStream_t stream) {
  const long long ngl = (long long)out * (in / 64);
  if (ngl >= (1LL << 31) - 64) return QG_ENOTSUP;
  const int ngroups = (int)ngl;
  const bool f32 = wt == QG_X_F32;
  const int per_step = f32 ? QStep<true>::kGroups : QStep<false>::kGroups;
  const long long steps = (ngl + per_step - 1) / per_step;
  const int threads = 256;  // eight warps; four CTAs per SM (at most 64 registers a thread)
  const int blocks = (int)std::max<long long>(1, std::min<long long>((steps + 7) / 8, 4LL * device_info().num_sms));
  const uint32_t mul = 1u << bits;
  if (bits == 4)
    return f32 ? launch(quant_kernel<4, true>, dim3(blocks), dim3(threads), 0, stream, w, ngroups, mul, packed, scales,
                        biases)
               : launch(quant_kernel<4, false>, dim3(blocks), dim3(threads), 0, stream, w, ngroups, mul, packed, scales,
                        biases);
  return f32 ? launch(quant_kernel<2, true>, dim3(blocks), dim3(threads), 0, stream, w, ngroups, mul, packed, scales,
                      biases)
             : launch(quant_kernel<2, false>, dim3(blocks), dim3(threads), 0, stream, w, ngroups, mul, packed, scales,
                      biases);
}

}  // namespace qg
