// quant.cu -- affine group-64 quantizer (encode) for the Q4_64A / Q2_64A formats ([ds4#844]:
// "Q4_64A and Q2_64A codes are derived from the serialized BF16 scale/bias"):
//   per group of 64 weights: lo = min, hi = max; scale = (hi - lo) / (2^bits - 1); bias = lo;
//   s = bf16(scale), b = bf16(bias) (nearest, ties to even);
//   q_j = clamp(rint((w_j - b) / s), 0, 2^bits - 1)   (0 when s = 0)
// The codes are decided as binary32 rint of the correctly rounded quotient (w - b) / s, bit for bit
// (a reciprocal multiply where no half-integer is near, the IEEE division where one is).
//
// HBM-bound: one pass over the weights (2 or 4 B each) writing bits/8 B per weight plus 4 B per
// group.  Eight lanes per group, each with one 16-byte word of bf16 (or two of fp32): coalesced
// 128-byte (256-byte) loads per group, min / max by three shuffles, each lane packs its eight
// codes (4 bits: one u32; 2 bits: half a u32, paired with the neighbouring lane).
#include <algorithm>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

// bf16 bits of a finite binary32, round to nearest, ties to even.
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

template <int BITS, bool F32>
__global__ void __launch_bounds__(256) quant_kernel(const void* __restrict__ w, int in, int ngroups,
                                                    uint32_t* __restrict__ packed, uint16_t* __restrict__ scales,
                                                    uint16_t* __restrict__ biases) {
  constexpr unsigned kQmax = (1u << BITS) - 1u;
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31, sub = lane & 7;
  const unsigned ngs = (unsigned)in / 64u;
  const int nwarps = gridDim.x * (blockDim.x / 32);
  const int warp0 = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  // four groups per warp and step; the loop is uniform per warp (shuffles below).  The next step's
  // words are requested before the current step is encoded (one step of loads in flight).
  const int stride = nwarps * 4;
  auto locate = [&](int base, unsigned& gc, unsigned& row, unsigned& g) {
    const int gi = base + (lane >> 3);
    gc = (unsigned)(gi < ngroups ? gi : ngroups - 1);
    row = gc / ngs;
    g = gc - row * ngs;
  };
  auto load = [&](int base, uint4 (&r)[2]) {
    unsigned gc, row, g;
    locate(base, gc, row, g);
    const size_t e0 = (size_t)row * in + (size_t)g * 64 + (size_t)sub * 8;  // this lane's 8 weights
    if (F32) {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(w) + e0);
      r[0] = __ldg(p);
      r[1] = __ldg(p + 1);
    } else {
      r[0] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(w) + e0));
    }
  };
  uint4 cur[2] = {}, nxt[2] = {};
  if (warp0 * 4 < ngroups) load(warp0 * 4, cur);
  for (int base = warp0 * 4; base < ngroups; base += stride) {
    if (base + stride < ngroups) load(base + stride, nxt);
    unsigned gc, row, g;
    locate(base, gc, row, g);
    const bool gv = base + (lane >> 3) < ngroups;
    float v[8];
    if (F32) {
      const uint32_t q[8] = {cur[0].x, cur[0].y, cur[0].z, cur[0].w, cur[1].x, cur[1].y, cur[1].z, cur[1].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(q[j]);
    } else {
      const uint32_t q[4] = {cur[0].x, cur[0].y, cur[0].z, cur[0].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(q[j] << 16);
        v[2 * j + 1] = __uint_as_float(q[j] & 0xFFFF0000u);
      }
    }
    cur[0] = nxt[0];
    cur[1] = nxt[1];
    float lo = v[0], hi = v[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) {
      lo = fminf(lo, v[j]);
      hi = fmaxf(hi, v[j]);
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    lo = __fadd_rn(lo, 0.f);  // -0 -> +0 (a min of -0 and +0 could be either)
    const float scale = __fdiv_rn(__fsub_rn(hi, lo), (float)kQmax);
    const uint32_t sb = f32_to_bf16_rne(scale), bb = f32_to_bf16_rne(lo);
    const float s = __uint_as_float(sb << 16), b = __uint_as_float(bb << 16);
    // t = (w - b) / s correctly rounded, then rint.  Fast path: t' = (w - b) * (1/s) differs from
    // the rounded quotient by at most 1.5 2^-23 |t| (< 3e-6 for |t| <= 16, the only range where the
    // rounding matters: outside it the clamp decides), so rint(t') = rint(t) unless t' lies within
    // 2^-16 of a half-integer; if any of the lane's eight does, the lane takes the exact quotients.
    uint32_t word = 0;
    if (s != 0.f) {
      const float rs = __frcp_rn(s);
      float t[8];
      bool near = false;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        t[j] = __fmul_rn(__fsub_rn(v[j], b), rs);
        near |= fabsf(__fsub_rn(t[j], rintf(t[j]))) > 0.4999847412109375f;  // 0.5 - 2^-16
      }
      if (near) {
#pragma unroll
        for (int j = 0; j < 8; ++j) t[j] = __fdiv_rn(__fsub_rn(v[j], b), s);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) word |= (uint32_t)fminf(fmaxf(rintf(t[j]), 0.f), (float)kQmax) << (BITS * j);
    }
    if (BITS == 4) {
      if (gv) packed[(size_t)row * (in / 8) + (size_t)g * 8 + sub] = word;
    } else {
      const uint32_t other = __shfl_xor_sync(0xffffffffu, word, 1);  // the next eight codes
      if (gv && (sub & 1) == 0) packed[(size_t)row * (in / 16) + (size_t)g * 4 + sub / 2] = word | (other << 16);
    }
    if (gv && sub == 0) {
      scales[gc] = (uint16_t)sb;
      biases[gc] = (uint16_t)bb;
    }
  }
}

}  // namespace

int quant_launch(const void* w, int wt, int out, int in, int bits, uint32_t* packed, uint16_t* scales,
                 uint16_t* biases, cudaStream_t stream) {
  const long long ngl = (long long)out * (in / 64);
  if (ngl >= (1LL << 31)) return QG_ENOTSUP;
  const int ngroups = (int)ngl;
  const int threads = 256;
  const long long want = (ngl + 31) / 32;  // four groups per warp, eight warps per block
  const int blocks = (int)std::max<long long>(1, std::min<long long>(want, 8LL * device_info().num_sms));
  const bool f32 = wt == QG_X_F32;
  if (bits == 4)
    return f32 ? launch(quant_kernel<4, true>, dim3(blocks), dim3(threads), 0, stream, w, in, ngroups, packed, scales, biases)
               : launch(quant_kernel<4, false>, dim3(blocks), dim3(threads), 0, stream, w, in, ngroups, packed, scales, biases);
  return f32 ? launch(quant_kernel<2, true>, dim3(blocks), dim3(threads), 0, stream, w, in, ngroups, packed, scales, biases)
             : launch(quant_kernel<2, false>, dim3(blocks), dim3(threads), 0, stream, w, in, ngroups, packed, scales, biases);
}

}  // namespace qg
