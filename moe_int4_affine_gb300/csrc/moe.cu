// moe.cu -- MoE decode pieces besides the expert GEMVs: the device router (top-K + softmax) and
// the standalone scalar-weighted chain with residual.  The expert gather itself runs on the
// streaming GEMV kernel (qgemv.cu) in its MoE gate/up and MoE down modes.
#include <algorithm>
#include <utility>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int kRouterMaxPerLane = 32;  // 32 lanes x 32 = 1024 experts

// Router top-K ([FFAI#14] commit "moeRouterTopK"; order (value desc, index asc) as in [FFAI#9]'s
// partial-sort commit).  One warp.  Each of k rounds takes, across the warp, the not-yet-taken
// expert with the largest logit, the lower index on equal logits.  Then the weights: softmax of
// the selected logits (renorm) or of all logits read at the selected ones.
__global__ void __launch_bounds__(32) router_kernel(const float* __restrict__ logits, int n, int k, int renorm,
                                                    uint32_t* __restrict__ idx_out, float* __restrict__ p_out) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x;
  float v[kRouterMaxPerLane];
  uint32_t taken = 0;  // bit j: expert lane + 32 j is selected or does not exist
  const int per = (n + 31) / 32;
#pragma unroll
  for (int j = 0; j < kRouterMaxPerLane; ++j) {
    const int e = lane + 32 * j;
    const bool live = j < per && e < n;
    v[j] = live ? logits[e] : 0.f;
    if (!live) taken |= 1u << j;
  }
  float sel_v[32];
  uint32_t sel_i[32];
  for (int s = 0; s < k; ++s) {
    // lane-local best: largest value, then the smallest index (= smallest j for a fixed lane)
    float bv = 0.f;
    int bj = -1;
#pragma unroll
    for (int j = 0; j < kRouterMaxPerLane; ++j) {
      if (taken & (1u << j)) continue;
      if (bj < 0 || v[j] > bv) {
        bv = v[j];
        bj = j;
      }
    }
    int bi = bj < 0 ? 0x7fffffff : lane + 32 * bj;
    bool has = bj >= 0;
    // warp arg-best over (has, value desc, index asc): a strict total order, so every lane ends
    // with the same winner
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      const bool oh = __shfl_xor_sync(0xffffffffu, has, off);
      const bool better = oh && (!has || ov > bv || (ov == bv && oi < bi));
      if (better) {
        bv = ov;
        bi = oi;
        has = oh;
      }
    }
    sel_v[s] = bv;
    sel_i[s] = (uint32_t)bi;
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
  }
  const float m = sel_v[0];
  float z = 0.f;
  if (renorm) {
    for (int s = 0; s < k; ++s) z += expf(sel_v[s] - m);
  } else {
    float zl = 0.f;
#pragma unroll
    for (int j = 0; j < kRouterMaxPerLane; ++j) {
      const int e = lane + 32 * j;
      if (j < per && e < n) zl += expf(v[j] - m);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zl += __shfl_xor_sync(0xffffffffu, zl, off);
    z = zl;
  }
  for (int s = lane; s < k; s += 32) {
    idx_out[s] = sel_i[s];
    p_out[s] = expf(sel_v[s] - m) / z;
  }
}

int router_launch(const float* logits, int n_experts, int k, int renorm, uint32_t* idx, float* p,
                  cudaStream_t stream) {
  return launch(router_kernel, dim3(1), dim3(32), 0, stream, logits, n_experts, k, renorm, idx, p);
}

// out[i] = residual[i] + sum_{k<8} p[k] * v[k][i], accumulated in slot order ([FFAI#14] scalar-FMA
// commit, "scalarFMAChain8").  Each thread handles 4 consecutive elements.
__global__ void __launch_bounds__(256) chain8_kernel(const float* __restrict__ p, const float* __restrict__ v,
                                                     const uint16_t* __restrict__ resid, float* __restrict__ out,
                                                     int n) {
  pdl_trigger();
  pdl_wait();
  float pk[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) pk[k] = __ldg(p + k);
  const int nthreads = gridDim.x * blockDim.x;
  const bool vec = (n & 3) == 0;
  for (int i4 = blockIdx.x * blockDim.x + threadIdx.x; i4 * 4 < n; i4 += nthreads) {
    const int i = i4 * 4;
    if (vec) {
      const uint2 rb = __ldg(reinterpret_cast<const uint2*>(resid + i));
      float4 acc = make_float4(bf16_bits_to_f32(rb.x & 0xFFFFu), bf16_bits_to_f32(rb.x >> 16),
                               bf16_bits_to_f32(rb.y & 0xFFFFu), bf16_bits_to_f32(rb.y >> 16));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(v + (size_t)k * n + i));
        acc.x = fmaf(pk[k], t.x, acc.x);
        acc.y = fmaf(pk[k], t.y, acc.y);
        acc.z = fmaf(pk[k], t.z, acc.z);
        acc.w = fmaf(pk[k], t.w, acc.w);
      }
      *reinterpret_cast<float4*>(out + i) = acc;
    } else {
      for (int ii = i; ii < min(i + 4, n); ++ii) {
        float acc = bf16_bits_to_f32(resid[ii]);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc = fmaf(pk[k], v[(size_t)k * n + ii], acc);
        out[ii] = acc;
      }
    }
  }
}

int chain8_launch(const float* p, const float* v, const uint16_t* residual, float* out, int n, cudaStream_t stream) {
  const int threads = 256;
  const int quads = (n + 3) / 4;
  int blocks = (quads + threads - 1) / threads;
  blocks = std::max(1, std::min(blocks, 4 * device_info().num_sms));
  return launch(chain8_kernel, dim3(blocks), dim3(threads), 0, stream, p, v, residual, out, n);
}

}  // namespace qg
