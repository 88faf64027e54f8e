// moe.cu -- MoE decode pieces besides the expert GEMVs: the device router (top-K + softmax) and
// the standalone scalar-weighted chain with residual.  The expert gather itself runs on the
// streaming GEMV kernel (gemv_kernel.cuh) in its MoE gate/up and MoE down modes.
#include <algorithm>
#include <utility>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int kRouterMaxPerLane = 32;  // 32 lanes x 32 = 1024 experts

// Order-preserving key of a finite float: larger floats give larger unsigned keys; -0 and +0 get
// the same key (they compare equal, so the index decides between them).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Router top-K ([FFAI#14] commit "moeRouterTopK"; order (value desc, index asc) as in [FFAI#9]'s
// partial-sort commit).  One warp; lane l holds experts l, l + 32, ... (PER of them).  A candidate is
// the 64-bit key (float_key(logit) << 32) | ~index, so the largest key is the largest logit with
// the lowest index on ties, and every lane agrees on it.  Round s takes the warp's largest key not
// yet taken; lane s keeps round s's selection.  Then the weights: softmax of the selected logits
// (renorm) or of all logits read at the selected ones.  Block b routes token b (logits row b,
// outputs row b of [T][k]).
template <int PER>
__global__ void __launch_bounds__(32) router_kernel(const float* __restrict__ logits, int n, int k, int renorm,
                                                    uint32_t* __restrict__ idx_out, float* __restrict__ p_out) {
  pdl_trigger();
  pdl_wait();
  logits += (size_t)blockIdx.x * n;
  idx_out += (size_t)blockIdx.x * k;
  p_out += (size_t)blockIdx.x * k;
  const int lane = threadIdx.x;
  float v[PER];
  unsigned long long key[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < n ? __ldg(logits + e) : 0.f;
    key[j] = e < n ? ((unsigned long long)float_key(v[j]) << 32) | (uint32_t)~(uint32_t)e : 0ull;
  }
  unsigned long long mine = 0;  // this lane's round's selection (lane s keeps round s)
  for (int s = 0; s < k; ++s) {
    unsigned long long best = key[0];
#pragma unroll
    for (int j = 1; j < PER; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
      best = o > best ? o : best;
    }
    if (lane == s) mine = best;
#pragma unroll
    for (int j = 0; j < PER; ++j) key[j] = key[j] == best ? 0ull : key[j];  // (keys are unique)
  }
  const uint32_t my_idx = ~(uint32_t)mine;
  const uint32_t kv = (uint32_t)(mine >> 32);
  const float my_v = __uint_as_float((kv & 0x80000000u) ? (kv & 0x7FFFFFFFu) : ~kv);
  const float m = __shfl_sync(0xffffffffu, my_v, 0);  // round 0 took the largest logit
  float z;
  if (renorm) {
    z = lane < k ? expf(my_v - m) : 0.f;
  } else {
    z = 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (lane + 32 * j < n) z += expf(v[j] - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  if (lane < k) {
    idx_out[lane] = my_idx;
    p_out[lane] = expf(my_v - m) / z;
  }
}

int router_batch_launch(const float* logits, int T, int n_experts, int k, int renorm, uint32_t* idx, float* p,
                        cudaStream_t stream) {
  const int per = (n_experts + 31) / 32;
  const dim3 grid((unsigned)T);
  if (per <= 1) return launch(router_kernel<1>, grid, dim3(32), 0, stream, logits, n_experts, k, renorm, idx, p);
  if (per <= 2) return launch(router_kernel<2>, grid, dim3(32), 0, stream, logits, n_experts, k, renorm, idx, p);
  if (per <= 4) return launch(router_kernel<4>, grid, dim3(32), 0, stream, logits, n_experts, k, renorm, idx, p);
  if (per <= 8) return launch(router_kernel<8>, grid, dim3(32), 0, stream, logits, n_experts, k, renorm, idx, p);
  if (per <= 16) return launch(router_kernel<16>, grid, dim3(32), 0, stream, logits, n_experts, k, renorm, idx, p);
  return launch(router_kernel<kRouterMaxPerLane>, grid, dim3(32), 0, stream, logits, n_experts, k, renorm, idx, p);
}

int router_launch(const float* logits, int n_experts, int k, int renorm, uint32_t* idx, float* p,
                  cudaStream_t stream) {
  return router_batch_launch(logits, 1, n_experts, k, renorm, idx, p, stream);
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

// The shared-expert step ([FFAI#14], scalar-FMA commit, sigmoidScalarFMAResidual):
//   out[i] = base[i] + sigmoid(gate) * value[i] (+ resid[i])
// gate read once per thread from device memory; 16-byte vectors when n % 4 == 0.
__global__ void __launch_bounds__(256) sigmoid_fma_kernel(const float* __restrict__ gate, const float* __restrict__ value,
                                                          const float* __restrict__ base,
                                                          const uint16_t* __restrict__ resid, float* __restrict__ out,
                                                          int n) {
  pdl_trigger();
  pdl_wait();
  const float s = 1.f / (1.f + expf(-__ldg(gate)));
  const int nthreads = gridDim.x * blockDim.x;
  const bool vec = (n & 3) == 0;
  for (int i4 = blockIdx.x * blockDim.x + threadIdx.x; i4 * 4 < n; i4 += nthreads) {
    const int i = i4 * 4;
    if (vec) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(value + i));
      const float4 b = __ldg(reinterpret_cast<const float4*>(base + i));
      float4 o = make_float4(fmaf(s, v.x, b.x), fmaf(s, v.y, b.y), fmaf(s, v.z, b.z), fmaf(s, v.w, b.w));
      if (resid) {
        const uint2 rb = __ldg(reinterpret_cast<const uint2*>(resid + i));
        o.x += bf16_bits_to_f32(rb.x & 0xFFFFu);
        o.y += bf16_bits_to_f32(rb.x >> 16);
        o.z += bf16_bits_to_f32(rb.y & 0xFFFFu);
        o.w += bf16_bits_to_f32(rb.y >> 16);
      }
      *reinterpret_cast<float4*>(out + i) = o;
    } else {
      for (int ii = i; ii < min(i + 4, n); ++ii) {
        float o = fmaf(s, value[ii], base[ii]);
        if (resid) o += bf16_bits_to_f32(resid[ii]);
        out[ii] = o;
      }
    }
  }
}

int sigmoid_fma_launch(const float* gate, const float* value, const float* base, const uint16_t* resid, float* out,
                       int n, cudaStream_t stream) {
  const int threads = 256;
  const int quads = (n + 3) / 4;
  int blocks = (quads + threads - 1) / threads;
  blocks = std::max(1, std::min(blocks, 4 * device_info().num_sms));
  return launch(sigmoid_fma_kernel, dim3(blocks), dim3(threads), 0, stream, gate, value, base, resid, out, n);
}

}  // namespace qg
