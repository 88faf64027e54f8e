// gemv_dense.cu -- dense dequant-GEMV launches: one matrix, or n in {2,3,4} matrices sharing x
// ([FFAI#14] "dequant_gemv_int4_*", "dequantGemvInt4Two/Three/Four", "ffai_batched_4_qgemv_fast").
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <set>
#include <tuple>

#include "gemv_kernel.cuh"

namespace qg {

GemvTune g_gemv_tune = {0, 0};

int gemv_tune(int ctas_per_sm) {
  if (ctas_per_sm < 0 || ctas_per_sm > 4) return QG_EINVAL;
  g_gemv_tune.ctas_per_sm = ctas_per_sm;
  return QG_OK;
}

int gemv_tune_split(int kcl) {
  if (kcl < 0 || kcl > 4) return QG_EINVAL;
  g_gemv_tune.kcl = kcl;
  return QG_OK;
}

int gemv_max_clusters(int dev, int C) {
  static std::atomic<int> cache[kGemvDevs][5];  // value + 1 once known
  if (C < 2 || C > 4 || dev < 0 || dev >= kGemvDevs) return 0;
  const int known = cache[dev][C].load(std::memory_order_relaxed);
  if (known) return known - 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(C * 16));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;  // (one CTA per SM whatever its shared memory: the registers decide)
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)C;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemv_kernel<kDense, 4, false, false, 4>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache[dev][C].store(n + 1, std::memory_order_relaxed);
  return n;
}

// QG_DEBUG_PLAN=1 in the environment (read once): each distinct GEMV shape's plan on stderr, once.
void gemv_debug_plan(int mode, const GemvArgs& a, int grid, size_t smem) {
  static const bool on = [] {
    const char* e = std::getenv("QG_DEBUG_PLAN");
    return e && e[0] && e[0] != '0';
  }();
  if (!on) return;
  static std::mutex mu;
  static std::set<std::tuple<int, int, int, int, int, int, int>> seen;
  std::lock_guard<std::mutex> lock(mu);
  if (!seen.insert({mode, a.total_rows, a.groups, a.nmat, a.nseg, a.xf32, a.bits}).second) return;
  std::fprintf(stderr,
               "qg plan: gemv mode %d rows %d groups %d (mats %d, segments %d, %s x, %d-bit): grid %d, K split %d "
               "(slice %d groups), rows per CTA %d, shared memory %zu B, x %s\n",
               mode, a.total_rows, a.groups, a.nmat, a.nseg, a.xf32 ? "fp32" : "bf16", a.bits, grid, a.kcl,
               a.slice_groups, a.rows_per_cta, smem, a.stage ? "staged by one bulk copy" : "loaded by the threads");
}

int gemv_dense_launch(const GemvMatArg* mats, int n, const void* x, int xt, int in, cudaStream_t stream,
                      const GemvExtras& ex) {
  if (n < 1 || n > 4) return QG_EINVAL;
  GemvArgs a = dense_args(mats, n, x, xt, in);
  apply_extras(a, ex);
  return plan_and_launch<kDense>(a, stream);
}

// Host-resident input in the launch chain: one CTA copies n16 16-byte words from page-locked host
// memory (read over the CPU-GPU link through its device mapping) into device memory.  It lets the
// next launch start at once (programmatic dependent launch) and waits for the previous one first:
// that one, or one before it, may still read dst.
__global__ void __launch_bounds__(256) ingest_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int n16) {
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
}

int ingest_launch(const void* src_dev_mapped, void* dst, size_t bytes, cudaStream_t stream) {
  if (bytes % 16 != 0 || bytes / 16 > (size_t)INT32_MAX) return QG_EINVAL;
  return launch(ingest_kernel, dim3(1), dim3(256), 0, stream, static_cast<const uint4*>(src_dev_mapped),
                static_cast<uint4*>(dst), (int)(bytes / 16));
}

// Gated RMSNorm, one head per block ([FFAI#14] gatedRmsNormQgemvInt4Fast: a Mamba2-style gated
// norm, silu(z) * w * rmsnorm(y), ahead of the GDN mixer's out-projection), written as fp32 into
// the workspace for the GEMV that follows:
//   x[j] = silu(z[j]) * gamma[j] * (y[j] / sqrt(mean over the head of y^2 + eps))
template <bool F32>
__global__ void __launch_bounds__(256) gated_norm_kernel(const void* __restrict__ y, const void* __restrict__ z,
                                                         const uint16_t* __restrict__ gamma, int head_dim,
                                                         float eps, float* __restrict__ x) {
  __shared__ float red[8];
  pdl_trigger();
  pdl_wait();
  const size_t h0 = (size_t)blockIdx.x * head_dim;
  auto ld = [](const void* p, size_t i) {
    return F32 ? __ldg(static_cast<const float*>(p) + i)
               : __uint_as_float((uint32_t)__ldg(static_cast<const uint16_t*>(p) + i) << 16);
  };
  float ss = 0.f;
  for (int i = threadIdx.x; i < head_dim; i += 256) {
    const float v = ld(y, h0 + i);
    ss = fmaf(v, v, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) t += red[w];
  const float rn = 1.f / sqrtf(t / (float)head_dim + eps);
  for (int i = threadIdx.x; i < head_dim; i += 256) {
    const float zz = ld(z, h0 + i);
    const float silu = zz / (1.f + expf(-zz));
    const float g = __uint_as_float((uint32_t)__ldg(gamma + h0 + i) << 16);
    x[h0 + i] = silu * g * (ld(y, h0 + i) * rn);
  }
}

int gated_norm_launch(const void* y, const void* z, int xt, const uint16_t* gamma, int n, int head_dim, float eps,
                      float* x, cudaStream_t stream) {
  if (head_dim < 1 || n % head_dim != 0) return QG_EINVAL;
  const dim3 grid((unsigned)(n / head_dim));
  return xt == QG_X_F32 ? launch(gated_norm_kernel<true>, grid, dim3(256), 0, stream, y, z, gamma, head_dim, eps, x)
                        : launch(gated_norm_kernel<false>, grid, dim3(256), 0, stream, y, z, gamma, head_dim, eps, x);
}

}  // namespace qg
