// gemv_dense.cu -- dense dequant-GEMV launches: one matrix, or n in {2,3,4} matrices sharing x
// ([FFAI#14] "dequant_gemv_int4_*", "dequantGemvInt4Two/Three/Four", "ffai_batched_4_qgemv_fast").
#include "gemv_kernel.cuh"

namespace qg {

GemvTune g_gemv_tune = {0};

int gemv_tune(int ctas_per_sm) {
  if (ctas_per_sm < 0 || ctas_per_sm > 4) return QG_EINVAL;
  g_gemv_tune = GemvTune{ctas_per_sm};
  return QG_OK;
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

}  // namespace qg
