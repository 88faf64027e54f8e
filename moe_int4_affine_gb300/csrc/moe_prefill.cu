// moe_prefill.cu -- the MoE layer for T tokens at once (prefill): every token routed to its top k of
// E experts, the tokens grouped by expert so that each expert's weights are read once per tile of
// up to n_tile of its tokens, on the tensor cores:
//   1. router     logits [T][E] -> idx, p [T][k]             (one warp per token)
//   2. plan       idx -> per-expert counts, tile offsets; the expert of every token tile and the
//                 grouped row of every (token, slot) pair (one CTA)
//   3. prep       X rows gathered into fp16 token tiles, grouped by expert (one block per pair;
//                 the tiles' padding rows are not written: an MMA output column depends on its own
//                 token row only, and padding outputs are never read)
//   4. gate/up    G, U [rows][inter] = grouped rows x W_g[e]^T, W_u[e]^T   (tcgen05, one launch)
//   5. prep       h = silu(G) * U into fp16 token tiles
//   6. down       D [rows][hidden] = h x W_d[e]^T                             (tcgen05)
//   7. combine    y[t] = residual[t] + sum_s p[t][s] * D[row of (t, s)]      (slot order)
// Each (token, slot) row is computed independently of the others, so the order of the rows within
// an expert's group (set by atomics in the plan) does not change any result.
// ([FFAI#9] moeGatherDequantGemmInt4 / mt_moe_gather_qmm_int4: the T*topK rows sorted by
// expert with CSR expert offsets, in row tiles of 8 to 64, built there from the top-K indices on
// the host; it loses to per-expert dispatches at T = 1 and is meant for prefill.  Here the offsets
// are built on the device, so no index readback precedes the expert GEMMs.)
#include <algorithm>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr int kPlanThreads = 1024;  // also the largest E: one thread per expert in the scan

// Token tile height: about twice the mean number of rows per expert (so that most experts fit in
// one tile and their weights are read once), a multiple of 16 in [16, 128].
int prefill_n_tile(int T, int k, int E) {
  const long long pairs = (long long)T * k;
  const long long mean = (pairs + E - 1) / E;
  const long long t = (2 * mean + 15) / 16 * 16;
  return (int)std::min<long long>(128, std::max<long long>(16, t));
}

// Token tiles that can be needed: every expert with rows adds at most one partial tile.
int prefill_max_tiles(int T, int k, int E, int n_tile) {
  const long long pairs = (long long)T * k;
  return (int)((pairs + n_tile - 1) / n_tile + std::min<long long>(E, pairs));
}

struct PrefillLayout {
  int n_tile, max_tiles, rows;
  size_t o_tile, o_pos, o_xt1, o_xs1, o_g, o_u, o_xt2, o_xs2, o_d, total;
};

size_t up256(size_t b) { return (b + 255) / 256 * 256; }

PrefillLayout prefill_layout(int T, int k, int E, int hidden, int inter) {
  PrefillLayout L{};
  L.n_tile = prefill_n_tile(T, k, E);
  L.max_tiles = prefill_max_tiles(T, k, E, L.n_tile);
  L.rows = L.max_tiles * L.n_tile;
  const size_t rows = (size_t)L.rows;
  size_t o = 0;
  L.o_tile = o;   o += up256((size_t)L.max_tiles * 4);
  L.o_pos = o;    o += up256((size_t)T * k * 4);
  L.o_xt1 = o;    o += up256(rows * hidden * 2);
  L.o_xs1 = o;    o += up256(rows * 4);
  L.o_g = o;      o += up256(rows * inter * 4);
  L.o_u = o;      o += up256(rows * inter * 4);
  L.o_xt2 = o;    o += up256(rows * inter * 2);
  L.o_xs2 = o;    o += up256(rows * 4);
  L.o_d = o;      o += up256(rows * hidden * 4);
  L.total = o + 256;  // slack for aligning the base
  return L;
}

// Step 2.  npairs = T k pairs (token t = i / k, slot i % k) with expert idx[i].
//   tile_expert[y]: the expert of token tile y (-1 past the last used tile);
//   pos[i]:         the grouped row of pair i (-1: an expert index >= E, which adds nothing and
//                   sets QG_STATUS_BAD_EXPERT).
// Expert e's rows start at tile offset toff[e] (exclusive scan of ceil(count_e / n_tile)).
__global__ void __launch_bounds__(kPlanThreads) moe_plan_kernel(const uint32_t* __restrict__ idx, int npairs, int E,
                                                                int n_tile, int max_tiles,
                                                                int* __restrict__ tile_expert, int* __restrict__ pos) {
  __shared__ int cnt[kPlanThreads];
  __shared__ int toff[kPlanThreads];
  __shared__ int wsum[kPlanThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();
  cnt[tid] = 0;
  for (int y = tid; y < max_tiles; y += kPlanThreads) tile_expert[y] = -1;
  __syncthreads();
  for (int i = tid; i < npairs; i += kPlanThreads) {
    const uint32_t e = idx[i];
    if (e < (uint32_t)E) {
      pos[i] = atomicAdd(&cnt[e], 1);  // rank within the expert's rows
    } else {
      pos[i] = -1;
      set_status(QG_STATUS_BAD_EXPERT);
    }
  }
  __syncthreads();
  // exclusive scan of the experts' tile counts
  const int own = tid < E ? (cnt[tid] + n_tile - 1) / n_tile : 0;
  int v = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) wsum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  const int incl = v + (warp > 0 ? wsum[warp - 1] : 0);
  if (tid < E) toff[tid] = incl - own;
  __syncthreads();
  if (tid < E) {
    for (int j = 0; j < own; ++j) tile_expert[toff[tid] + j] = tid;
  }
  for (int i = tid; i < npairs; i += kPlanThreads) {
    const uint32_t e = idx[i];
    if (e < (uint32_t)E) pos[i] = toff[e] * n_tile + pos[i];
  }
}

// Step 7.  One thread per four elements of one token's output row.
__global__ void __launch_bounds__(256) moe_combine_kernel(const float* __restrict__ p, const int* __restrict__ pos,
                                                          int k, const float* __restrict__ D, int hidden,
                                                          const uint16_t* __restrict__ residual,
                                                          float* __restrict__ y) {
  const int t = blockIdx.y;
  const int i = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
  pdl_trigger();
  pdl_wait();
  if (i >= hidden) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (residual) {
    const uint2 r = *reinterpret_cast<const uint2*>(residual + (size_t)t * hidden + i);
    acc = make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xFFFF0000u), __uint_as_float(r.y << 16),
                      __uint_as_float(r.y & 0xFFFF0000u));
  }
  for (int s = 0; s < k; ++s) {
    const int r = pos[t * k + s];
    if (r < 0) continue;
    const float ps = p[t * k + s];
    const float4 d = __ldg(reinterpret_cast<const float4*>(D + (size_t)r * hidden + i));
    acc.x = fmaf(ps, d.x, acc.x);
    acc.y = fmaf(ps, d.y, acc.y);
    acc.z = fmaf(ps, d.z, acc.z);
    acc.w = fmaf(ps, d.w, acc.w);
  }
  *reinterpret_cast<float4*>(y + (size_t)t * hidden + i) = acc;
}

}  // namespace

size_t moe_prefill_workspace_bytes(const qg_int4_weight* down, int T) {
  if (!down || T < 1) return 0;
  size_t best = 0;
  for (int k = 1; k <= 8; ++k)  // the tile height depends on k: room for any k <= 8
    best = std::max(best, prefill_layout(T, k, down->n_mat, down->out, down->in).total);
  return best;
}

int moe_prefill_launch(const float* logits, int T, int renorm, const qg_int4_weight* gate, const qg_int4_weight* up,
                       const qg_int4_weight* down, int k, const uint16_t* X, const uint16_t* residual, float* Y,
                       uint32_t* idx, float* p, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const int E = gate->n_mat, hidden = gate->in, inter = gate->out;
  if (E > kPlanThreads || (long long)T * k >= (1LL << 30)) return QG_ENOTSUP;
  const PrefillLayout L = prefill_layout(T, k, E, hidden, inter);
  if (ws_bytes < L.total) return QG_EWORKSPACE;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~(uintptr_t)255);
  int* tile_expert = reinterpret_cast<int*>(base + L.o_tile);
  int* pos = reinterpret_cast<int*>(base + L.o_pos);
  uint8_t* xt1 = base + L.o_xt1;
  float* xs1 = reinterpret_cast<float*>(base + L.o_xs1);
  float* G = reinterpret_cast<float*>(base + L.o_g);
  float* U = reinterpret_cast<float*>(base + L.o_u);
  uint8_t* xt2 = base + L.o_xt2;
  float* xs2 = reinterpret_cast<float*>(base + L.o_xs2);
  float* D = reinterpret_cast<float*>(base + L.o_d);

  int rc = router_batch_launch(logits, T, E, k, renorm, idx, p, stream);
  if (rc != QG_OK) return rc;
  rc = launch(moe_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, static_cast<const uint32_t*>(idx), T * k, E,
              L.n_tile, L.max_tiles, tile_expert, pos);
  if (rc != QG_OK) return rc;
  rc = qgemm_prep_pairs_launch(X, T, hidden, pos, T * k, k, L.n_tile, xt1, xs1, stream);
  if (rc != QG_OK) return rc;
  const qg_int4_weight gu[2] = {*gate, *up};
  float* const gy[2] = {G, U};
  rc = qgemm_tc_grouped_launch(gu, 2, xt1, xs1, L.max_tiles, L.n_tile, tile_expert, gy, stream);
  if (rc != QG_OK) return rc;
  rc = qgemm_prep_swiglu_launch(G, U, inter, pos, T * k, L.n_tile, xt2, xs2, stream);
  if (rc != QG_OK) return rc;
  float* const dy[1] = {D};
  rc = qgemm_tc_grouped_launch(down, 1, xt2, xs2, L.max_tiles, L.n_tile, tile_expert, dy, stream);
  if (rc != QG_OK) return rc;
  const int threads = 256;
  const dim3 grid((unsigned)((hidden / 4 + threads - 1) / threads), (unsigned)T);
  return launch(moe_combine_kernel, grid, dim3(threads), 0, stream, static_cast<const float*>(p),
                static_cast<const int*>(pos), k, static_cast<const float*>(D), hidden, residual, Y);
}

}  // namespace qg
