// qgemm_tc.cu -- tensor-core dequant-GEMM for T token rows ([FFAI#9] "Ops.dequantGemmDynamicM"):
//   Y[t][r] = sum_j w[r][j] * X[t][j],   w[r][j] = scale[r][j/64] * q[r][j] + bias[r][j/64]
// on the 5th-generation tensor cores (tcgen05.mma, accumulator in tensor memory), sm_103a.
//
// Work split: one CTA per (128 weight rows, n_tile tokens) tile; the MMA is D[128 x n_tile] +=
// A[128 x 16] * B[n_tile x 16]^T with A = the dequantized weights (fp16, in tensor memory, one
// weight row per lane) and B = the tokens (fp16, K-major in shared memory with the 128-byte
// swizzle), D fp32 in tensor memory.
//   * A pipeline stage covers GPS 64-column quantization groups (GPS = 2, K = 128; GPS = 4, K = 256
//     for tiles of at most 64 tokens, which halves the stage hand-overs that pace small tiles).
//     Two producer warp groups (4 warps each, one thread per weight row) fill them: group h makes
//     groups GPS j + 2 q + h of stage j (four groups, one group each, for the small tiles).  (The
//     warp after the MMA warp issues the stages' token-tile copies.)  A
//     thread streams its row's packed codes through a per-thread cp.async ring (WRING of its
//     groups ahead) -- with the scale and bias words (4-byte copies, through L1), or, for tiles of
//     128 tokens and more, with the scales and biases as 16-byte chunks of 8 groups in registers --
//     dequantizes the 64 weights of a group with packed half-precision arithmetic (w = s * q + b,
//     one rounding to fp16) and writes them with one tensor-memory store (tcgen05.st, 32 columns of
//     its row's lane) into the stage's A columns.
//     For tiles of at most 64 or at least 128 tokens (and in a multiple of 512; in grouped mode
//     with two CTAs per SM too) the weights come instead by TMA
//     tensor copies, eight groups of the 128 rows at a time (see kCodeBox), issued by a weight
//     loader warp into a ring of chunks; the producers read their row's codes from the swizzled
//     boxes.  The weights do not depend on the previous kernel, so they start streaming before the
//     dependency wait, which only the token loader and the epilogue take.
//   * The token tile of a stage is one contiguous block of the workspace (written there, already
//     swizzled, by the prep kernel) and arrives by a single bulk copy (TMA engine) into a ring of
//     token slots of its own (deeper than the A stages where shared memory allows).
//   * One thread of the MMA warp issues four K=16 MMAs per group and commits each stage to the
//     stage's "empty" mbarrier and to its token slot's; a final commit releases the epilogue, which
//     reads the accumulator from tensor memory (tcgen05.ld), applies each token's power-of-two
//     input scale and writes Y.
//   * Small token tiles are paced by the MMA instructions themselves: an M = 128, K = 16 MMA
//     occupies its issuing thread for 65-100 SM cycles whatever N is (measured), so a 128-row tile
//     of K = 5120 (320 MMAs) needs about 16 us from one thread.  Tiles of at most 64 tokens
//     therefore run four producer warp groups (one group per thread and stage) and two issuing
//     threads, each on its own accumulator, added in the epilogue (see MW and PG below).
//   * Every mbarrier wait is bounded (2 s): on a timeout the CTA records QG_STATUS_TIMEOUT, stops
//     issuing, drains what it has in flight and frees its tensor memory before returning.
//   * Grouped (MoE) mode: token tile y belongs to expert tile_expert[y]; the CTA reads it first
//     and takes that expert's slab of every matrix (unused tiles exit before any setup).  Tiles
//     of at most 64 tokens there run two CTAs per SM (256 tensor-memory columns each).
//
// Numerics: each token row of X is scaled by a power of two 2^(14 - e_t) (e_t = floor(log2 max|x_t|)),
// putting its largest magnitude in [2^14, 2^15), then rounded to fp16.  A bf16 value (8 significant
// bits) is exact in fp16 down to 2^-17 after scaling (fp16's subnormal step is 2^-24), i.e. for every
// element within 2^31 of its row's largest; smaller ones are off by at most 2^-25 (scaled).  Scales
// and biases convert to fp16 exactly when they lie in fp16's normal range (2^-14 <= |v| < 65504, or
// zero: required); the dequantized weight w~ = fl16(s q + b) is one fp16 rounding, |w~ - w| <=
// 2^-11 |w| (|w| >= 2^-14) or 2^-25.  The products of fp16 operands are exact in fp32; each MMA of
// K = 16 adds its 16 products to the fp32 accumulator with one rounding, taken here as at most
// 2^-23 relative to the magnitudes involved (the tensor cores' internal alignment and rounding are
// undocumented; this allows for truncation).  Over K: |y - y_exact| <= (2^-11 + (K / 16 + 1) 2^-23)
// sum |w x| plus the 2^-25 terms: 5.3e-4 at K = 5120, 6.2e-4 at K = 17408, 7.3e-4 at K = 32768 --
// inside the 1e-3 sum |w x| acceptance bound at every supported K.  Excluded inputs: token elements
// more than 2^31 below their row's largest, and weights below 2^-14 in magnitude, where the
// absolute terms above apply instead (the 1e-6 absolute part of the bound covers them only for
// rows of small magnitude).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {
namespace {

constexpr int kBM = 128;                     // weight rows per CTA (MMA M)
constexpr int kGK = 64;                      // columns of one quantization group = K of one stage
constexpr int kMaxN = 256;                   // tokens per CTA (MMA N, tensor-memory columns)
constexpr int kProducerWarps = 8;            // two warp groups of 4: one thread per weight row each
constexpr int kProducers = kProducerWarps * 32;
constexpr int kThreads = kProducers + 64;     // then the MMA warp and the token-tile loader (the
                                              // kernel's kWMma, kWLoad; kWCode for the tensor copies)
// CTMA (the one-CTA kernel): the weights arrive by TMA tensor copies in chunks of eight
// groups for the CTA's 128 rows -- the codes as two 128-row x 128-byte boxes (128-byte swizzle),
// then the scales and the biases as 128-row x 16-byte boxes -- instead of one cp.async per thread,
// group and word.  Each thread owns a weight row, so a warp's per-thread copies touch 32 rows'
// lines at once; the copy engine issues a box's lines without that per-request cost.
constexpr uint32_t kCodeBox = 128 * 128;            // one codes box (four groups of 128 rows)
constexpr uint32_t kSbBox = 128 * 16;               // one scales (or biases) box (eight groups)
constexpr uint32_t kCSlot = 2 * kCodeBox + 2 * kSbBox;  // one chunk: 36 KB (a multiple of 1024)
constexpr int kMaxStages = 4;
constexpr int kAccCols = 256;                // tensor memory: columns 0..255 accumulator, then per stage
constexpr int kACols = kGK / 2;              //   32 columns (64 fp16 per lane) of A per group,
// weight ring entry (one group per producer thread): the codes, plus the scale and bias words when
// they come through the ring (SBREG = false) rather than 16-byte chunks held in registers
__host__ __device__ constexpr int wstage_bytes(bool sbreg) { return sbreg ? kProducers * 32 : kProducers * 40; }
constexpr int kSmemBudget = 220 * 1024;

// One weight of a (multi-projection) call; its 128-row tiles are grid columns tile0, tile0 + 1, ...
struct TcMat {
  const uint32_t* packed;
  const uint16_t* scales;
  const uint16_t* biases;
  float* y;  // [T][out]
  int out;
  int tile0;
  long long ew, esb;  // grouped mode: expert e's codes at packed + e * ew, scales, biases at + e * esb
};
constexpr int kTcMaxMats = 4;

struct TcArgs {
  // CTMA: per matrix, tensor maps of the codes ([n_mat][out][in / 8] u32, box 32 x 128 x 1, 128-byte
  // swizzle), scales and biases ([n_mat][out][in / 64] u16, box 8 x 128 x 1)
  CUtensorMap tm_codes[kTcMaxMats], tm_scales[kTcMaxMats], tm_biases[kTcMaxMats];
  TcMat mat[kTcMaxMats];  // matrices sharing the tokens (same in)
  int nmat;
  // grouped (MoE) mode: token tile y belongs to expert tile_expert[y] (< 0: no tile, the CTA
  // exits); every matrix is then a stack of experts (TcMat::ew, esb)
  const int* tile_expert;
  const uint8_t* xt;  // token tiles: [n_tiles][k groups][n_tile][128 B], swizzled, fp16
  const float* xs;    // [n_tiles * n_tile] per-token output scale
  int in, T;
  int n_tile;
  int stages;   // A stages (tensor memory)
  int tstages;  // token-tile slots (shared memory; at least stages): loaded that many stages ahead
  uint32_t idesc;
};

// ---------------------------------------------------------------- tcgen05 / async helpers
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand with the 128-byte swizzle, 8-row groups 1024 bytes
// apart (stride byte offset), descriptor version 1, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;              // leading byte offset (not used by swizzled K-major layouts)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset
  d |= (uint64_t)1 << 46;              // version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}

// D (+)= A B with A in tensor memory (lane m = row m, K packed two fp16 per 32-bit column).
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// 32 consecutive 32-bit columns of this thread's lane (warp w % 4 owns lanes 32 (w % 4) .. + 31).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
// 32 lanes x 8 / 16 / 32 consecutive fp32 columns of tensor memory into registers (no wait).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* v) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
// Both barriers' phases complete?  The two tests are issued together (one latency, not two).
__device__ __forceinline__ bool test_wait2(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %3;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q, [%2], %4;\n\t"
      "and.pred p, p, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b0)), "r"(smem_u32(b1)), "r"(p0), "r"(p1)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// One box of a 3-D tensor map into shared memory, completion counted on bar in bytes.
__device__ __forceinline__ void tma3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// fp16x2 arithmetic on raw bits
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// bf16 bits (low 16 of v) -> fp16, in both halves
__device__ __forceinline__ uint32_t bf16_to_f16x2(uint32_t v) {
  const float f = __uint_as_float(v << 16);
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.f16.f32 t, %1;\n\tmov.b32 %0, {t, t};\n\t}" : "=r"(h) : "f"(f));
  return h;
}

// Eight codes of one u32 word (low nibble first) -> four fp16x2 words of w = s * q + b in the order
// (q0, q4), (q1, q5), (q2, q6), (q3, q7).  1024 + q is exact as the fp16 with exponent 10 and the
// nibble as its low mantissa bits; subtracting 1024 is exact, the fma rounds once.
__device__ __forceinline__ uint4 dequant8(uint32_t w, uint32_t s2, uint32_t b2) {
  const uint32_t k1024 = 0x64006400u;
  uint4 r;
  r.x = hfma2(hsub2((w & 0x000F000Fu) | k1024, k1024), s2, b2);
  r.y = hfma2(hsub2(((w >> 4) & 0x000F000Fu) | k1024, k1024), s2, b2);
  r.z = hfma2(hsub2(((w >> 8) & 0x000F000Fu) | k1024, k1024), s2, b2);
  r.w = hfma2(hsub2(((w >> 12) & 0x000F000Fu) | k1024, k1024), s2, b2);
  return r;
}

// TMEMC: tensor-memory columns the CTA allocates.  512: accumulator in columns 0-255 (N <= 256), A
// stages from column 256 (up to four).  256: accumulator in columns 0-63 (N <= 64), up to three A
// stages from column 64 -- two such CTAs share an SM (with at most half its shared memory each), so
// one CTA's start and epilogue overlap the other's main loop (many short tiles: grouped mode).
// SBREG: scales and biases as 16-byte chunks in registers (faster for token tiles of 128 and more:
// T = 256 54.3 -> 49.6 us) or as 4-byte copies through the weight ring (faster for small tiles).
// GPS: quantization groups per pipeline stage (K = 64 GPS).  Four halve the number of stage
// hand-overs for small token tiles (accumulator N <= 64 in columns 0-63, up to three A stages of 128
// columns from column 64); two otherwise.
// CTMA: the weights by TMA tensor copies (kCSlot chunks, a ring of WRING of them; see kCodeBox).
// MW: MMA-issuing warps.  An MMA instruction occupies its issuing thread for about 65 cycles
// whatever N is (measured), so small token tiles are issue-bound with one: with MW = 2 (four-group
// stages, N <= 64) a second MMA warp (the one after the weight loader) issues groups 2 and 3 of
// every stage into a second accumulator in the last 64 tensor-memory columns, and the epilogue adds
// the two.
// PG: producer warp groups (4 with the tensor copies and four-group stages: one group per thread
// and stage; warps 8 .. 15 then make groups 2, 3 and do not take part in the epilogue).
template <int WRING, int TMEMC, bool SBREG, int GPS, bool CTMA = false, int MW = 1, int PG = 2>
__global__ void __launch_bounds__((CTMA ? 128 * PG + 96 : kThreads) + (MW - 1) * 32, TMEMC == 256 ? 2 : 1)
    qgemm_tc_kernel(const __grid_constant__ TcArgs a) {
  static_assert(GPS == 2 || (GPS == 4 && TMEMC == 512), "four groups per stage: one-CTA kernel only");
  static_assert(!CTMA || !SBREG, "tensor copies: ring scales only");
  static_assert(MW == 1 || (MW == 2 && CTMA && GPS == 4 && TMEMC == 512), "two MMA warps: the small-tile kernel");
  static_assert(PG == 2 || (PG == 4 && CTMA && GPS == 4), "four producer groups: tensor copies, four-group stages");
  constexpr uint32_t kAcc2 = 448;  // MW = 2: the second accumulator's first column
  constexpr int kPW = 4 * PG;       // producer warps; then the MMA, token-loader, weight-loader warps
  constexpr int kWMma = kPW, kWLoad = kPW + 1, kWCode = kPW + 2;
  constexpr int kQS = GPS / PG;     // groups per producer thread and stage
  constexpr int kJC = 8 / PG;       // a thread's groups per weight chunk (eight groups)
  constexpr uint32_t kABase = (TMEMC == 512 && GPS == 2) ? (uint32_t)kAccCols : 64u;
  constexpr uint32_t kAStageT = (uint32_t)(GPS * kACols);  // A columns of one stage
  constexpr int kWStageBytes = wstage_bytes(SBREG);
  constexpr size_t kRingBytes = CTMA ? (size_t)WRING * kCSlot : (size_t)WRING * kWStageBytes;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* basep = smem_raw + (base - raw);
  const int S = a.stages, D = a.tstages;
  const uint32_t btile = (uint32_t)a.n_tile * 128u;  // token tile of one group (the stage)
  const uint32_t stage_bytes = GPS * btile;  // the token tiles of a stage's groups
  const uint32_t wring = base + (uint32_t)D * stage_bytes;  // weight staging ring (CTMA: chunks, 1024-aligned)
  // full[s] / empty[s]: A stage s written by the producers / its MMAs done; bfull[t] / tempty[t]:
  // token slot t's bytes landed / the MMAs that read it done
  uint64_t* full = reinterpret_cast<uint64_t*>(basep + (size_t)D * stage_bytes + kRingBytes);
  uint64_t* empty = full + S;
  uint64_t* bfull = empty + S;
  uint64_t* tempty = bfull + D;
  uint64_t* done = tempty + D;
  // CTMA: cfull[c]: chunk slot c's bytes landed; cempty[c]: every producer warp has read it
  uint64_t* cfull = done + 1;
  uint64_t* cempty = cfull + (CTMA ? WRING : 0);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cempty + (CTMA ? WRING : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int mi = 0;  // this CTA's matrix: the last one whose first tile is at or before blockIdx.x
  while (mi + 1 < a.nmat && (int)blockIdx.x >= a.mat[mi + 1].tile0) ++mi;
  TcMat mt = a.mat[mi];
  int ez = 0;  // the expert (the tensor maps' third coordinate)
  if (a.tile_expert) {  // grouped: the tile table is the previous kernel's output
    pdl_wait();
    const int e = a.tile_expert[blockIdx.y];
    if (e < 0) return;  // (before any barrier, tensor memory or copy: the whole CTA leaves)
    ez = e;
    mt.packed += (size_t)e * (size_t)mt.ew;
    mt.scales += (size_t)e * (size_t)mt.esb;
    mt.biases += (size_t)e * (size_t)mt.esb;
  }
  const int m0 = ((int)blockIdx.x - mt.tile0) * kBM;
  const int tile = blockIdx.y, n0 = tile * a.n_tile;
  const int nk = a.in / kGK;         // groups
  const int nst = (nk + GPS - 1) / GPS;  // pipeline stages (GPS groups each)

  if (warp == kWMma) {
    if (lane == 0) {
      for (int s = 0; s < S; ++s) {
        mbar_init(full + s, kPW);
        mbar_init(empty + s, MW);  // (one commit from each MMA warp)
      }
      for (int t = 0; t < D; ++t) {
        mbar_init(bfull + t, 1);
        mbar_init(tempty + t, MW);
      }
      mbar_init(done, MW);
      if constexpr (CTMA) {
        for (int c = 0; c < WRING; ++c) {
          mbar_init(cfull + c, 1);
          mbar_init(cempty + c, kPW);
        }
      }
      *abort_flag = 0;
      mbar_fence_init();
    }
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEMC)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Only the token tiles and their scales come from the previous kernel (the staging kernel): the
  // token loader and the epilogue wait for it; the weights start streaming at once.
  pdl_trigger();

  if (warp < kPW) {
    // ---------------- producers: thread (row r, warp group h) makes group 2 j + h of every stage j
    const int r = tid & (kBM - 1), h = tid >> 7;
    const int row = m0 + r;
    const bool rv = row < mt.out;
    const int rowc = rv ? row : mt.out - 1;
    const int ngs = a.in / 64;
    const int my_n = (nk - h + 1) / 2;  // groups of this thread
    // group 2 jj + h: codes advance by 16 words per jj, the scale / bias index by 2
    const uint32_t* wp = mt.packed + (size_t)rowc * (a.in / 8) + (size_t)h * 8;
    const size_t e0 = (size_t)rowc * ngs + h;  // scale / bias element of this thread's group 0
    const size_t n_sb = (size_t)mt.out * ngs;
    const uint32_t wcode = wring + (uint32_t)tid * 16;  // chunk c at + c * kProducers * 16
    const uint32_t wsb = wring + kProducers * 32 + (uint32_t)tid * 8;  // (SBREG = false)
    const int odd = (int)(e0 & 1);  // which half of a copied 32-bit word holds s and b
    auto wissue = [&](int jj) {  // this thread's copies for its group jj (an empty group past the end)
      if (jj < my_n) {
        const uint32_t g = (uint32_t)(jj % WRING) * kWStageBytes;
        const uint32_t* src = wp + (size_t)jj * 16;
        cp16(wcode + g, src, rv ? 16u : 0u);
        cp16(wcode + g + kProducers * 16, src + 4, rv ? 16u : 0u);
        if constexpr (!SBREG) {
          const size_t e = e0 + 2 * (size_t)jj, eo = e & ~(size_t)1;
          const uint32_t nb = rv ? (eo + 1 < n_sb ? 4u : 2u) : 0u;
          cp4(wsb + g, mt.scales + eo, nb);
          cp4(wsb + g + 4, mt.biases + eo, nb);
        }
      }
      cp_commit();
    };
    // Scales and biases: 16-byte chunks of 8 consecutive elements (4 of this thread's groups) held
    // in registers, the next chunk loaded while the current one is used.  At the array's end (or
    // for arrays not 16-byte aligned) element by element, nothing read past the end.
    const bool sb_vec = ((reinterpret_cast<uintptr_t>(mt.scales) | reinterpret_cast<uintptr_t>(mt.biases)) & 15u) == 0;
    auto ld_chunk = [&](size_t q, uint4& sc, uint4& bc) {
      if (sb_vec && 8 * q + 8 <= n_sb) {
        sc = __ldg(reinterpret_cast<const uint4*>(mt.scales) + q);
        bc = __ldg(reinterpret_cast<const uint4*>(mt.biases) + q);
      } else {
        uint32_t s4[4] = {0u, 0u, 0u, 0u}, b4[4] = {0u, 0u, 0u, 0u};
        for (int i = 0; i < 8; ++i) {
          const size_t el = 8 * q + (size_t)i;
          if (el < n_sb) {
            s4[i >> 1] |= (uint32_t)__ldg(mt.scales + el) << (16 * (i & 1));
            b4[i >> 1] |= (uint32_t)__ldg(mt.biases + el) << (16 * (i & 1));
          }
        }
        sc = make_uint4(s4[0], s4[1], s4[2], s4[3]);
        bc = make_uint4(b4[0], b4[1], b4[2], b4[3]);
      }
    };
    auto pick16 = [](const uint4& v, int o) {  // element o (0..7) of a chunk
      const int w = o >> 1;
      const uint32_t x = w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
      return (o & 1) ? x >> 16 : x & 0xFFFFu;
    };
    size_t qc = e0 >> 3;  // the chunk in s_cur / b_cur
    uint4 s_cur{}, b_cur{}, s_nxt{}, b_nxt{};
    if constexpr (SBREG) {
      ld_chunk(qc, s_cur, b_cur);
      ld_chunk(qc + 1, s_nxt, b_nxt);
    }
    if constexpr (!CTMA) {
#pragma unroll 1
      for (int jj = 0; jj < WRING - 1; ++jj) wissue(jj);
    }
    uint32_t csl = 0;  // CTMA: the current chunk's slot

    for (int j = 0; j < nst; ++j) {  // stage j: groups GPS j + 2 q + h, q < GPS / 2 (thread group jj)
      const int s = j % S;
      if (j >= S && !mbar_wait(empty + s, (uint32_t)(j / S - 1) & 1u)) *abort_flag = 1;
      if (*abort_flag) break;
      tc_fence_after();  // the MMAs that read this stage's A columns have completed
#pragma unroll
      for (int q = 0; q < kQS; ++q) {
        const int jj = kQS * j + q;  // this thread's group PG jj + h (its jj-th)
        if constexpr (CTMA) {
          if (jj % kJC == 0) {  // chunk jj / kJC (groups 8 c ..): its bytes, then this row's scales and biases
            const int c = jj / kJC;
            csl = wring + (uint32_t)(c % WRING) * kCSlot;
            if (!mbar_wait(cfull + c % WRING, (uint32_t)(c / WRING) & 1u)) *abort_flag = 1;
            s_cur = lds128(csl + 2 * kCodeBox + (uint32_t)r * 16u);
            b_cur = lds128(csl + 2 * kCodeBox + kSbBox + (uint32_t)r * 16u);
          }
        } else {
          wissue(jj + WRING - 1);
          cp_wait<WRING - 1>();  // group jj of this thread has landed
        }
        const bool live = PG * jj + h < nk && !(CTMA && __any_sync(0xffffffffu, *abort_flag != 0));
        if (live) {  // (uniform per warp: tcgen05.st is a warp-wide instruction)
          uint4 c0, c1;
          uint32_t s2, b2;
          if constexpr (CTMA) {
            // group o of the chunk: codes box o / 4, 16-byte pieces 2 (o % 4) and 2 (o % 4) + 1 of
            // row r, each at its swizzled place (piece i of row r at i ^ (r % 8))
            const int o = (PG * jj + h) & 7;
            const uint32_t ra = csl + (uint32_t)(o >> 2) * kCodeBox + (uint32_t)r * 128u;
            const uint32_t sw = (uint32_t)(r & 7);
            c0 = lds128(ra + (((uint32_t)(2 * (o & 3)) ^ sw) << 4));
            c1 = lds128(ra + (((uint32_t)(2 * (o & 3) + 1) ^ sw) << 4));
            s2 = bf16_to_f16x2(pick16(s_cur, o));
            b2 = bf16_to_f16x2(pick16(b_cur, o));
          } else if constexpr (SBREG) {
            const uint32_t g = (uint32_t)(jj % WRING) * kWStageBytes;
            c0 = lds128(wcode + g);
            c1 = lds128(wcode + g + kProducers * 16);
            const size_t e = e0 + 2 * (size_t)jj;  // (advances 2 per group: at most one chunk)
            if ((e >> 3) != qc) {
              s_cur = s_nxt;
              b_cur = b_nxt;
              ++qc;
              ld_chunk(qc + 1, s_nxt, b_nxt);
            }
            s2 = bf16_to_f16x2(pick16(s_cur, (int)(e & 7)));
            b2 = bf16_to_f16x2(pick16(b_cur, (int)(e & 7)));
          } else {
            const uint32_t g = (uint32_t)(jj % WRING) * kWStageBytes;
            c0 = lds128(wcode + g);
            c1 = lds128(wcode + g + kProducers * 16);
            const uint32_t sw = lds32(wsb + g), bw = lds32(wsb + g + 4);
            s2 = bf16_to_f16x2(odd ? sw >> 16 : sw & 0xFFFFu);
            b2 = bf16_to_f16x2(odd ? bw >> 16 : bw & 0xFFFFu);
          }
          const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          uint32_t v[32];  // column 4 ch + i: the fp16 pair i of 8-column chunk ch
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 d = dequant8(cw[ch], s2, b2);
            v[4 * ch + 0] = d.x;
            v[4 * ch + 1] = d.y;
            v[4 * ch + 2] = d.z;
            v[4 * ch + 3] = d.w;
          }
          tmem_st32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) +
                        (kABase + kAStageT * (uint32_t)s + (uint32_t)(kACols * (PG * q + h))),
                    v);
        }
        if constexpr (CTMA) {
          if (jj % kJC == kJC - 1) {  // this warp has read the chunk
            __syncwarp();
            if (lane == 0) mbar_arrive(cempty + (jj / kJC) % WRING);
          }
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(full + s);
    }
    cp_wait<0>();
  } else if (warp == kWLoad) {
    // ---------------- token-tile loader: stage j's tiles (contiguous in the workspace), one bulk
    // copy each, issued as soon as the stage is free
    if (lane == 0) {
      pdl_wait();
      int issued = 0;
      for (int j = 0; j < nst; ++j) {
        const int t = j % D;
        if (j >= D && !mbar_wait(tempty + t, (uint32_t)(j / D - 1) & 1u)) *abort_flag = 1;
        if (*abort_flag) break;
        const uint32_t bytes = (uint32_t)min(GPS, nk - GPS * j) * btile;
        mbar_arrive_expect_tx(bfull + t, bytes);
        bulk_g2s(base + (uint32_t)t * stage_bytes, a.xt + ((size_t)tile * nk + (size_t)GPS * j) * btile, bytes,
                 bfull + t);
        ++issued;
      }
      // every bulk copy issued here has landed before the CTA can exit (normally long since: the MMA
      // thread waited for it); the latest use of each slot may be outstanding
      for (int j = max(0, issued - D); j < issued; ++j) mbar_wait(bfull + j % D, (uint32_t)(j / D) & 1u);
    }
  } else if (CTMA && warp == kWCode) {
    // ---------------- weight-chunk loader: chunk c (groups 8c .. 8c + 7 of the CTA's 128 rows) into
    // slot c % WRING as soon as every producer warp has read the chunk before it there
    if (lane == 0) {
      const int nch = (nk + 7) / 8;
      const int y0 = m0;  // first row within the matrix
      int issued = 0;
      for (int c = 0; c < nch; ++c) {
        const int sl = c % WRING;
        if (c >= WRING && !mbar_wait(cempty + sl, (uint32_t)(c / WRING - 1) & 1u)) *abort_flag = 1;
        if (*abort_flag) break;
        const uint32_t d = wring + (uint32_t)sl * kCSlot;
        mbar_arrive_expect_tx(cfull + sl, kCSlot);
        tma3d(d, &a.tm_codes[mi], 64 * c, y0, ez, cfull + sl);
        tma3d(d + kCodeBox, &a.tm_codes[mi], 64 * c + 32, y0, ez, cfull + sl);
        tma3d(d + 2 * kCodeBox, &a.tm_scales[mi], 8 * c, y0, ez, cfull + sl);
        tma3d(d + 2 * kCodeBox + kSbBox, &a.tm_biases[mi], 8 * c, y0, ez, cfull + sl);
        ++issued;
      }
      // every copy issued here has landed before the CTA can exit
      for (int c = max(0, issued - WRING); c < issued; ++c) mbar_wait(cfull + c % WRING, (uint32_t)(c / WRING) & 1u);
    }
  } else if ((warp == kWMma || (MW == 2 && warp == kPW + 3)) && lane == 0) {
    // ---------------- MMA issuer (MW = 2: issuer m takes groups 2 m, 2 m + 1 of each stage into
    // its own accumulator)
    const int m = warp == kWMma ? 0 : 1;
    const uint32_t dacc = tmem + (m ? kAcc2 : 0u);
    const int gi0 = MW == 2 ? 2 * m : 0, gi1 = MW == 2 ? 2 * m + 2 : GPS;
    // B descriptors: token slot t and K step k add (t * stage_bytes + 32 k) / 16 to the start
    // address field (bits 0-13: shared addresses stay below 2^18, so the field never carries).
    const uint64_t db0 = smem_desc(base);
    const uint32_t dstage = stage_bytes >> 4;
    int s = 0, t = 0;
    uint32_t ph = 0, pt = 0;  // parities of A stage s's and token slot t's current uses
    for (int j = 0; j < nst; ++j) {
      // (fast path: both already complete; else the bounded waits, which also watch the flag)
      if (!test_wait2(full + s, ph, bfull + t, pt)) {
        if (!mbar_wait(full + s, ph) || !mbar_wait(bfull + t, pt)) *abort_flag = 1;
        if (*abort_flag) break;
      }
      tc_fence_after();  // the producers' tensor-memory stores are complete
      const uint64_t db = db0 + (uint64_t)(t * dstage);
      const uint32_t ta = tmem + kABase + kAStageT * (uint32_t)s;
      const int ng = min(gi1, nk - GPS * j);
      for (int gi = gi0; gi < ng; ++gi) {
#pragma unroll
        for (int k = 0; k < kGK / 16; ++k)
          mma_f16_ta(dacc, ta + kACols * gi + 8 * k, db + (uint64_t)(gi * (btile >> 4)) + 2 * k, a.idesc,
                     (j | (gi - gi0) | k) != 0 ? 1u : 0u);
      }
      mma_commit(empty + s);
      mma_commit(tempty + t);
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
      if (++t == D) {
        t = 0;
        pt ^= 1u;
      }
    }
    mma_commit(done);  // arrives once every MMA issued above has completed
  }

  // ---------------- epilogue: warps w and w + 4 read lanes 32 (w % 4) .. + 31, half of the columns each
  if (warp < 8) {
    pdl_wait();  // (the token scales; and Y is written only after the kernels before this one are done)
    const bool ok = mbar_wait(done, 0);
    tc_fence_after();
    if (ok && !*abort_flag) {
      const int q = warp & 3;
      const int row = m0 + q * 32 + lane;
      const int half = a.n_tile / 2;  // multiple of 8
      const int c0 = (warp >> 2) * half;
      const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0;
      // W columns from cc: one wait per load (32 columns at a time where they fit, 16 with two
      // accumulators); the token scales loaded one per lane before it and passed round by shuffles
      // (17408 x 5120, T = 256: 42.0 -> 39.6 us against eight columns per wait)
      auto emit = [&](int cc, auto wc) {
        constexpr int W = decltype(wc)::value;
        const int tq = n0 + c0 + cc + (lane & (W - 1));
        const float xsl = tq < a.T ? __ldg(a.xs + tq) : 0.f;
        uint32_t v[W];
        auto ld = [](uint32_t ta, uint32_t* r) {
          if constexpr (W == 32) tmem_ld32(ta, r); else if constexpr (W == 16) tmem_ld16(ta, r); else tmem_ld8(ta, r);
        };
        ld(tl + (uint32_t)cc, v);
        if (MW == 2 && nk > 2) {  // (the second issuer's partial sum: groups 2, 3 of each stage)
          uint32_t w2[W];
          ld(tl + kAcc2 + (uint32_t)cc, w2);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int j = 0; j < W; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(w2[j]));
        }
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int j = 0; j < W; ++j) {
          const int t = n0 + c0 + cc + j;
          const float xv = __shfl_sync(0xffffffffu, xsl, j);
          if (row < mt.out && t < a.T) mt.y[(size_t)t * mt.out + row] = __uint_as_float(v[j]) * xv;
        }
      };
      int cc = 0;
      // (two CTAs per SM: eight, the other CTA's main loop hides the latency and the registers
      // stay fewer)
      constexpr int kW = MW == 2 ? 16 : TMEMC == 256 ? 8 : 32;
      for (; cc + kW <= half; cc += kW) emit(cc, std::integral_constant<int, kW>{});
      for (; cc < half; cc += 8) emit(cc, std::integral_constant<int, 8>{});
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEMC) : "memory");
  }
}

// ---------------------------------------------------------------- prep: X -> scaled fp16 token tiles
// One CTA per token row n < n_tiles * n_tile.  Row n of tile n / n_tile, group kc: 128 bytes at
// ((tile * nk + kc) * n_tile + n % n_tile) * 128, the 16-byte chunk j (columns 8j .. 8j + 7 of the
// group) at position j ^ (n % 8), its eight values in the column order 0, 4, 1, 5, 2, 6, 3, 7 (the
// order the dequantized weights use).  Rows n >= T are zero.  Grouped mode (rowpos != null): block
// t converts X row t once and writes it as rows rowpos[t kdiv + s], s < kdiv (< 0: none) -- the
// token's (token, slot) pairs placed in their experts' tiles; the tiles' padding rows are left
// unwritten (each MMA output column depends on its own token row only, and padding outputs are
// never read).
constexpr int kPrepThreads = 256;
constexpr int kPrepMaxChunks = 16;  // 16-byte chunks per thread: in <= 16 * 256 * 8 = 32768
constexpr int kPrepMaxFan = 8;      // grouped rows per token (top k <= 8)

__global__ void __launch_bounds__(kPrepThreads) qgemm_prep_kernel(const uint16_t* __restrict__ X, int T, int in,
                                                                   int n_tile, const int* __restrict__ rowpos,
                                                                   int kdiv, uint8_t* __restrict__ xt,
                                                                   float* __restrict__ xs) {
  __shared__ uint32_t red[kPrepThreads / 32];
  const int nk = in / 64, nch = in / 8;
  pdl_trigger();
  pdl_wait();
  const int src = (int)blockIdx.x;
  const int nfan = rowpos ? min(kdiv, kPrepMaxFan) : 1;
  int dn[kPrepMaxFan];  // the rows this block writes (< 0: none)
  bool any = false;
#pragma unroll
  for (int s = 0; s < kPrepMaxFan; ++s) {
    dn[s] = s < nfan ? (rowpos ? rowpos[(size_t)src * kdiv + s] : src) : -1;
    any |= dn[s] >= 0;
  }
  if (!any) return;  // (uniform per block)
  const bool live = src < T;
  const uint4* xr = reinterpret_cast<const uint4*>(X + (size_t)(live ? src : 0) * in);
  // one round of loads; the largest |x| from the bit patterns (|bf16| bits are ordered like values)
  uint4 raw[kPrepMaxChunks];
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < kPrepMaxChunks; ++i) {
    const int ch = (int)threadIdx.x + i * kPrepThreads;
    raw[i] = live && ch < nch ? __ldg(xr + ch) : make_uint4(0u, 0u, 0u, 0u);
    mx = __vmaxu2(mx, raw[i].x & 0x7FFF7FFFu);
    mx = __vmaxu2(mx, raw[i].y & 0x7FFF7FFFu);
    mx = __vmaxu2(mx, raw[i].z & 0x7FFF7FFFu);
    mx = __vmaxu2(mx, raw[i].w & 0x7FFF7FFFu);
  }
  mx = max(mx & 0xFFFFu, mx >> 16);
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0;
#pragma unroll
  for (int w = 0; w < kPrepThreads / 32; ++w) mx = max(mx, red[w]);
  const float m = __uint_as_float(mx << 16);
  // 2^(14 - e) with e = floor(log2 m): the row's largest magnitude lands in [2^14, 2^15)
  const int e = m > 0.f ? (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127 : 0;
  const float sc = live && m > 0.f ? exp2i(min(max(14 - e, -126), 127)) : 0.f;
#pragma unroll
  for (int s = 0; s < kPrepMaxFan; ++s)
    if ((int)threadIdx.x == s && dn[s] >= 0) xs[dn[s]] = live && m > 0.f ? exp2i(min(max(e - 14, -126), 127)) : 0.f;
#pragma unroll
  for (int i = 0; i < kPrepMaxChunks; ++i) {
    const int ch = (int)threadIdx.x + i * kPrepThreads;
    if (ch >= nch) break;
    const int kc = ch >> 3, j = ch & 7;
    const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    float f[8];  // the chunk's 8 values, scaled
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[2 * q] = __uint_as_float(w[q] << 16) * sc;
      f[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u) * sc;
    }
    // fp16 pairs in the column order 0, 4, 1, 5, 2, 6, 3, 7 (low half first)
    uint4 o;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o.x) : "f"(f[4]), "f"(f[0]));
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o.y) : "f"(f[5]), "f"(f[1]));
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o.z) : "f"(f[6]), "f"(f[2]));
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o.w) : "f"(f[7]), "f"(f[3]));
#pragma unroll
    for (int s = 0; s < kPrepMaxFan; ++s) {
      if (dn[s] < 0) continue;
      const int tile = dn[s] / n_tile, nl = dn[s] % n_tile;
      uint8_t* dst = xt + (((size_t)tile * nk + kc) * n_tile + nl) * 128 + (size_t)((j ^ (nl & 7)) << 4);
      *reinterpret_cast<uint4*>(dst) = o;
    }
  }
}

// The down projection's token tiles in grouped (MoE) mode: block i makes row n = rowpos[i] (< 0:
// nothing), h = silu(G[n]) * U[n] (fp32 [rows][in], the grouped gate/up outputs), scaled by a power
// of two and stored as above.  Two passes over the row (its largest |h|, then the conversion; the
// second reads hit L2), so in is not limited by registers.
__device__ __forceinline__ void swiglu8(const float* __restrict__ G, const float* __restrict__ U, size_t off,
                                        float (&h)[8]) {
  const float4* g4 = reinterpret_cast<const float4*>(G + off);
  const float4* u4 = reinterpret_cast<const float4*>(U + off);
  const float4 ga = __ldg(g4), gb = __ldg(g4 + 1), ua = __ldg(u4), ub = __ldg(u4 + 1);
  const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
  const float u[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
  for (int q = 0; q < 8; ++q) h[q] = g[q] / (1.f + expf(-g[q])) * u[q];
}

__global__ void __launch_bounds__(kPrepThreads) qgemm_prep_swiglu_kernel(const float* __restrict__ G,
                                                                          const float* __restrict__ U, int in,
                                                                          int n_tile, const int* __restrict__ rowpos,
                                                                          uint8_t* __restrict__ xt,
                                                                          float* __restrict__ xs) {
  __shared__ float red[kPrepThreads / 32];
  const int nk = in / 64, nch = in / 8;
  pdl_trigger();
  pdl_wait();
  const int n = rowpos[blockIdx.x];
  if (n < 0) return;  // (uniform per block)
  const bool live = true;
  const size_t row0 = (size_t)n * in;
  float mx = 0.f;
  if (live) {
    for (int ch = threadIdx.x; ch < nch; ch += kPrepThreads) {
      float h[8];
      swiglu8(G, U, row0 + (size_t)ch * 8, h);
#pragma unroll
      for (int q = 0; q < 8; ++q) mx = fmaxf(mx, fabsf(h[q]));
    }
  }
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0.f;
#pragma unroll
  for (int w = 0; w < kPrepThreads / 32; ++w) mx = fmaxf(mx, red[w]);
  const int e = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127 : 0;
  const float sc = mx > 0.f ? exp2i(min(max(14 - e, -126), 127)) : 0.f;
  if (threadIdx.x == 0) xs[n] = mx > 0.f ? exp2i(min(max(e - 14, -126), 127)) : 0.f;
  const int tile = n / n_tile, nl = n % n_tile;
  for (int ch = threadIdx.x; ch < nch; ch += kPrepThreads) {
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (live) {
      swiglu8(G, U, row0 + (size_t)ch * 8, f);
#pragma unroll
      for (int q = 0; q < 8; ++q) f[q] *= sc;
    }
    const int kc = ch >> 3, j = ch & 7;
    uint4 o;  // fp16 pairs in the column order 0, 4, 1, 5, 2, 6, 3, 7 (low half first)
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o.x) : "f"(f[4]), "f"(f[0]));
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o.y) : "f"(f[5]), "f"(f[1]));
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o.z) : "f"(f[6]), "f"(f[2]));
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(o.w) : "f"(f[7]), "f"(f[3]));
    uint8_t* dst = xt + (((size_t)tile * nk + kc) * n_tile + nl) * 128 + (size_t)((j ^ (nl & 7)) << 4);
    *reinterpret_cast<uint4*>(dst) = o;
  }
}

struct TcPlan {
  int n_tile, n_tiles, stages, wring;  // (ctma: wring = chunks in the ring)
  size_t smem;
  bool ctma;   // weights by TMA tensor copies (tiles of at most 64 tokens)
  int mw = 1;  // MMA-issuing warps
  int pg = 2;  // producer warp groups
  int tstages;  // token-tile slots (>= stages)
  int tmem;    // tensor-memory columns per CTA (512, or 256 for two CTAs per SM)
  bool sbreg;  // scales and biases in registers (token tiles of 128 and more, one CTA per SM)
  int gps;     // quantization groups per pipeline stage (4 for tiles of at most 64 tokens)
};

// Pipeline depth and weight ring for a token tile of n_tile rows (a multiple of 16, <= kMaxN).
TcPlan tc_plan_ntile(int n_tile) {
  TcPlan p{};
  p.n_tile = n_tile;
  p.n_tiles = 1;
  p.sbreg = n_tile >= 128;
  p.gps = n_tile <= 64 ? 4 : 2;
  const size_t kWStageBytes = (size_t)wstage_bytes(p.sbreg);
  const size_t stage = (size_t)p.gps * p.n_tile * 128;  // token tiles of a stage's groups
  const size_t fixed = 1024 + 64 + 8 * 32;          // alignment slack, barriers, slot, flag
  // stages: at most kMaxStages (tensor-memory columns for A); the rest of shared memory goes to the
  // weight ring (memory latency)
  // (four-group stages: three fit the tensor memory after a 64-column accumulator)
  p.stages = (int)std::min<size_t>(p.gps == 4 ? 3 : kMaxStages, (kSmemBudget - fixed - 2 * (size_t)kWStageBytes) / stage);
  const size_t left = kSmemBudget - fixed - (size_t)p.stages * stage;
  p.wring = left >= 16 * (size_t)kWStageBytes ? 16 : left >= 8 * (size_t)kWStageBytes ? 8 : left >= 4 * (size_t)kWStageBytes ? 4 : 2;
  // scale/bias copies through L1 (tiles of 32 to 64 tokens): an eight-group ring leaves more shared
  // memory to L1 (17408x5120 T = 32: 39.5 -> 37.3 us against sixteen groups; 16-token tiles keep
  // sixteen: T = 8 39.3 us against 47.1 with eight)
  if (!p.sbreg && n_tile >= 32 && p.wring > 8) p.wring = 8;
  p.smem = fixed + (size_t)p.stages * stage + (size_t)p.wring * kWStageBytes;
  p.tstages = p.stages;
  p.tmem = 512;
  return p;
}

// Two CTAs per SM (grouped mode, n_tile <= 64): 256 tensor-memory columns (three A stages) and at
// most kSmemHalf bytes of shared memory each.
constexpr size_t kSmemHalf = 110 * 1024;
TcPlan tc_plan_ntile_pair(int n_tile) {
  TcPlan p{};
  p.n_tile = n_tile;
  p.n_tiles = 1;
  p.sbreg = false;
  p.gps = 2;
  const size_t kWStageBytes = (size_t)wstage_bytes(false);
  p.tmem = 256;
  const size_t stage = 2 * (size_t)n_tile * 128;
  const size_t fixed = 1024 + 64 + 8 * 32;
  p.stages = (int)std::min<size_t>(3, (kSmemHalf - fixed - 2 * (size_t)kWStageBytes) / stage);
  const size_t left = kSmemHalf - fixed - (size_t)p.stages * stage;
  // a four-group weight ring: less shared memory leaves more L1 for the scale/bias loads (faster
  // than eight groups: MoE prefill T = 256, 232.7 -> 219.0 us)
  p.wring = left >= 4 * (size_t)kWStageBytes ? 4 : 2;
  p.smem = fixed + (size_t)p.stages * stage + (size_t)p.wring * kWStageBytes;
  p.tstages = p.stages;
  return p;
}

// The weights by tensor copies: scale rows a multiple of 16 bytes (in a multiple of 512, which the
// tensor maps' strides need).  Three (four-group) or four (two-group) A stages in tensor memory; a
// ring of three weight chunks (108 KB; two for 256-token tiles); the rest of the shared memory to
// token-tile slots (up to twelve), so that the token tiles load ahead of the A stages.
TcPlan tc_plan_ctma(int n_tile) {
  TcPlan p = tc_plan_ntile(n_tile);
  const size_t stage = (size_t)p.gps * p.n_tile * 128;
  const size_t fixed = 1024 + 16 + 8 * (2 * 4 + 2 * 12 + 1 + 2 * 3);  // alignment slack, slot and flag, barriers
  p.ctma = true;
  p.sbreg = false;
  // tensor-memory A stages: three of four groups after a 64-column accumulator, or four of two
  // groups after a 256-column one
  p.stages = p.gps == 4 ? 3 : 4;
  p.wring = stage > 48 * 1024 ? 2 : 3;  // (256-token tiles: two chunks, two token slots)
  // small tiles: two MMA issuers (their accumulators fit beside three A stages) and four producer
  // warp groups
  p.mw = p.gps == 4 ? 2 : 1;
  p.pg = p.gps == 4 ? 4 : 2;
  p.tstages = (int)std::min<size_t>(12, (kSmemBudget - fixed - (size_t)p.wring * kCSlot) / stage);
  p.smem = fixed + (size_t)p.tstages * stage + (size_t)p.wring * kCSlot;
  return p;
}

constexpr bool g_tc_ctma = true;  // (the tensor-copy kernel where it applies)

// The grouped two-CTAs-per-SM kernel with the weights by tensor copies: three A stages (two for
// 64-token tiles) and two weight chunks in half the shared memory each.
TcPlan tc_plan_ntile_pair_ctma(int n_tile) {
  TcPlan p = tc_plan_ntile_pair(n_tile);
  const size_t stage = 2 * (size_t)n_tile * 128;
  const size_t fixed = 1024 + 16 + 8 * (2 * 3 + 2 * 3 + 1 + 2 * 2);
  p.ctma = true;
  p.wring = 2;
  p.stages = (int)std::min<size_t>(3, (kSmemHalf - fixed - 2 * (size_t)kCSlot) / stage);
  p.tstages = p.stages;
  p.smem = fixed + (size_t)p.stages * stage + 2 * (size_t)kCSlot;
  return p;
}

TcPlan tc_plan(int out, int in, int T) {
  (void)out;
  const int n_tile = std::min(kMaxN, (T + 15) / 16 * 16);
  // (measured at 17408 x 5120: tensor copies T = 8 28.7 -> 25.8 us, T = 128 37.0 -> 35.3, T = 256
  // 44.8 -> 40.7; at T = 96 the ring copies are faster, 32.7 against 34.1)
  const bool ctma = g_tc_ctma && in % 512 == 0 && (n_tile <= 64 || n_tile >= 128);
  TcPlan p = ctma ? tc_plan_ctma(n_tile) : tc_plan_ntile(n_tile);
  p.n_tiles = (T + p.n_tile - 1) / p.n_tile;
  return p;
}

// cuTensorMapEncodeTiled from the driver (no link against it: the runtime hands out its address).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// The three tensor maps of a weight (stack) for the tensor-copy kernel: codes [n_mat][out][in / 8]
// u32 in boxes of 32 x 128 x 1 with the 128-byte swizzle; scales and biases [n_mat][out][in / 64] u16
// in boxes of 8 x 128 x 1.  Rows and columns past the ends read as zero.
bool encode_weight_maps(const qg_int4_weight& w, CUtensorMap* codes, CUtensorMap* scales, CUtensorMap* biases) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || w.in % 512 != 0) return false;
  const cuuint64_t nm = (cuuint64_t)w.n_mat, out = (cuuint64_t)w.out;
  const cuuint32_t es[3] = {1, 1, 1};
  const cuuint64_t dc[3] = {(cuuint64_t)w.in / 8, out, nm};
  const cuuint64_t sc[2] = {(cuuint64_t)w.in / 2, out * (cuuint64_t)(w.in / 2)};
  const cuuint32_t bc[3] = {32, 128, 1};
  if (enc(codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(w.packed), dc, sc, bc, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const cuuint64_t ds[3] = {(cuuint64_t)w.in / 64, out, nm};
  const cuuint64_t ss[2] = {(cuuint64_t)w.in / 32, out * (cuuint64_t)(w.in / 32)};
  const cuuint32_t bs[3] = {8, 128, 1};
  for (int i = 0; i < 2; ++i) {
    if (enc(i ? biases : scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(i ? w.biases : w.scales), ds,
            ss, bs, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

int tc_launch(const TcArgs& a, const TcPlan& p, dim3 grid, cudaStream_t stream) {
  auto go = [&](auto k) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) != cudaSuccess)
      return (int)QG_ELAUNCH;
    // two CTAs per SM: a shared-memory carve-out that just fits both (the rest stays L1, which the
    // scale/bias loads use); the one-CTA kernel keeps the driver's choice
    const int carve = (int)std::min<size_t>(100, (2 * p.smem + 2048) * 100 / (228 * 1024) + 1);
    if (p.tmem == 256 && cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, carve) != cudaSuccess)
      return (int)QG_ELAUNCH;
    return launch(k, grid, dim3((unsigned)((p.ctma ? 128 * p.pg + 96 : kThreads) + (p.mw - 1) * 32)), p.smem, stream, a);
  };
  if (p.ctma) {
    if (p.tmem == 256) return go(qgemm_tc_kernel<2, 256, false, 2, true>);
    if (p.gps == 2) return p.wring == 3 ? go(qgemm_tc_kernel<3, 512, false, 2, true>) : go(qgemm_tc_kernel<2, 512, false, 2, true>);
    if (p.wring == 3 && p.mw == 2)
      return p.pg == 4 ? go(qgemm_tc_kernel<3, 512, false, 4, true, 2, 4>) : go(qgemm_tc_kernel<3, 512, false, 4, true, 2>);
    if (p.wring == 3 && p.pg == 4) return go(qgemm_tc_kernel<3, 512, false, 4, true, 1, 4>);
    return p.wring == 3 ? go(qgemm_tc_kernel<3, 512, false, 4, true>) : go(qgemm_tc_kernel<2, 512, false, 4, true>);
  }
  if (p.tmem == 256) {
    switch (p.wring) {
      case 4:
        return go(qgemm_tc_kernel<4, 256, false, 2>);
      default:
        return go(qgemm_tc_kernel<2, 256, false, 2>);
    }
  }
  if (p.sbreg) {
    switch (p.wring) {
      case 16:
        return go(qgemm_tc_kernel<16, 512, true, 2>);
      case 8:
        return go(qgemm_tc_kernel<8, 512, true, 2>);
      case 4:
        return go(qgemm_tc_kernel<4, 512, true, 2>);
      default:
        return go(qgemm_tc_kernel<2, 512, true, 2>);
    }
  }
  if (p.gps == 4) {
    switch (p.wring) {
      case 16:
        return go(qgemm_tc_kernel<16, 512, false, 4>);
      case 8:
        return go(qgemm_tc_kernel<8, 512, false, 4>);
      case 4:
        return go(qgemm_tc_kernel<4, 512, false, 4>);
      default:
        return go(qgemm_tc_kernel<2, 512, false, 4>);
    }
  }
  switch (p.wring) {
    case 16:
      return go(qgemm_tc_kernel<16, 512, false, 2>);
    case 8:
      return go(qgemm_tc_kernel<8, 512, false, 2>);
    case 4:
      return go(qgemm_tc_kernel<4, 512, false, 2>);
    default:
      return go(qgemm_tc_kernel<2, 512, false, 2>);
  }
}

// instruction descriptor (kind::f16): D fp32 (bits 4-5 = 1), A and B fp16 (bits 7-12 = 0), both
// K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28
uint32_t tc_idesc(int n_tile) { return (1u << 4) | ((uint32_t)(n_tile >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24); }

}  // namespace

size_t qgemm_tc_workspace_bytes(const qg_int4_weight* w, int T) {
  if (T < 1) return 0;
  const TcPlan p = tc_plan(w->out, w->in, T);
  const size_t rows = (size_t)p.n_tiles * p.n_tile;
  return rows * (size_t)w->in * 2 + rows * sizeof(float) + 256;
}

int qgemm_tc_launch_multi(const qg_int4_weight* w, int n, const uint16_t* X, int T, float* const* Y, void* ws,
                          size_t ws_bytes, cudaStream_t stream) {
  if (n < 1 || n > kTcMaxMats) return QG_EINVAL;
  const TcPlan p = tc_plan(w[0].out, w[0].in, T);
  const size_t rows = (size_t)p.n_tiles * p.n_tile;
  const size_t xt_bytes = rows * (size_t)w[0].in * 2;
  if (ws_bytes < qgemm_tc_workspace_bytes(&w[0], T)) return QG_EWORKSPACE;
  uint8_t* xt = static_cast<uint8_t*>(ws);
  float* xs = reinterpret_cast<float*>(xt + xt_bytes);
  int rc = launch(qgemm_prep_kernel, dim3((unsigned)rows), dim3(kPrepThreads), 0, stream, X, T, w[0].in, p.n_tile,
                  static_cast<const int*>(nullptr), 1, xt, xs);
  if (rc != QG_OK) return rc;
  TcArgs a{};
  int tiles = 0;
  for (int i = 0; i < n; ++i) {
    a.mat[i] = TcMat{w[i].packed, w[i].scales, w[i].biases, Y[i], w[i].out, tiles, 0, 0};
    tiles += (w[i].out + kBM - 1) / kBM;
    if (p.ctma && !encode_weight_maps(w[i], &a.tm_codes[i], &a.tm_scales[i], &a.tm_biases[i])) return QG_ELAUNCH;
  }
  a.nmat = n;
  a.xt = xt;
  a.xs = xs;
  a.in = w[0].in;
  a.T = T;
  a.n_tile = p.n_tile;
  a.stages = p.stages;
  a.tstages = p.tstages;
  a.idesc = tc_idesc(p.n_tile);
  return tc_launch(a, p, dim3((unsigned)tiles, (unsigned)p.n_tiles), stream);
}

int qgemm_tc_launch(const qg_int4_weight* w, const uint16_t* X, int T, float* Y, void* ws, size_t ws_bytes,
                    cudaStream_t stream) {
  return qgemm_tc_launch_multi(w, 1, X, T, &Y, ws, ws_bytes, stream);
}

constexpr bool g_tc_pair = true;  // grouped mode: two CTAs per SM for token tiles of at most 64 rows

int qgemm_prep_pairs_launch(const uint16_t* X, int T, int in, const int* rowpos, int npairs, int k, int n_tile,
                            uint8_t* xt, float* xs, cudaStream_t stream) {
  if (k < 1 || k > kPrepMaxFan || npairs != T * k) return QG_EINVAL;
  return launch(qgemm_prep_kernel, dim3((unsigned)T), dim3(kPrepThreads), 0, stream, X, T, in, n_tile, rowpos, k,
                xt, xs);
}

int qgemm_prep_swiglu_launch(const float* G, const float* U, int in, const int* rowpos, int npairs, int n_tile,
                             uint8_t* xt, float* xs, cudaStream_t stream) {
  return launch(qgemm_prep_swiglu_kernel, dim3((unsigned)npairs), dim3(kPrepThreads), 0, stream, G, U, in, n_tile,
                rowpos, xt, xs);
}

int qgemm_tc_grouped_launch(const qg_int4_weight* w, int n, const uint8_t* xt, const float* xs, int n_tiles,
                            int n_tile, const int* tile_expert, float* const* Y, cudaStream_t stream) {
  if (n < 1 || n > kTcMaxMats || n_tile < 16 || n_tile > kMaxN || n_tile % 16 != 0 || n_tiles < 1) return QG_EINVAL;
  const bool pair = n_tile <= 64 && g_tc_pair;
  const TcPlan p = pair ? (w[0].in % 512 == 0 ? tc_plan_ntile_pair_ctma(n_tile) : tc_plan_ntile_pair(n_tile))
                        : tc_plan_ntile(n_tile);
  TcArgs a{};
  int tiles = 0;
  for (int i = 0; i < n; ++i) {
    a.mat[i] = TcMat{w[i].packed, w[i].scales, w[i].biases, Y[i], w[i].out, tiles,
                     (long long)w[i].out * (w[i].in / 8), (long long)w[i].out * (w[i].in / 64)};
    tiles += (w[i].out + kBM - 1) / kBM;
    if (p.ctma && !encode_weight_maps(w[i], &a.tm_codes[i], &a.tm_scales[i], &a.tm_biases[i])) return QG_ELAUNCH;
  }
  a.nmat = n;
  a.tile_expert = tile_expert;
  a.xt = xt;
  a.xs = xs;
  a.in = w[0].in;
  a.T = n_tiles * n_tile;
  a.n_tile = n_tile;
  a.stages = p.stages;
  a.tstages = p.tstages;
  a.idesc = tc_idesc(n_tile);
  return tc_launch(a, p, dim3((unsigned)tiles, (unsigned)n_tiles), stream);
}

}  // namespace qg
