// Tensor-core product kernel shared by the three NS products.
//
//   out[i, j] = alpha * sum_k Aop[i, k] * Bop[k, j] + beta * addend[i, j]
//
// bf16 operands (or fp32 operands read as tf32, F32) staged by TMA into
// 128-byte-swizzled shared memory, fp32 accumulation in TMEM by tcgen05.mma
// (M = 128, or 256 across a CTA pair with SM2; N = 256; K = 16 per
// instruction, 8 for tf32), fp32 epilogue, one rounding of the output (to
// bf16, or to tf32 in fp32 storage where it feeds another product).
//
// With the optional fp32 diagonal (GroupArgs::diag_out / diag_in) the
// polynomial product stores B = D + O as an fp32 vector D = diag(B) and a bf16
// matrix O with zero diagonal, and the update computes (a + D) X + O X; near
// convergence B is close to a multiple of the identity, so this keeps the
// dominant part of B out of bf16 rounding.
//
// Template parameters:
//   A_MN  the A operand is stored MN-major ([k][i], i contiguous) instead of
//         K-major ([i][k], k contiguous);
//   B_MN  the same for B ([k][j] instead of [j][k]);
//   SYM   the output is symmetric: only lower-triangle tiles are scheduled and
//         every value with j <= i is written to (i, j) and to (j, i), so the
//         stored matrix is bit-symmetric (one triangle computed and mirrored,
//         prime-rl PR #3873, Summary item 1; Megatron-LM PR #6381, Summary);
//         with GemmParams::half_out only inside the diagonal 256 x 256
//         blocks, the rest of the upper triangle being read transposed by the
//         consumers (GroupArgs::half_a / half_b);
//   CL    CTAs per cluster, 1 or 2.  With 2, the two CTAs of a cluster compute
//         row tiles 2p and 2p + 1 of the same column tile, whose B-operand
//         panel they share: each loads one half of it with a multicast TMA
//         copy into both CTAs' shared memory, and each MMA commit releases the
//         stage in both CTAs.  Half the B-operand bytes per CTA come from L2;
//   WOUT  (update products only) the last update of a Muon step: the
//         epilogue updates the fp32 master weights in place of storing the
//         iterate (GroupArgs::w_out), prefetching their rows one chunk ahead,
//         with the launch's factors (1, GemmParams::w_decay / w_lrs) or each
//         group's own (2, GemmParams::w_decay_g / w_lrs_g);
//   SM2   (CL == 2 only) the pair runs 2-SM MMAs instead: one thread of CTA 0
//         issues M = 256 tcgen05.mma.cta_group::2 over A tiles held by both
//         CTAs (128 rows each) and a B panel split in halves between them,
//         so each CTA stores and loads only its own half of the panel
//         (32 KB stages instead of 48 KB, 6 of them); each CTA's TMEM holds
//         its own 128 rows of the accumulator.
//
// Uses (m <= n internally; Y = the tall input kept in its own orientation):
//   Gram X X^T       <false, false, true>   both operands = rows of X
//   Gram Y^T Y       <true,  true,  true>   both operands = columns of Y
//   b A + c A A      <false, false, true>   A A = A A^T for a bit-symmetric A
//   a X + B X        <false, true,  false>  X read MN-major
//   a Y + Y B        <false, false, false>  B = B^T bitwise
//
// Roles (64 + 32 * kEpiWarps threads, one CTA per SM, persistent):
//   warp 0 lane 0   TMA producer: fills a kStages-deep ring of operand stages
//   warp 1 lane 0   MMA issuer (with SM2 in CTA 0 of the pair only):
//                   tcgen05.mma per K slice of a stage into one of two
//                   256-column TMEM accumulators, commits release the stage
//   warps 2..       epilogue: each warp reads its 32-lane TMEM quarter for its
//                   share of the columns (two warps per quarter by default),
//                   prefetches the addend one 32-column chunk ahead, runs the
//                   fp32 epilogue, stores bf16, then frees the accumulator
// The double-buffered accumulator lets the epilogue of tile t overlap the
// main loop of tile t + 1.
//
// In a whole NS call the kernel waits, per unit, for the previous product of
// the same matrix through per-matrix completion counters (GroupArgs::dep_*),
// and publishes its own units' completion, so consecutive kernels overlap.
//
// Every wait on an mbarrier or a counter is bounded (clock64 budget).  When
// one runs out the kernel records MUON_NS_DEVERR_WAIT_TIMEOUT in the error
// word, every role leaves its loop, the producer waits (bounded) for its
// copies in flight, the MMA issuer waits (bounded) for its MMAs, and TMEM is
// freed before return.
#pragma once

#include <cstdint>
#include <type_traits>

#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "tile_sched.h"

namespace mns {

constexpr int kBlockK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int kABytes = kTileM * 128;          // A tile: 128 rows of 128 bytes (16 KB)
constexpr int kBBytes = kTileN * 128;          // B panel: 256 rows of 128 bytes (32 KB)
constexpr int kMaxStages = 8;
constexpr int kTmemCols = 2 * kTileN;          // two fp32 accumulators
// Diagonal units of symmetric products on CTA pairs load each row tile once
// (it is both the A tile and a half of the B panel); MNS_DIAG_ONCE=0 loads
// both operands as on every other unit.
#ifndef MNS_DIAG_ONCE
#define MNS_DIAG_ONCE 1
#endif


// Output staging: each epilogue warp stages 32 x 32 output chunks (bf16: 2 KB,
// rows of 64 bytes, 64-byte TMA swizzle; fp32: 4 KB, 128-byte rows and swizzle)
// that bulk tensor stores write out.
constexpr int kMnChunk = 64;                   // MN elements per 128-byte row
constexpr int kMnChunkBytes = kMnChunk * kBlockK * 2;  // 8 KB

// Per element type: bf16 operands (kind::f16 MMA, K = 16 per instruction) or
// fp32 operands read as tf32 (kind::tf32, K = 8).  A stage always holds one
// 128-byte swizzle row of K per operand row: 64 bf16 or 32 fp32, so a stage is
// 48 KB either way; the fp32 variant keeps 3 stages to leave shared memory for
// its 4 KB output chunks.
template <bool F32>
struct ElemCfg {
  static constexpr int kBytes = F32 ? 4 : 2;
  static constexpr int kBlockK = 128 / kBytes;                    // K per stage
  static constexpr int kMmaK = F32 ? 8 : 16;                      // K per tcgen05.mma
  static constexpr int kMnChunk = 128 / kBytes;                   // MN elements per 128-byte row
  static constexpr int kMnChunkBytes = kMnChunk * kBlockK * kBytes;  // 8 KB or 4 KB
  static constexpr int kMnStep = kMmaK * 128;  // bytes between MMA K steps, MN-major
  static constexpr int kChunkBytes = 32 * 32 * kBytes;            // 32 x 32 output chunk
  static constexpr int kAddVec = 32 * kBytes / 16;                 // 16-byte vectors per chunk row
};

// Epilogue warps: 4 or 8, i.e. one or two per TMEM lane quarter.  The
// symmetric products (mirrored stores) always take 8; the update takes 8 when
// its contraction is short (K <= 1024, little main-loop time per tile to hide
// the epilogue behind) and 4 otherwise (measured on GB300).
template <int EPI_WARPS>
struct Epi {
  static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "4 or 8 epilogue warps");
  static constexpr int kWarps = EPI_WARPS;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kCtaThreads = 64 + kThreads;  // + producer warp + MMA warp
  static constexpr int kChunksPerWarp = (kTileN / 32) / (kWarps / 4);
};

// Shared memory of one CTA: the operand ring and the epilogue's staging.
//   Staging buffers per epilogue warp: symmetric products need two at once
//   (the chunk and its transpose), and so do fp32 updates that also store
//   their transpose (GemmParams::tmOutT); the bf16 update double-buffers with
//   4 warps and single-buffers with 8.
//   Ring: a stage holds the CTA's A tile and the B rows it keeps, the whole
//   256-row panel (48 KB) or, with 2-SM MMAs, its 128-row half (32 KB); 4
//   stages of 48 KB for bf16 and 3 for fp32 (larger staging), and with 2-SM
//   MMAs as many 32 KB stages as fit, at most 6.
template <bool SYM, int EPI_WARPS, bool F32 = false, bool SM2 = false>
struct Smem {
  static constexpr int kBufs = (SYM || F32) ? 2 : (EPI_WARPS == 4 ? 2 : 1);
  static constexpr int kStagingBytes = EPI_WARPS * kBufs * ElemCfg<F32>::kChunkBytes;
  static constexpr int kStageBytes = kABytes + (SM2 ? kBBytes / 2 : kBBytes);
  // 227 KB per CTA, less an upper bound of the kernel's static shared memory
  // (barriers, and the update's per-column coefficients) and 1 KB of alignment.
  static constexpr int kRingMax = 232448 - (SYM ? 1024 : 4608) - kStagingBytes - 1024;
  static constexpr int kFit = kRingMax / kStageBytes;
  static constexpr int kStages = SM2 ? (kFit < 6 ? kFit : 6) : (F32 ? 3 : 4);
  static constexpr int kSmemBytes = kStages * kStageBytes + kStagingBytes + 1024;
  static_assert(kStages >= 2 && kStages <= kMaxStages, "ring depth");
  static_assert(kSmemBytes <= kRingMax + kStagingBytes + 1024, "shared memory");
};

// Byte offset of element (row, col) of a 32 x 32 bf16 staging chunk: rows of
// 64 bytes, 16-byte granule index XOR ((row >> 1) & 3) (the 64-byte TMA
// swizzle), so that 32 lanes writing 32 different rows hit distinct banks.
__device__ __forceinline__ uint32_t stage_off(int row, int col) {
  const int g = (col >> 3) ^ ((row >> 1) & 3);
  return static_cast<uint32_t>(row * 64 + g * 16 + (col & 7) * 2);
}

// The same for a 32 x 32 fp32 chunk: rows of 128 bytes, granule XOR (row & 7)
// (the 128-byte TMA swizzle).
__device__ __forceinline__ uint32_t stage_off32(int row, int col) {
  const int g = (col >> 2) ^ (row & 7);
  return static_cast<uint32_t>(row * 128 + g * 16 + (col & 3) * 4);
}

// Byte offset of 16-byte granule `g` (0..7) of row `row` of a 32 x 64 bf16
// staging box: rows of 128 bytes, granule XOR (row & 7) (the 128-byte TMA
// swizzle, on a 1024-byte aligned buffer).
__device__ __forceinline__ uint32_t stage_off_wide(int row, int g) {
  return static_cast<uint32_t>(row * 128 + ((g ^ (row & 7)) << 4));
}

// Round an fp32 value to the nearest tf32 (10-bit mantissa, ties to even),
// kept in fp32 storage: the tensor core reads tf32 by dropping the low 13
// bits, so values stored this way reach it exactly.  Inputs here are finite.
__device__ __forceinline__ uint32_t round_tf32_bits(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0xFFFu + ((u >> 13) & 1u);
  return u & 0xFFFFE000u;
}

// A launch covers up to kMaxGroups stacks ("groups") of same-shape matrices,
// each with its own tensor maps and sizes; the tile spaces of the groups are
// concatenated, so one persistent launch keeps every SM busy across stacks.
constexpr int kMaxGroups = 8;

struct GroupArgs {
  long long tile_begin;  // first tile of this group in the launch's tile space
  TileSpace space;
  int M, N, K;           // output rows, output columns, contraction length
  int num_kb;            // ceil(K / kBlockK)
  const void* addend;    // [batch][M][N] (bf16, or fp32 for F32) with row stride ld, or nullptr
  long long ld;
  long long bstride;
  // Diagonal kept in fp32 (both optional):
  //   diag_out  SYM only: the fp32 value of each diagonal element is written to
  //             diag_out[b * M + i] and 0 is stored on the bf16 diagonal;
  //   diag_in   the addend coefficient becomes beta + diag_in[...], indexed by
  //             the output row (diag_per_col == 0) or column (== 1).
  float* diag_out;
  const float* diag_in;
  // Unscaled operands (optional): with norms != nullptr the operands are the
  // raw G of each matrix and s = 1 / (norms[b] + eps) is applied in the
  // epilogue, so the first step needs no scaled copy of G:
  //   SYM (Gram)      out = alpha s^2 acc
  //   FULL (update)   out = alpha s acc + (beta + diag) s addend
  const float* norms;
  // Operands read from a half-stored symmetric matrix (GemmParams::half_out
  // of the product that wrote it): k-blocks past the operand rows' diagonal
  // 256-block are read transposed, MN-major, through tmA2 / tmB2.
  int half_a, half_b;
  // Per-matrix completion counters of a whole NS call (both optional):
  //   dep_sig   every finished unit adds kDepUnit to dep_sig[b] once its
  //             outputs are written (each epilogue warp of the unit's CTAs
  //             adds its share);
  //   dep_wait  the unit's operands and addend come from the previous product
  //             of the same matrix: it waits until dep_wait[b] >= dep_target
  //             (GemmParams::dep_flags), not for the whole previous grid.
  int* dep_sig;
  const int* dep_wait;
  int dep_target;
  // Last update of a Muon step (FULL bf16 products only, optional): instead
  // of storing the iterate, each output value o, rounded to bf16 as it would
  // be stored, updates the fp32 master in place,
  //   w_out[b][i][j] = w_decay * w_out[b][i][j] - w_lrs * o,
  // with w_out laid out like the output ([batch][M][N], row stride ld), and
  // w_decay = 1 - lr wd, w_lrs = lr scale (GemmParams::w_decay / w_lrs, or
  // w_decay_g / w_lrs_g for WOUT = 2).
  float* w_out;
};

// The group arguments are read with a run-time group index: at 144 bytes each
// entry starts on a 16-byte boundary.  Two more floats (152 bytes) measured
// the fused Muon step 2.5 % slower on GB300, so per-group additions go to the
// end of GemmParams instead.
static_assert(sizeof(GroupArgs) % 16 == 0, "GroupArgs entries 16-byte aligned");

// Counter increment per finished unit of the tile space, whatever the
// launch's CTAs per unit and epilogue warps.
constexpr int kDepUnit = 16;

struct GemmParams {
  CUtensorMap tmA[kMaxGroups];    // A operand (rows of the output)
  CUtensorMap tmB[kMaxGroups];    // B operand (columns of the output)
  // Output in 32-row boxes: 32 x 32 (bf16: 64-byte swizzle; fp32: 128-byte),
  // or 32 x 64 with the 128-byte swizzle for the 4-warp bf16 update.
  CUtensorMap tmOut[kMaxGroups];
  // FULL only, optional: the transposed output [batch][N][M] (same boxes),
  // written when out_t != 0.  The fp32 path keeps its iterate in both
  // orientations so that every tensor-core operand is K-major.
  CUtensorMap tmOutT[kMaxGroups];
  CUtensorMap tmA2[kMaxGroups];   // MN-major maps of half-stored operands
  CUtensorMap tmB2[kMaxGroups];
  GroupArgs grp[kMaxGroups];
  int num_groups;
  long long total_tiles;
  float alpha, beta, eps;
  int diag_per_col;
  int round_tf32;     // F32 only: store outputs rounded to tf32 (they feed an MMA)
  int out_t;          // FULL only: also write the transposed output through tmOutT
  // SYM only: half storage.  A value is mirrored only inside its diagonal
  // 256 x 256 block; elsewhere only the lower triangle is written, and
  // consumers read the upper part from it transposed (GroupArgs::half_a/b).
  int half_out;
  // Waits are per matrix (GroupArgs::dep_wait): the kernel starts on matrices
  // whose inputs are ready while the previous grid still runs, and waits for
  // the previous grid only before it exits, so that its completion still
  // implies that of every earlier kernel in the stream.
  int dep_flags;
  // GroupArgs::w_out with one pair of factors for every group (WOUT = 1):
  // 1 - lr wd and lr scale.
  float w_decay, w_lrs;
  int* err;           // device error word, or nullptr
  long long budget;   // clock64 cycles per wait
  // The same factors for each group (WOUT = 2).
  float w_decay_g[kMaxGroups], w_lrs_g[kMaxGroups];
};

// Group owning global tile t (groups are few; a linear scan).
__device__ __forceinline__ int find_group(const GemmParams& P, long long t) {
  int g = 0;
  while (g + 1 < P.num_groups && t >= P.grp[g + 1].tile_begin) ++g;
  return g;
}

namespace detail {

// Shared-memory addresses of the kernel's mbarriers, laid out consecutively:
// full[kMaxStages], empty[kMaxStages], tfull[2], tempty[2], mma_done.
struct Sync {
  uint32_t base;
  __device__ __forceinline__ uint32_t full(int s) const { return base + 8u * s; }
  __device__ __forceinline__ uint32_t empty(int s) const { return base + 8u * (kMaxStages + s); }
  __device__ __forceinline__ uint32_t tfull(int i) const { return base + 8u * (2 * kMaxStages + i); }
  __device__ __forceinline__ uint32_t tempty(int i) const { return base + 8u * (2 * kMaxStages + 2 + i); }
  __device__ __forceinline__ uint32_t mma_done() const { return base + 8u * (2 * kMaxStages + 4); }
};

__device__ __forceinline__ void raise_error(volatile int* abort_flag, int* err) {
  *abort_flag = 1;
  if (err) atomicOr(err, 1);
}

// Poll of one mbarrier phase; cluster-scope acquire where another CTA of the
// cluster arrives on the barrier.
template <bool CLUSTER>
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
  return CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
}

// Bounded wait.  Returns false (and raises the abort flag on expiry) if the
// phase did not complete within the budget or another role aborted.
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, int* err,
                                             long long budget) {
  if (try_wait<CLUSTER>(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (try_wait<CLUSTER>(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      raise_error(abort_flag, err);
      return false;
    }
  }
}

// Bounded wait until a per-matrix completion counter reaches `target`
// (acquire at GPU scope).  Gives up early once any kernel has set the error
// word: the counter may then never get there.
__device__ __forceinline__ bool wait_count(const int* c, int target, volatile int* abort_flag,
                                           int* err, long long budget) {
  if (ptx::ld_acquire_gpu(c) >= target) return true;
  const long long t0 = clock64();
  while (true) {
    __nanosleep(64);
    if (ptx::ld_acquire_gpu(c) >= target) return true;
    if (*abort_flag) return false;
    if (err != nullptr && *reinterpret_cast<volatile int*>(err) != 0) {
      *abort_flag = 1;
      return false;
    }
    if (clock64() - t0 > budget) {
      raise_error(abort_flag, err);
      return false;
    }
  }
}

// Bounded wait until the producer has seen the inputs of `units` units
// complete (CTA-scope acquire of its shared-memory count).
__device__ __forceinline__ bool wait_seen(uint32_t addr, int units, volatile int* abort_flag,
                                          int* err, long long budget) {
  if (ptx::ld_acquire_cta_shared(addr) >= units) return true;
  const long long t0 = clock64();
  while (true) {
    if (ptx::ld_acquire_cta_shared(addr) >= units) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      raise_error(abort_flag, err);
      return false;
    }
  }
}

// Bounded wait used on the way out: ignores the abort flag.
template <bool CLUSTER = false>
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long budget) {
  const long long t0 = clock64();
  while (!try_wait<CLUSTER>(bar, parity)) {
    if (clock64() - t0 > budget) return;
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values rounded to bf16 (nearest, ties to even) in one packed
// conversion; `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace detail

template <bool A_MN, bool B_MN, bool SYM, int EPI_WARPS, bool F32, int CL = 1, bool SM2 = false, int WOUT = 0>
__global__ void __launch_bounds__(Epi<EPI_WARPS>::kCtaThreads, 1)
    ns_tc_gemm(const __grid_constant__ GemmParams P) {
  static_assert(CL == 1 || CL == 2, "clusters of one or two CTAs");
  static_assert(!SM2 || CL == 2, "2-SM MMAs run on CTA pairs");
  static_assert(!WOUT || (!SYM && !F32), "master-weight output: bf16 update products only");
  using EC = ElemCfg<F32>;
  using R = Smem<SYM, EPI_WARPS, F32, SM2>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 5];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  // Units whose inputs the producer has seen complete (per-matrix counters),
  // handed to the epilogue warps by a CTA-scope release.
  __shared__ int dep_seen_sh;
  constexpr int kEpiWarps = Epi<EPI_WARPS>::kWarps;
  constexpr int kEpiThreads = Epi<EPI_WARPS>::kThreads;
  constexpr int kChunksPerWarp = Epi<EPI_WARPS>::kChunksPerWarp;
  __shared__ __align__(16) float colc_sh[SYM ? 1 : kEpiWarps][kChunksPerWarp * 32];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &abort_sh;
  // Units of the tile space are walked with a static stride: one unit per
  // CTA, or per cluster of two (CTA rank r then takes row tile 2p + r).
  const uint32_t crank = CL == 2 ? ptx::cluster_ctarank() : 0u;
  const long long unit0 = CL == 2 ? static_cast<long long>(ptx::cluster_id_x()) : blockIdx.x;
  const long long ustride = CL == 2 ? static_cast<long long>(ptx::cluster_count_x()) : gridDim.x;
  auto row_tile = [&](int u) { return CL == 2 ? 2 * u + static_cast<int>(crank) : u; };
  // 2-SM MMAs: CTA 0 of the pair issues them and owns the operand-full and
  // accumulator-empty barriers; both CTAs load their halves and drain their
  // own TMEM rows.
  const bool leader = crank == 0;

  const uint32_t smem_base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  detail::Sync sy;
  sy.base = ptx::smem_u32(&bars[0]);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < R::kStages; ++s) {
      ptx::mbar_init(sy.full(s), 1);
      // One MMA commit per CTA of a multicast pair; the pair's single commit
      // with 2-SM MMAs.
      ptx::mbar_init(sy.empty(s), (CL == 2 && !SM2) ? 2 : 1);
    }
    ptx::mbar_init(sy.tfull(0), 1);
    ptx::mbar_init(sy.tfull(1), 1);
    // Every epilogue thread arrives; with 2-SM MMAs one lane per epilogue
    // warp of both CTAs (on CTA 0's barrier).
    ptx::mbar_init(sy.tempty(0), SM2 ? 2 * kEpiWarps : kEpiThreads);
    ptx::mbar_init(sy.tempty(1), SM2 ? 2 * kEpiWarps : kEpiThreads);
    ptx::mbar_init(sy.mma_done(), 1);
    *abort_flag = 0;
    dep_seen_sh = 0;
    ptx::fence_barrier_init();
    for (int g = 0; g < P.num_groups; ++g) {
      ptx::prefetch_tensormap(&P.tmA[g]);
      ptx::prefetch_tensormap(&P.tmB[g]);
      ptx::prefetch_tensormap(&P.tmOut[g]);
    }
  }
  // The peer CTA's copies, commits and arrivals target this CTA's barriers:
  // both must be initialised before either CTA issues one.
  if (SM2) {
    __syncthreads();
    ptx::cluster_sync();
  }
  if (warp == 0) {
    if (SM2) {
      ptx::tmem_alloc_pair(ptx::smem_u32(&tmem_base_sh), kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (CL == 2 && !SM2) ptx::cluster_sync();
  const uint32_t tmem_base = tmem_base_sh;
  // Every CTA is resident from the start (one per SM), so the next kernel may
  // be scheduled now: its CTAs take SMs as ours exit and finish their prologue
  // meanwhile.  Nothing produced by the previous kernel is touched before this
  // grid's dependency has completed.
  ptx::griddep_launch_dependents();
  if (!P.dep_flags) ptx::griddep_wait();

  const long long total = P.total_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0;   // stages with a load issued at least once
      uint32_t issued_phase = 0;  // parity of the last load issued per stage
      int units_seen = 0;         // units whose inputs are known complete
      for (long long t = unit0; t < total; t += ustride) {
        const int gr = find_group(P, t);
        const GroupArgs& G = P.grp[gr];
        const CUtensorMap* tmA = &P.tmA[gr];
        const CUtensorMap* tmB = &P.tmB[gr];
        const int num_kb = G.num_kb;
        int b, I, J;
        tile_decode(G.space, t - G.tile_begin, &b, &I, &J);
        I = row_tile(I);
        const int row0 = I * kTileM;
        const int col0 = J * kTileN;
        // k-block from which an operand of a half-stored matrix is read
        // transposed (num_kb: never), as in the MMA issuer.
        const int kb_a = G.half_a ? min(256 * ((I >> 1) + 1) / EC::kBlockK, num_kb) : num_kb;
        const int kb_b = G.half_b ? min(256 * (J + 1) / EC::kBlockK, num_kb) : num_kb;
        // Diagonal unit of a symmetric product on a CTA pair: the B panel is
        // the pair's own two A tiles (rows 256 J .. 256 J + 255), so each CTA
        // loads its row tile once and both operands are read from it.
        const bool diag = MNS_DIAG_ONCE && SYM && CL == 2 && J == (I >> 1);
        // The operands of matrix b are complete once the previous product
        // has finished all of its units.  Every unit is then counted for the
        // epilogue, which reads the same inputs' addend and diagonal.
        if (G.dep_wait != nullptr) {
          if (!detail::wait_count(G.dep_wait + b, G.dep_target, abort_flag, P.err, P.budget)) break;
          ptx::fence_proxy_async_global();
        }
        ptx::st_release_cta_shared(ptx::smem_u32(&dep_seen_sh), ++units_seen);
        bool ok = true;
        // Up to three segments of fixed operand majorness, each naming its
        // tensor maps at compile time (a map chosen per k-block at run time
        // made every product about 25 % slower on GB300).
        auto ploop = [&](auto amn_t, auto bmn_t, int kb0, int kb1) {
          constexpr bool AMN = decltype(amn_t)::value;
          constexpr bool BMN = decltype(bmn_t)::value;
          // Past the switch the operand is read through the MN-major map of
          // the half-stored matrix.
          const CUtensorMap* mA = (AMN && !A_MN) ? &P.tmA2[gr] : tmA;
          const CUtensorMap* mB = (BMN && !B_MN) ? &P.tmB2[gr] : tmB;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!detail::wait_bounded<SM2>(sy.empty(stage), phase ^ 1u, abort_flag, P.err,
                                           P.budget)) {
              ok = false;
              return;
            }
            const uint32_t sa = smem_base + stage * R::kStageBytes;
            const uint32_t sb = sa + kABytes;
            const int k0 = kb * EC::kBlockK;
            constexpr int kNch = kTileN / EC::kMnChunk;  // MN-major chunks of the B panel
            if (SM2) {
              // This CTA's A tile and its half of the B panel, into its own
              // shared memory; all bytes of the pair are counted on CTA 0's
              // barrier, which expects both CTAs' stages.  On a diagonal unit
              // the A tile is also this CTA's half of the panel.
              const uint32_t fb = ptx::mapa(sy.full(stage), 0);
              if (leader) ptx::mbar_arrive_expect_tx(sy.full(stage), diag ? 2 * kABytes : 2 * R::kStageBytes);
              if (AMN) {
#pragma unroll
                for (int c = 0; c < kTileM / EC::kMnChunk; ++c)
                  ptx::tma_load_3d_pair(sa + c * EC::kMnChunkBytes, mA, fb, row0 + c * EC::kMnChunk, k0, b);
              } else {
                ptx::tma_load_3d_pair(sa, mA, fb, k0, row0, b);
              }
              if (diag) {
              } else if (BMN) {
#pragma unroll
                for (int c = 0; c < kNch / 2; ++c)
                  ptx::tma_load_3d_pair(sb + c * EC::kMnChunkBytes, mB, fb,
                                        col0 + (static_cast<int>(crank) * (kNch / 2) + c) * EC::kMnChunk, k0, b);
              } else {
                ptx::tma_load_3d_pair(sb, mB, fb, k0, col0 + static_cast<int>(crank) * (kTileN / 2), b);
              }
            } else if (CL == 2 && diag) {
              // Multicast pair, diagonal unit: each CTA's half of the shared
              // panel is its own A tile, so only the panel is loaded and the A
              // operand is read from this CTA's half of it.
              ptx::mbar_arrive_expect_tx(sy.full(stage), kBBytes);
              if (BMN) {
#pragma unroll
                for (int c = 0; c < kNch / 2; ++c) {
                  const int cg = static_cast<int>(crank) * (kNch / 2) + c;
                  ptx::tma_load_3d_mc(sb + cg * EC::kMnChunkBytes, mB, sy.full(stage),
                                      col0 + cg * EC::kMnChunk, k0, b, 0x3);
                }
              } else {
                ptx::tma_load_3d_mc(sb + crank * (kBBytes / 2), mB, sy.full(stage), k0,
                                    col0 + static_cast<int>(crank) * (kTileN / 2), b, 0x3);
              }
            } else {
              ptx::mbar_arrive_expect_tx(sy.full(stage), R::kStageBytes);
              if (AMN) {
#pragma unroll
                for (int c = 0; c < kTileM / EC::kMnChunk; ++c)
                  ptx::tma_load_3d(sa + c * EC::kMnChunkBytes, mA, sy.full(stage),
                                   row0 + c * EC::kMnChunk, k0, b);
              } else {
                ptx::tma_load_3d(sa, mA, sy.full(stage), k0, row0, b);
              }
              if (CL == 2) {
                // This CTA's half of the shared panel, into both CTAs.
                if (BMN) {
#pragma unroll
                  for (int c = 0; c < kNch / 2; ++c) {
                    const int cg = static_cast<int>(crank) * (kNch / 2) + c;
                    ptx::tma_load_3d_mc(sb + cg * EC::kMnChunkBytes, mB, sy.full(stage),
                                        col0 + cg * EC::kMnChunk, k0, b, 0x3);
                  }
                } else {
                  ptx::tma_load_3d_mc(sb + crank * (kBBytes / 2), mB, sy.full(stage), k0,
                                      col0 + static_cast<int>(crank) * (kTileN / 2), b, 0x3);
                }
              } else if (BMN) {
#pragma unroll
                for (int c = 0; c < kNch; ++c)
                  ptx::tma_load_3d(sb + c * EC::kMnChunkBytes, mB, sy.full(stage),
                                   col0 + c * EC::kMnChunk, k0, b);
              } else {
                ptx::tma_load_3d(sb, mB, sy.full(stage), k0, col0, b);
              }
            }
            issued_mask |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == R::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        };
        using kA = std::integral_constant<bool, A_MN>;
        using kB = std::integral_constant<bool, B_MN>;
        using kT = std::integral_constant<bool, true>;
        const int s1 = kb_a < kb_b ? kb_a : kb_b;
        const int s2 = kb_a < kb_b ? kb_b : kb_a;
        ploop(kA{}, kB{}, 0, s1);
        if (ok && s2 > s1) {
          if (kb_a < kb_b)
            ploop(kT{}, kB{}, s1, s2);
          else
            ploop(kA{}, kT{}, s1, s2);
        }
        if (ok && num_kb > s2) ploop(kT{}, kT{}, s2, num_kb);
        if (!ok) break;
      }
      // Wait for every copy still in flight before the CTA can exit (with
      // 2-SM MMAs CTA 0's barriers count the copies of both CTAs).
      if (!SM2 || leader) {
#pragma unroll
        for (int s = 0; s < R::kStages; ++s)
          if (issued_mask & (1u << s))
            detail::drain_wait<SM2>(sy.full(s), (issued_phase >> s) & 1u, P.budget);
      }
      if (CL == 2) {
        // The other CTA's MMA commits also arrive on this CTA's empty
        // barriers: wait until the last fill of every stage has been released
        // (a stage never filled passes at once).
        for (int s = 0; s < R::kStages; ++s) {
          detail::drain_wait<SM2>(sy.empty(stage), phase ^ 1u, P.budget);
          if (++stage == R::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && (!SM2 || leader)) {
      // ---------------------------------------------------------- MMA issuer
      // (2-SM MMAs: M = 256, the pair's two row tiles at once.)
      constexpr int kMmaM = SM2 ? 2 * kTileM : kTileM;
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t tphase = 0;
      for (long long t = unit0; t < total; t += ustride) {
        const int gr = find_group(P, t);
        const GroupArgs& G = P.grp[gr];
        const int num_kb = G.num_kb;
        // In a symmetric product, a tile on an even row tile I = 2J lies on the
        // diagonal 256-column block with its right half entirely above the
        // diagonal: only its left 128 columns are computed (N = 128).  A 2-SM
        // MMA shares N between the pair's row tiles and always takes 256.
        bool half_n = false;
        int tI = 0, tJ = 0;
        if (SYM || G.half_a || G.half_b) {
          int b;
          tile_decode(G.space, t - G.tile_begin, &b, &tI, &tJ);
          tI = row_tile(tI);
          half_n = SYM && !SM2 && (tI & 1) == 0 && tJ == (tI >> 1);
        }
        // Diagonal unit of a pair (as in the producer): one copy of each row
        // tile serves as both operands.  2-SM MMAs read the B panel halves
        // from the A tiles; multicast pairs read A from this CTA's panel half.
        const bool diag = MNS_DIAG_ONCE && SYM && CL == 2 && tJ == (tI >> 1);
        const uint32_t a_off = (diag && !SM2) ? static_cast<uint32_t>(kABytes + crank * (kBBytes / 2)) : 0u;
        const uint32_t b_off = (diag && SM2) ? 0u : static_cast<uint32_t>(kABytes);
        // k-block from which an operand of a half-stored matrix is read
        // transposed (num_kb: never).
        const int kb_a = G.half_a ? min(256 * ((tI >> 1) + 1) / EC::kBlockK, num_kb) : num_kb;
        const int kb_b = G.half_b ? min(256 * (tJ + 1) / EC::kBlockK, num_kb) : num_kb;
        if (!detail::wait_bounded<SM2>(sy.tempty(buf), tphase ^ 1u, abort_flag, P.err, P.budget))
          break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * kTileN);
        bool ok = true;
        // The main loop runs in up to three segments of fixed operand
        // majorness, so that the descriptors stay compile-time constants: the
        // tensor pipe is fed from this one thread.
        auto kloop = [&](auto amn_t, auto bmn_t, int kb0, int kb1) {
          constexpr bool AMN = decltype(amn_t)::value;
          constexpr bool BMN = decltype(bmn_t)::value;
          constexpr uint32_t id_full = F32 ? ptx::idesc_tf32_f32(kMmaM, kTileN, AMN, BMN)
                                           : ptx::idesc_bf16_f32(kMmaM, kTileN, AMN, BMN);
          constexpr uint32_t id_half = F32 ? ptx::idesc_tf32_f32(kTileM, kTileN / 2, AMN, BMN)
                                           : ptx::idesc_bf16_f32(kTileM, kTileN / 2, AMN, BMN);
          const uint32_t idesc = half_n ? id_half : id_full;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!detail::wait_bounded<SM2>(sy.full(stage), phase, abort_flag, P.err, P.budget)) {
              ok = false;
              return;
            }
            ptx::tc_fence_after();
            const uint32_t sa = smem_base + stage * R::kStageBytes + a_off;
            const uint32_t sb = smem_base + stage * R::kStageBytes + b_off;
#pragma unroll
            for (int kk = 0; kk < EC::kBlockK / EC::kMmaK; ++kk) {
              // K-major: an MMA's K slice is 32 bytes further along the swizzle
              // row; MN-major: kMmaK k-rows of 128 bytes further down.
              const uint64_t ad =
                  AMN ? ptx::sw128_desc(sa + kk * EC::kMnStep, EC::kMnChunkBytes, 1024)
                      : ptx::sw128_desc(sa + kk * 32, 16, 1024);
              const uint64_t bd =
                  BMN ? ptx::sw128_desc(sb + kk * EC::kMnStep, EC::kMnChunkBytes, 1024)
                      : ptx::sw128_desc(sb + kk * 32, 16, 1024);
              if (F32 && SM2)
                ptx::mma_tf32_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
              else if (F32)
                ptx::mma_tf32(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
              else if (SM2)
                ptx::mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
              else
                ptx::mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            if (SM2)
              ptx::mma_commit_pair(sy.empty(stage), 0x3);
            else if (CL == 2)
              ptx::mma_commit_mc(sy.empty(stage), 0x3);
            else
              ptx::mma_commit(sy.empty(stage));
            if (++stage == R::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        };
        using kA = std::integral_constant<bool, A_MN>;
        using kB = std::integral_constant<bool, B_MN>;
        using kT = std::integral_constant<bool, true>;
        const int s1 = kb_a < kb_b ? kb_a : kb_b;
        const int s2 = kb_a < kb_b ? kb_b : kb_a;
        kloop(kA{}, kB{}, 0, s1);
        if (ok && s2 > s1) {
          if (kb_a < kb_b)
            kloop(kT{}, kB{}, s1, s2);
          else
            kloop(kA{}, kT{}, s1, s2);
        }
        if (ok && num_kb > s2) kloop(kT{}, kT{}, s2, num_kb);
        if (!ok) break;
        if (SM2)
          ptx::mma_commit_pair(sy.tfull(buf), 0x3);
        else
          ptx::mma_commit(sy.tfull(buf));
        buf ^= 1;
        if (buf == 0) tphase ^= 1u;
      }
      // Every MMA issued by this thread has finished once this arrives.
      if (SM2)
        ptx::mma_commit_pair(sy.mma_done(), 0x1);
      else
        ptx::mma_commit(sy.mma_done());
      detail::drain_wait<SM2>(sy.mma_done(), 0, P.budget);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    // Warp e = warp - 2 reads TMEM lane quarter q = warp % 4 (the lanes a warp
    // may access) and owns kChunksPerWarp 32-column chunks of the tile.
    const int e = warp - 2;
    const int q = warp & 3;
    const int c_begin = (e >> 2) * kChunksPerWarp;
    const int r_in_tile = q * 32 + lane;
    float* colc = colc_sh[SYM ? 0 : e];
    constexpr int kBufs = R::kBufs;
    constexpr int kCB = EC::kChunkBytes;
    constexpr int kAV = EC::kAddVec;  // 16-byte addend vectors per lane and chunk
    // The 4-warp bf16 update stores 32 x 64 boxes (update_epi_warps).
    constexpr bool kWide = !SYM && !F32 && EPI_WARPS == 4;
    static_assert(!kWide || (kBufs * kCB == 4096 && kChunksPerWarp % 2 == 0), "wide staging box");
    const uint32_t stg = smem_base + R::kStages * R::kStageBytes + static_cast<uint32_t>(e * kBufs * kCB);
    int buf = 0;
    uint32_t tphase = 0;
    // Completion counter of the last unit, published by lane 0 once its bulk
    // stores have completed; every epilogue warp of the unit's CTAs adds
    // kSigShare, kDepUnit in all.
    constexpr int kSigShare = kDepUnit / (CL * kEpiWarps);
    static_assert(kSigShare * CL * kEpiWarps == kDepUnit, "counter share");
    int* pend_sig = nullptr;
    int units_done = 0;  // units of this CTA taken so far (as counted by the producer)
    for (long long t = unit0; t < total; t += ustride) {
      const int gr = find_group(P, t);
      const GroupArgs& G = P.grp[gr];
      const CUtensorMap* tmOut = &P.tmOut[gr];
      const CUtensorMap* tmOutT = &P.tmOutT[gr];
      int b, I, J;
      tile_decode(G.space, t - G.tile_begin, &b, &I, &J);
      I = row_tile(I);
      // A row tile past the last one (second CTA of a cluster, odd row-tile
      // count) was computed on zero-filled operands: nothing to store.
      const int n_chunks = (CL == 2 && I * kTileM >= G.M) ? 0 : kChunksPerWarp;
      // Muon step (GroupArgs::w_out): the master weights of this warp's 32
      // rows are read and written coalesced, lane l taking row 4 it + l / 8,
      // columns 4 (l % 8) .. + 3 of a chunk in pass it = 0..7, and loaded
      // one chunk ahead; chunk 0 before the accumulator wait, which hides its
      // latency.  W is written by no other kernel of the call, so it may be
      // read early.
      constexpr bool kW = WOUT != 0;
      const bool wmode = kW && G.w_out != nullptr;
      float* wbase = wmode ? G.w_out + static_cast<long long>(b) * G.bstride : nullptr;
      // The factors: the launch's (WOUT 1) or this group's (WOUT 2).
      const float w_decay = WOUT == 2 ? P.w_decay_g[gr] : P.w_decay;
      const float w_lrs = WOUT == 2 ? P.w_lrs_g[gr] : P.w_lrs;
      const int wr0 = I * kTileM + q * 32;  // first row of this warp
      uint4 wv[kW ? 8 : 1];
      auto load_w = [&](int cc, uint4 (&dst)[kW ? 8 : 1]) {
        const int col = J * kTileN + (c_begin + cc) * 32 + 4 * (lane & 7);
#pragma unroll
        for (int it = 0; it < (kW ? 8 : 1); ++it) {
          const int row = wr0 + 4 * it + (lane >> 3);
          if (row < G.M && col + 4 <= G.N)
            dst[it] = ptx::ld_global_v4(wbase + static_cast<long long>(row) * G.ld + col);
        }
      };
      if (wmode && n_chunks > 0) load_w(0, wv);
      int ready = 0;
      if (lane == 0)
        ready = detail::wait_bounded<SM2>(sy.tfull(buf), tphase, abort_flag, P.err, P.budget) ? 1 : 0;
      // The addend, diagonal and norms read below come from earlier products
      // of matrix b, and the buffers written below were read by them: the
      // producer's acquire of their counter is passed on through shared
      // memory.
      if (lane == 0 && ready) {
        if (G.dep_wait != nullptr &&
            !detail::wait_seen(ptx::smem_u32(&dep_seen_sh), units_done + 1, abort_flag, P.err, P.budget))
          ready = 0;
      }
      ++units_done;
      ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
      if (!ready) break;
      __syncwarp();
      ptx::tc_fence_after();

      const long long gi = static_cast<long long>(I) * kTileM + r_in_tile;
      const int warp_row_max = I * kTileM + q * 32 + 31;
      const bool row_ok = gi < G.M;
      const uint8_t* addm =
          G.addend ? static_cast<const uint8_t*>(G.addend) + static_cast<long long>(b) * G.bstride * EC::kBytes
                   : nullptr;
      const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                              static_cast<uint32_t>(buf * kTileN);
      const int col_base = J * kTileN + c_begin * 32;  // first column of this warp
      // Half storage keeps the diagonal 256 x 256 blocks whole, and a 2-SM
      // unit on one has computed all of it (single-CTA tiles compute only the
      // left half of an upper diagonal tile, N = 128): its warps store every
      // chunk as computed, above the diagonal too, and mirror nothing.  (The
      // tensor cores give bit-identical values at (i, j) and (j, i) of a
      // product of symmetric operands: the same exact products summed in the
      // same k order.)
      const bool diag_direct =
          SYM && SM2 && P.half_out && (col_base >> 8) == ((I * kTileM + q * 32) >> 8);
      // Addend coefficient: per row (row-indexed diagonal or none) ...
      float mscale = 1.0f;  // per-matrix scale of unscaled operands
      if (G.norms != nullptr) mscale = 1.0f / (ptx::ld_global_f32(G.norms + b) + P.eps);
      const float alpha_t = SYM ? P.alpha * (mscale * mscale) : P.alpha * mscale;
      float row_coef = P.beta;
      if (!SYM && G.diag_in != nullptr && !P.diag_per_col && row_ok)
        row_coef += ptx::ld_global_f32(G.diag_in + static_cast<long long>(b) * G.M + gi);
      row_coef *= mscale;
      // ... or per column, staged in shared memory for this warp's columns.
      const bool col_mode = !SYM && G.diag_in != nullptr && P.diag_per_col;
      if (col_mode) {
#pragma unroll
        for (int v = 0; v < kChunksPerWarp; ++v) {
          const int col = col_base + v * 32 + lane;
          colc[v * 32 + lane] =
              (P.beta + (col < G.N ? ptx::ld_global_f32(G.diag_in + static_cast<long long>(b) * G.N + col) : 0.0f)) *
              mscale;
        }
        __syncwarp();
      }
      // Addend values of one chunk (kAV 16-byte vectors of 8 bf16 or 4 fp32),
      // prefetched one chunk ahead so their latency overlaps the previous
      // chunk's work.  The addend, diagonal and norms are read with plain
      // (coherent) global loads: in a whole call the kernel that wrote them
      // may still be running, which the non-coherent read-only path does not
      // allow.
      constexpr int kPer = 16 / EC::kBytes;  // elements per 16-byte vector
      auto load_addend = [&](int cc, uint4 (&dst)[kAV]) {
        const int gj0 = col_base + cc * 32;
#pragma unroll
        for (int g = 0; g < kAV; ++g) dst[g] = make_uint4(0u, 0u, 0u, 0u);
        if (addm == nullptr || !row_ok || gj0 >= G.N || (SYM && gj0 > gi && !diag_direct)) return;
        const uint4* src = reinterpret_cast<const uint4*>(addm + (gi * G.ld + gj0) * EC::kBytes);
#pragma unroll
        for (int g = 0; g < kAV; ++g)
          if (gj0 + kPer * g + kPer <= G.N) dst[g] = ptx::ld_global_v4(src + g);
      };
      // Staging-chunk offset of element (row, col) for this element type.
      auto soff = [](int row, int col) -> uint32_t {
        return F32 ? stage_off32(row, col) : stage_off(row, col);
      };
      int groups = 0;  // bulk groups this tile has committed (lane 0)
      uint4 av[kAV];
      load_addend(0, av);

#pragma unroll 1
      for (int cc = 0; cc < n_chunks; ++cc) {
        const int gj0 = col_base + cc * 32;
        if (gj0 >= G.N) break;                   // warp-uniform
        if (SYM && gj0 > warp_row_max && !diag_direct) break;  // warp-uniform: above the diagonal
        uint4 an[kAV];
        if (cc + 1 < kChunksPerWarp) load_addend(cc + 1, an);
        uint32_t v[32];
        ptx::tmem_ld_32cols(t_lane + static_cast<uint32_t>((c_begin + cc) * 32), v);
        ptx::tmem_wait_ld();
        // Rows beyond M hold zeros (zero-filled operands); their stores are clipped.
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = alpha_t * __uint_as_float(v[j]);
        if (addm != nullptr) {
          float x[32];
#pragma unroll
          for (int g = 0; g < kAV; ++g) {
            const uint32_t w4[4] = {av[g].x, av[g].y, av[g].z, av[g].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              if (F32) {
                x[4 * g + h] = __uint_as_float(w4[h]);
              } else {
                x[8 * g + 2 * h] = detail::bf16_lo(w4[h]);
                x[8 * g + 2 * h + 1] = detail::bf16_hi(w4[h]);
              }
            }
          }
          if (col_mode) {
            const float4* cp = reinterpret_cast<const float4*>(colc + cc * 32);
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              const float4 k4 = cp[h];
              f[4 * h + 0] = fmaf(k4.x, x[4 * h + 0], f[4 * h + 0]);
              f[4 * h + 1] = fmaf(k4.y, x[4 * h + 1], f[4 * h + 1]);
              f[4 * h + 2] = fmaf(k4.z, x[4 * h + 2], f[4 * h + 2]);
              f[4 * h + 3] = fmaf(k4.w, x[4 * h + 3], f[4 * h + 3]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = fmaf(row_coef, x[j], f[j]);
          }
        }
        if (SYM && G.diag_out != nullptr && row_ok && gi >= gj0 && gi < gj0 + 32) {
          // The diagonal element goes to the fp32 side vector; 0 is stored.
          float dval = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (gj0 + j == gi) {
              dval = f[j];
              f[j] = 0.0f;
            }
          }
          G.diag_out[static_cast<long long>(b) * G.M + gi] = dval;
        }
        if (wmode) {
          // Muon step: the master weights take this chunk's values in place
          // of the stored iterate, w = w_decay w - w_lrs bf16(f).  The rounded
          // values go through the warp's staging chunk (fp32, 128-byte rows,
          // 128-byte swizzle: conflict-free both ways), so that W moves in
          // whole 128-byte rows.
          uint4 wn[kW ? 8 : 1];
          if (cc + 1 < n_chunks) load_w(cc + 1, wn);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint32_t lo = detail::pack_bf16x2(f[4 * g], f[4 * g + 1]);
            const uint32_t hi = detail::pack_bf16x2(f[4 * g + 2], f[4 * g + 3]);
            ptx::st_shared_v4(stg + stage_off32(lane, 4 * g), lo << 16, lo & 0xFFFF0000u, hi << 16,
                              hi & 0xFFFF0000u);
          }
          __syncwarp();
          const int col = gj0 + 4 * (lane & 7);
#pragma unroll
          for (int it = 0; it < (kW ? 8 : 1); ++it) {
            const int rr = 4 * it + (lane >> 3);
            const int row = wr0 + rr;
            if (row < G.M && col + 4 <= G.N) {
              uint32_t o4[4];
              ptx::ld_shared_v4(stg + stage_off32(rr, 4 * (lane & 7)), o4);
              const float w[4] = {__uint_as_float(wv[it].x), __uint_as_float(wv[it].y),
                                  __uint_as_float(wv[it].z), __uint_as_float(wv[it].w)};
              ptx::st_global_v4(wbase + static_cast<long long>(row) * G.ld + col,
                                __float_as_uint(fmaf(-w_lrs, __uint_as_float(o4[0]), w_decay * w[0])),
                                __float_as_uint(fmaf(-w_lrs, __uint_as_float(o4[1]), w_decay * w[1])),
                                __float_as_uint(fmaf(-w_lrs, __uint_as_float(o4[2]), w_decay * w[2])),
                                __float_as_uint(fmaf(-w_lrs, __uint_as_float(o4[3]), w_decay * w[3])));
            }
          }
          __syncwarp();  // the staging chunk is rewritten by the next chunk
#pragma unroll
          for (int g = 0; g < (kW ? 8 : 1); ++g) wv[g] = wn[g];
#pragma unroll
          for (int g = 0; g < kAV; ++g) av[g] = an[g];
          continue;
        }
        // Output words: 32 fp32 (rounded to tf32 when they feed an MMA) or 16
        // pairs of bf16; ew(j) is element j as raw bits.
        constexpr int kW = F32 ? 32 : 16;
        uint32_t w[kW];
#pragma unroll
        for (int h = 0; h < kW; ++h) {
          if (F32)
            w[h] = P.round_tf32 ? round_tf32_bits(f[h]) : __float_as_uint(f[h]);
          else
            w[h] = detail::pack_bf16x2(f[2 * h], f[2 * h + 1]);
        }
        auto st_elem = [&](uint32_t addr, int j) {
          if (F32)
            ptx::st_shared_u32(addr, w[j]);
          else
            ptx::st_shared_u16(addr, static_cast<uint16_t>((w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu));
        };
        auto st_row = [&](uint32_t d) {  // this lane's row of the chunk, 16 bytes at a time
#pragma unroll
          for (int g = 0; g < kW / 4; ++g)
            ptx::st_shared_v4(d + soff(lane, g * kPer), w[4 * g], w[4 * g + 1], w[4 * g + 2],
                              w[4 * g + 3]);
        };
        // Stage the chunk in shared memory and write it with bulk tensor
        // stores (rows beyond M or columns beyond N are clipped by the TMA).
        const int R0 = I * kTileM + q * 32;  // first row of this warp (multiple of 32)
        // Box of 32 rows staged at `src` to (row y, column x) of output
        // `which` (0: [M][N], 1: the transposed [N][M]).
        auto put = [&](uint32_t src, int x, int y, int which) {
          if (lane == 0) ptx::tma_store_3d(which ? tmOutT : tmOut, src, x, y, b);
        };
        // Before a box is stored: its staging writes visible to the async proxy.
        auto put_begin = [&]() {
          ptx::fence_proxy_async_smem();
          __syncwarp();
        };
        // After: one bulk group per stored chunk.
        auto put_end = [&]() {
          if (lane == 0) {
            ptx::bulk_commit();
            ++groups;
          }
        };
        if (lane == 0) {
          if (kWide) {
            if (!(cc & 1)) ptx::bulk_wait_read<0>();
          } else if (kBufs == 2 && !SYM && !P.out_t) {
            ptx::bulk_wait_read<1>();
          } else {
            ptx::bulk_wait_read<0>();
          }
        }
        __syncwarp();
        if (kWide) {
          // Chunks 2k and 2k + 1 fill one 32 x 64 box (4 KB, 128-byte rows):
          // the even chunk waited above for the previous box's read; the odd
          // chunk, or a last even one, stores the box.  Columns past N (the
          // unwritten half of a last even chunk's box) are clipped by the TMA.
          const int h = cc & 1;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            ptx::st_shared_v4(stg + stage_off_wide(lane, h * 4 + g), w[4 * g], w[4 * g + 1],
                              w[4 * g + 2], w[4 * g + 3]);
          const bool more = cc + 1 < n_chunks && gj0 + 32 < G.N;
          if (h == 1 || !more) {
            put_begin();
            put(stg, gj0 - h * 32, R0, 0);
            put_end();
          }
        } else if (!SYM && P.out_t) {
          // The chunk at (R0, gj0) and its transpose at (gj0, R0) of the
          // transposed output.
          const uint32_t d = stg;
          const uint32_t tr = stg + kCB;
          st_row(d);
#pragma unroll
          for (int j = 0; j < 32; ++j) st_elem(tr + soff(j, lane), j);
          put_begin();
          put(d, gj0, R0, 0);
          put(tr, R0, gj0, 1);
          put_end();
        } else if (!SYM) {
          const uint32_t d = stg + static_cast<uint32_t>((kBufs == 2 ? (cc & 1) : 0) * kCB);
          st_row(d);
          put_begin();
          put(d, gj0, R0, 0);
          put_end();
        } else if (diag_direct || (gj0 < R0 && P.half_out && (gj0 >> 8) != (R0 >> 8))) {
          // Half storage: the chunk alone, outside the diagonal 256-blocks and
          // (diag_direct) inside them.
          st_row(stg);
          put_begin();
          put(stg, gj0, R0, 0);
          put_end();
        } else if (gj0 < R0) {
          // Below the diagonal: the chunk at (R0, gj0) and its transpose at (gj0, R0).
          const uint32_t d = stg;
          const uint32_t tr = stg + kCB;
          st_row(d);
#pragma unroll
          for (int j = 0; j < 32; ++j) st_elem(tr + soff(j, lane), j);
          put_begin();
          put(d, gj0, R0, 0);
          put(tr, R0, gj0, 0);
          put_end();
        } else {
          // Diagonal 32 x 32 block (gj0 == R0): entry (r, j) takes the value
          // computed at (max(r, j), min(r, j)), so the block is bit-symmetric.
          const uint32_t d = stg;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j <= lane) st_elem(d + soff(lane, j), j);
            if (j < lane) st_elem(d + soff(j, lane), j);
          }
          put_begin();
          put(d, gj0, R0, 0);
          put_end();
        }
#pragma unroll
        for (int g = 0; g < kAV; ++g) av[g] = an[g];
      }
      ptx::tc_fence_before();
      if (SM2) {
        // One arrival per warp, on CTA 0's barrier: the pair's next MMAs
        // write both CTAs' accumulators.
        __syncwarp();
        if (lane == 0) {
          if (leader)
            ptx::mbar_arrive(sy.tempty(buf));
          else
            ptx::mbar_arrive_remote(ptx::mapa(sy.tempty(buf), 0));
        }
      } else {
        ptx::mbar_arrive(sy.tempty(buf));
      }
      if (lane == 0) {
        // Every tile commits exactly kChunksPerWarp bulk groups (empty ones
        // pad the chunks it did not store), so once all but the last
        // kChunksPerWarp have completed, the previous unit's stores, issued a
        // whole tile ago, have landed: publish that unit now, without waiting
        // for this unit's stores.
        for (; groups < kChunksPerWarp; ++groups) ptx::bulk_commit();
        if (pend_sig != nullptr) {
          ptx::bulk_wait_complete<kChunksPerWarp>();
          ptx::fence_proxy_async_global();
          ptx::red_release_gpu_add(pend_sig, kSigShare);
        }
        pend_sig = G.dep_sig != nullptr ? G.dep_sig + b : nullptr;
      }
      buf ^= 1;
      if (buf == 0) tphase ^= 1u;
    }
    // Staging buffers stay valid until every bulk store of this warp is done.
    if (lane == 0) {
      ptx::bulk_wait_all();
      if (pend_sig != nullptr && !*abort_flag) {
        ptx::fence_proxy_async_global();
        ptx::red_release_gpu_add(pend_sig, kSigShare);
      }
    }
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // Neither CTA of a cluster leaves while the other may still address it.
  if (CL == 2) ptx::cluster_sync();
  if (warp == 0) {
    __syncwarp();
    if (SM2)
      ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
  if (P.dep_flags) ptx::griddep_wait();
}

}  // namespace mns
