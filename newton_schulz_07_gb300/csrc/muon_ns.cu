// C-ABI entry points (include/muon_ns.h): argument checks, workspace layout,
// TMA tensor maps and the launch sequence of one batched NS call.
//
//   norm (ns_norm_partial) -> steps x [Gram, poly, update]
//
// The first step reads G itself and applies s = 1 / (||G||_F + eps) in its
// epilogues, so no scaled copy of G is made; steps == 0 runs the norm and the
// scale kernel (ns_scale) instead.  Each product launch takes one pair mode
// from its longest contraction (pair_mode in internal.h), and builds its tile
// space and B-operand boxes from it.
//
// Tall inputs (rows > cols) are never transposed in memory (bf16): with
// Y = X^T kept in the input's orientation, A = Y^T Y reads Y MN-major, and the
// update Y' = a Y + Y B reads B K-major (B is bit-symmetric), so the result
// lands in the input orientation directly.  The fp32 mode keeps every operand
// K-major and holds the iterate in both orientations instead.
//
// The iterate ping-pongs between the workspace and `out`, starting where the
// parity of `steps` makes the last step write `out`; only in place
// (out == G) with an odd step count is the result copied once at the end.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "muon_ns.h"
#include "gemm_launch.cuh"
#include "gemm_tc.cuh"
#include "internal.h"
#include "muon_step.cuh"
#include "norm.cuh"

namespace {


constexpr long long kMaxDim = 1 << 20;
constexpr float kDefaultCoeffs[3] = {3.4445f, -4.7750f, 2.0315f};
constexpr long long kWaitBudgetCycles = 4000000000LL;  // about 2 s at 2 GHz
std::atomic<long long> g_wait_budget{0};  // 0: kWaitBudgetCycles (muon_ns_set_wait_budget)
std::atomic<int> g_inject_stall{0};       // muon_ns_inject_stall

struct Problem {
  long long batch, R, C, m, n;
  bool T;    // rows > cols: the input is kept tall (Y = X^T)
  bool f32;  // fp32 stacks and iterates (tf32 tensor cores) instead of bf16
};

struct Layout {
  // deps: per-matrix completion counters of the three products (int [3][batch]),
  // right after the norm kernel's tickets so that one memset clears both.
  size_t error, tickets, deps, partials, norms, diag, x, a, b, total;
  size_t y2, w;  // fp32 mode only: a second tall-orientation iterate and the wide copy
  size_t x_bytes, a_bytes;
  int chunks;
};

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int check_shape(long long batch, long long rows, long long cols, Problem* p, bool* empty) {
  if (batch < 0 || rows < 0 || cols < 0) return MUON_NS_ERR_INVALID_ARG;
  if (batch > kMaxDim || rows > kMaxDim || cols > kMaxDim) return MUON_NS_ERR_INVALID_ARG;
  if (rows * cols >= (1LL << 31)) return MUON_NS_ERR_INVALID_ARG;
  if (rows % 8 != 0 || cols % 8 != 0) return MUON_NS_ERR_ALIGNMENT;
  p->batch = batch;
  p->R = rows;
  p->C = cols;
  p->T = rows > cols;
  p->f32 = false;
  p->m = p->T ? cols : rows;
  p->n = p->T ? rows : cols;
  *empty = batch == 0 || rows == 0 || cols == 0;
  return MUON_NS_OK;
}

// Grid of a per-matrix memory-bound kernel: x over a matrix's chunks, y over
// the stack up to the hardware's 65535 (the kernels loop over the rest).
dim3 batch_grid(long long chunks, long long batch) {
  return dim3(static_cast<unsigned>(chunks), static_cast<unsigned>(batch < 65535 ? batch : 65535));
}

Layout make_layout(const Problem& p) {
  Layout L;
  const size_t eb = p.f32 ? 4 : 2;  // bytes per element of G, X, A, B
  const long long vec = p.R * p.C / (p.f32 ? 4 : 8);
  L.chunks = static_cast<int>((vec + mns::kNormChunkVec - 1) / mns::kNormChunkVec);
  if (L.chunks < 1) L.chunks = 1;
  size_t off = 0;
  L.error = off;
  off += 256;
  L.tickets = off;
  L.deps = off + 4 * static_cast<size_t>(p.batch);
  off = round_up(off + 16 * static_cast<size_t>(p.batch), 256);
  L.partials = off;
  off = round_up(off + 4 * static_cast<size_t>(p.batch) * L.chunks, 256);
  L.norms = off;
  off = round_up(off + 4 * static_cast<size_t>(p.batch), 256);
  L.diag = off;
  off = round_up(off + 4 * static_cast<size_t>(p.batch) * p.m, 1024);
  L.x = off;
  L.x_bytes = eb * static_cast<size_t>(p.batch) * p.R * p.C;
  off = round_up(off + L.x_bytes, 1024);
  L.a = off;
  L.a_bytes = eb * static_cast<size_t>(p.batch) * p.m * p.m;
  off = round_up(off + L.a_bytes, 1024);
  L.b = off;
  off = round_up(off + L.a_bytes, 1024);
  L.y2 = L.w = off;
  if (p.f32) {
    off = round_up(off + L.x_bytes, 1024);
    L.w = off;
    off = round_up(off + L.x_bytes, 1024);
  }
  L.total = off;
  return L;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ----------------------------------------------------------------- devices --

struct DevInfo {
  int checked;
  int status;
  int sms;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

int current_device_info(DevInfo* out, int* dev_out = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MUON_NS_ERR_UNSUPPORTED_DEVICE;
  }
  if (dev < 0 || dev >= 64) return MUON_NS_ERR_UNSUPPORTED_DEVICE;
  if (dev_out) *dev_out = dev;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return MUON_NS_ERR_CUDA;
    }
    d.status = (major == 10 && minor == 3) ? MUON_NS_OK : MUON_NS_ERR_UNSUPPORTED_DEVICE;
    d.sms = sms;
    d.checked = 1;
  }
  *out = d;
  return d.status;
}

// ------------------------------------------------------------- tensor maps --

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 3-D map over a bf16 (or fp32) stack [batch][rows][inner] (inner
// contiguous) with a box of box_inner x box_rows x 1; 128-byte swizzle for
// operand tiles, 64-byte (bf16) or 128-byte (fp32) for 32 x 32 output chunks.
bool make_map(CUtensorMap* map, const void* base, long long inner, long long rows,
              long long batch, int box_inner, int box_rows, bool f32 = false,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  const long long eb = f32 ? 4 : 2;
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner * eb),
                           static_cast<cuuint64_t>(inner * rows * eb)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
         const_cast<void*>(base), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- launches --

// Output map: [batch][M][N], 32-row boxes of 128-byte rows with the 128-byte
// swizzle (fp32 32 x 32, or bf16 32 x 64 for `wide` outputs), or of 64-byte
// rows with the 64-byte swizzle (bf16 32 x 32).
bool make_out_map(CUtensorMap* map, const void* base, long long M, long long N, long long batch,
                  bool f32, bool wide = false) {
  const bool b128 = f32 || wide;
  return make_map(map, base, N, M, batch, (wide && !f32) ? 64 : 32, 32, f32,
                  b128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

// K per pipeline stage and M/N elements per 128-byte row (the TMA box sizes).
inline int block_k(bool f32) { return f32 ? mns::ElemCfg<true>::kBlockK : mns::ElemCfg<false>::kBlockK; }
inline int mn_chunk(bool f32) { return f32 ? mns::ElemCfg<true>::kMnChunk : mns::ElemCfg<false>::kMnChunk; }

int grid_for(long long tiles, int sms) {
  const long long g = tiles < sms ? tiles : sms;
  return static_cast<int>(g < 1 ? 1 : g);
}

int to_status(cudaError_t e) { return e == cudaSuccess ? MUON_NS_OK : MUON_NS_ERR_CUDA; }

// One stack's buffers for one NS step.  All stacks of one launch share the
// orientation (p.T), because operand majorness is a kernel template argument.
struct StepIO {
  Problem p;
  const uint16_t* X;   // the iterate, or the raw G in the first step
  uint16_t* A;         // Gram output / polynomial input
  uint16_t* B;         // polynomial output (zero diagonal) / update input
  float* D;            // fp32 diagonal of B
  const float* norms;  // non-null in the first step: X is unscaled
  uint16_t* Xn;        // update output
  uint16_t* Xt;        // update only, optional: the transposed output
  bool half;           // A and B are half-stored (lower triangle and diagonal 256-blocks)
  // Optional per-matrix completion counters int [3][batch] (Gram, poly,
  // update), cleared at the start of the call, and the step index: each
  // product waits for the previous product of the same matrix through them
  // instead of for the whole previous kernel.
  int* dep;
  int step;
  // Update only, optional: the last update of a Muon step updates these fp32
  // master weights ([batch][rows][cols]) in place of storing Xn:
  // W = w_decay W - w_lrs bf16(Xn).
  float* W;
  float w_decay, w_lrs;
};

// Counter value per matrix after one step of a product: its units per matrix
// (CTA pairs for bf16) times the kernel's increment per unit.
long long dep_per_step(int sym, long long M, long long N) {
  return mns::make_tile_space(sym, 1, static_cast<int>(M), static_cast<int>(N), 1).total *
         static_cast<long long>(mns::kDepUnit);
}
long long dep_per_step_sym(const Problem& p) { return dep_per_step(1, p.m, p.m); }

// A launch waits through counters only if every group has them; otherwise
// it waits for the whole previous kernel (its groups still signal).
bool all_have_dep(const StepIO* io, int ng) {
  for (int i = 0; i < ng; ++i)
    if (io[i].dep == nullptr) return false;
  return true;
}
long long dep_per_step_update(const Problem& p) {
  return p.T ? dep_per_step(0, p.n, p.m) : dep_per_step(0, p.m, p.n);
}

// The fused bf16 calls store A and B half (each product reads the missing
// triangle transposed); the per-step entry points keep them full.
#ifndef MNS_HALF_SYM
#define MNS_HALF_SYM 1
#endif
// Whole calls order their products through per-matrix counters (StepIO::dep);
// MNS_DEP_FLAGS=0 orders them by whole kernels.
#ifndef MNS_DEP_FLAGS
#define MNS_DEP_FLAGS 1
#endif

// Launch parameters (about 4 KB) are built on the host and copied at launch.
mns::GemmParams* new_params(int ng, float alpha, float beta, float eps, int* err) {
  static thread_local mns::GemmParams P;
  std::memset(&P, 0, sizeof(P));
  P.num_groups = ng;
  P.alpha = alpha;
  P.beta = beta;
  P.eps = eps;
  P.err = err;
  const long long budget = g_wait_budget.load();
  P.budget = budget > 0 ? budget : kWaitBudgetCycles;
  return &P;
}

// Rows of a K-major B-operand box: each CTA of a pair loads half the panel.
inline int b_box_rows(mns::PairMode mode) { return mode != mns::kSingle ? mns::kTileN / 2 : mns::kTileN; }

void set_group(mns::GemmParams* P, int i, int sym, long long batch, long long M, long long N,
               long long K, long long* total, bool f32, mns::PairMode mode) {
  mns::GroupArgs& G = P->grp[i];
  G.space = mns::make_tile_space(sym, static_cast<int>(batch), static_cast<int>(M),
                                 static_cast<int>(N), mode != mns::kSingle ? 1 : 0);
  G.tile_begin = *total;
  *total += G.space.total;
  G.M = static_cast<int>(M);
  G.N = static_cast<int>(N);
  G.K = static_cast<int>(K);
  G.num_kb = static_cast<int>((K + block_k(f32) - 1) / block_k(f32));
  G.ld = N;
  G.bstride = M * N;
}

int run_gram(const StepIO* io, int ng, float eps, int* err, int sms, cudaStream_t st) {
  mns::GemmParams* P = new_params(ng, 1.0f, 0.0f, eps, err);
  long long total = 0;
  const bool T = io[0].p.T, f32 = io[0].p.f32;
  const int bk = block_k(f32), mc = mn_chunk(f32);
  P->round_tf32 = 1;  // A feeds the next product
  P->half_out = io[0].half ? 1 : 0;
  int max_k = 0;
  for (int i = 0; i < ng; ++i)
    if (io[i].p.n > max_k) max_k = static_cast<int>(io[i].p.n);
  const mns::PairMode mode = mns::pair_mode(f32, max_k);
  // A first step has no earlier product to wait on, only the norm kernel, so
  // a launch that holds one waits for the whole previous kernel, whatever
  // step its other groups are at.
  bool by_counter = all_have_dep(io, ng);
  for (int i = 0; i < ng; ++i) by_counter = by_counter && io[i].step > 0;
  for (int i = 0; i < ng; ++i) {
    const Problem& p = io[i].p;
    set_group(P, i, 1, p.batch, p.m, p.m, p.n, &total, f32, mode);
    P->grp[i].norms = io[i].norms;
    // Signals the Gram counter; waits for the previous step's update.
    if (io[i].dep != nullptr) P->grp[i].dep_sig = io[i].dep;
    if (by_counter) {
      P->grp[i].dep_wait = io[i].dep + 2 * p.batch;
      P->grp[i].dep_target = static_cast<int>(io[i].step * dep_per_step_update(p));
      P->dep_flags = 1;
    }
    if (!make_out_map(&P->tmOut[i], io[i].A, p.m, p.m, p.batch, f32)) return MUON_NS_ERR_CUDA;
    if (!T) {
      // X [batch][m][n]: rows of X are the K-major operand rows.
      if (!make_map(&P->tmA[i], io[i].X, p.n, p.m, p.batch, bk, mns::kTileM, f32) ||
          !make_map(&P->tmB[i], io[i].X, p.n, p.m, p.batch, bk, b_box_rows(mode), f32))
        return MUON_NS_ERR_CUDA;
    } else {
      // Y [batch][n][m]: columns of Y are the operand rows, read MN-major.
      if (!make_map(&P->tmA[i], io[i].X, p.m, p.n, p.batch, mc, bk, f32)) return MUON_NS_ERR_CUDA;
      P->tmB[i] = P->tmA[i];
    }
  }
  P->total_tiles = total;
  const int grid = grid_for(total, sms);
  if (f32)
    return to_status(T ? mns::launch_sym_mnmn_f32(*P, mode, grid, st) : mns::launch_sym_kk_f32(*P, mode, grid, st));
  return to_status(T ? mns::launch_sym_mnmn(*P, mode, grid, st) : mns::launch_sym_kk(*P, mode, grid, st));
}

int run_poly(const StepIO* io, int ng, float b, float c, int* err, int sms, cudaStream_t st) {
  mns::GemmParams* P = new_params(ng, c, b, 0.0f, err);
  long long total = 0;
  const bool f32 = io[0].p.f32;
  const int bk = block_k(f32);
  P->round_tf32 = 1;  // B feeds the update product
  P->half_out = io[0].half ? 1 : 0;
  int max_k = 0;
  for (int i = 0; i < ng; ++i)
    if (io[i].p.m > max_k) max_k = static_cast<int>(io[i].p.m);
  const mns::PairMode mode = mns::pair_mode(f32, max_k);
  for (int i = 0; i < ng; ++i) {
    const long long m = io[i].p.m, batch = io[i].p.batch;
    set_group(P, i, 1, batch, m, m, m, &total, f32, mode);
    P->grp[i].addend = io[i].A;
    P->grp[i].diag_out = io[i].D;
    // Signals the poly counter; waits for this step's Gram.
    if (io[i].dep != nullptr) P->grp[i].dep_sig = io[i].dep + batch;
    if (all_have_dep(io, ng)) {
      P->grp[i].dep_wait = io[i].dep;
      P->grp[i].dep_target = static_cast<int>((io[i].step + 1) * dep_per_step_sym(io[i].p));
      // Injected stall: a target the Gram kernel never reaches.
      if (io[i].step == 0 && g_inject_stall.load()) P->grp[i].dep_target += 1;
      P->dep_flags = 1;
    }
    if (io[i].half) {
      // A is half-stored: both operands read its upper part transposed.
      P->grp[i].half_a = P->grp[i].half_b = 1;
      if (!make_map(&P->tmA2[i], io[i].A, m, m, batch, mn_chunk(f32), bk, f32)) return MUON_NS_ERR_CUDA;
      P->tmB2[i] = P->tmA2[i];
    }
    if (!make_map(&P->tmA[i], io[i].A, m, m, batch, bk, mns::kTileM, f32) ||
        !make_map(&P->tmB[i], io[i].A, m, m, batch, bk, b_box_rows(mode), f32) ||
        !make_out_map(&P->tmOut[i], io[i].B, m, m, batch, f32))
      return MUON_NS_ERR_CUDA;
  }
  P->total_tiles = total;
  const int grid = grid_for(total, sms);
  return to_status(f32 ? mns::launch_sym_kk_f32(*P, mode, grid, st) : mns::launch_sym_kk(*P, mode, grid, st));
}

// `round_out`: fp32 mode only, the result feeds another step's products.
int run_update(const StepIO* io, int ng, float alpha_x, float eps, bool round_out, int* err,
               int sms, cudaStream_t st) {
  mns::GemmParams* P = new_params(ng, 1.0f, alpha_x, eps, err);
  long long total = 0;
  const bool T = io[0].p.T, f32 = io[0].p.f32;
  const int bk = block_k(f32), mc = mn_chunk(f32);
  int max_k = 0;
  P->diag_per_col = T ? 1 : 0;  // (a + D_i) scales row i of X, or column i of Y
  P->round_tf32 = round_out ? 1 : 0;
  P->out_t = io[0].Xt != nullptr ? 1 : 0;
  for (int i = 0; i < ng; ++i)
    if (io[i].p.m > max_k) max_k = static_cast<int>(io[i].p.m);
  const mns::PairMode mode = mns::pair_mode(f32, max_k);
  // The Muon step's last update (master-weight output) runs its own kernels,
  // always with 4 epilogue warps.
  bool wout = false;
  for (int i = 0; i < ng; ++i) wout = wout || io[i].W != nullptr;
  for (int i = 0; wout && i < ng; ++i)
    if (io[i].W == nullptr) return MUON_NS_ERR_INVALID_ARG;  // all groups of a launch or none
  // The 4-warp bf16 update writes 32 x 64 output boxes.
  const bool wide_out = !f32 && (wout || mns::update_epi_warps(mode, max_k) == 4);
  if (!f32 && P->out_t) return MUON_NS_ERR_INVALID_ARG;  // transposed outputs are fp32 only
  for (int i = 0; i < ng; ++i) {
    const Problem& p = io[i].p;
    if (!T) {
      // Xn [m][n] = a X + B X: A operand = rows of B, B operand = X read MN-major.
      set_group(P, i, 0, p.batch, p.m, p.n, p.m, &total, f32, mode);
      if (!make_map(&P->tmA[i], io[i].B, p.m, p.m, p.batch, bk, mns::kTileM, f32) ||
          !make_map(&P->tmB[i], io[i].X, p.n, p.m, p.batch, mc, bk, f32) ||
          !make_out_map(&P->tmOut[i], io[i].Xn, p.m, p.n, p.batch, f32, wide_out))
        return MUON_NS_ERR_CUDA;
    } else {
      // Yn [n][m] = a Y + Y B: A operand = rows of Y, B operand = rows of B (= columns).
      set_group(P, i, 0, p.batch, p.n, p.m, p.m, &total, f32, mode);
      if (!make_map(&P->tmA[i], io[i].X, p.m, p.n, p.batch, bk, mns::kTileM, f32) ||
          !make_map(&P->tmB[i], io[i].B, p.m, p.m, p.batch, bk, b_box_rows(mode), f32) ||
          !make_out_map(&P->tmOut[i], io[i].Xn, p.n, p.m, p.batch, f32, wide_out))
        return MUON_NS_ERR_CUDA;
    }
    P->grp[i].addend = io[i].X;
    P->grp[i].diag_in = io[i].D;
    P->grp[i].norms = io[i].norms;
    if (io[i].W != nullptr) {
      if (f32) return MUON_NS_ERR_INVALID_ARG;  // the Muon step runs the bf16 NS
      P->grp[i].w_out = io[i].W;
      P->w_decay_g[i] = io[i].w_decay;
      P->w_lrs_g[i] = io[i].w_lrs;
    }
    // Signals the update counter; waits for this step's polynomial.
    if (io[i].dep != nullptr) P->grp[i].dep_sig = io[i].dep + 2 * p.batch;
    if (all_have_dep(io, ng)) {
      P->grp[i].dep_wait = io[i].dep + p.batch;
      P->grp[i].dep_target = static_cast<int>((io[i].step + 1) * dep_per_step_sym(p));
      P->dep_flags = 1;
    }
    if (io[i].half) {
      // B is half-stored: its rows are the A operand (wide) or the B operand
      // (tall); past the diagonal block they are read transposed.
      CUtensorMap* alt = T ? &P->tmB2[i] : &P->tmA2[i];
      (T ? P->grp[i].half_b : P->grp[i].half_a) = 1;
      if (!make_map(alt, io[i].B, p.m, p.m, p.batch, mc, bk, f32)) return MUON_NS_ERR_CUDA;
    }
    // Transposed output: [batch][N][M] of this launch's [batch][M][N] output.
    if (io[i].Xt != nullptr &&
        !make_out_map(&P->tmOutT[i], io[i].Xt, T ? p.m : p.n, T ? p.n : p.m, p.batch, f32))
      return MUON_NS_ERR_CUDA;
  }
  P->total_tiles = total;
  const int grid = grid_for(total, sms);
  if (f32)
    return to_status(T ? mns::launch_full_kk_f32(*P, mode, max_k, grid, st)
                       : mns::launch_full_kmn_f32(*P, mode, max_k, grid, st));
  if (wout) {
    // One pair of factors for the launch unless the groups differ: the
    // launch-wide kernel reads them without indexing the group arguments.
    bool per_group = false;
    for (int i = 1; i < ng; ++i)
      per_group = per_group || io[i].w_decay != io[0].w_decay || io[i].w_lrs != io[0].w_lrs;
    P->w_decay = io[0].w_decay;
    P->w_lrs = io[0].w_lrs;
    return to_status(T ? mns::launch_full_kk_w(*P, mode, grid, per_group, st)
                       : mns::launch_full_kmn_w(*P, mode, grid, per_group, st));
  }
  return to_status(T ? mns::launch_full_kk(*P, mode, max_k, grid, st)
                     : mns::launch_full_kmn(*P, mode, max_k, grid, st));
}

// `clear`: zero the tickets first (callers that clear them together with the
// dependency counters pass false).
int run_normalize(const Problem& p, const Layout& L, const void* G, void* X, float eps,
                  uint8_t* ws, cudaStream_t st, bool clear = true) {
  const long long vec = p.R * p.C / (p.f32 ? 4 : 8);
  if (clear && cudaMemsetAsync(ws + L.tickets, 0, 4 * static_cast<size_t>(p.batch), st) != cudaSuccess)
    return MUON_NS_ERR_CUDA;
  const dim3 grid = batch_grid(L.chunks, p.batch);
  const int nb = static_cast<int>(p.batch);
  if (mns::launch_pdl(p.f32 ? mns::ns_norm_partial<true> : mns::ns_norm_partial<false>, grid, dim3(mns::kNormThreads), 0, st,
                      reinterpret_cast<const uint4*>(G), vec, L.chunks, nb,
                      reinterpret_cast<float*>(ws + L.partials),
                      reinterpret_cast<unsigned int*>(ws + L.tickets),
                      reinterpret_cast<float*>(ws + L.norms)) != cudaSuccess)
    return MUON_NS_ERR_CUDA;
  if (X == nullptr) return MUON_NS_OK;  // norms only
  if (mns::launch_pdl(p.f32 ? mns::ns_scale<true> : mns::ns_scale<false>, grid, dim3(mns::kNormThreads), 0, st,
                      reinterpret_cast<const uint4*>(G), reinterpret_cast<uint4*>(X), vec, nb,
                      reinterpret_cast<const float*>(ws + L.norms), eps) != cudaSuccess)
    return MUON_NS_ERR_CUDA;
  return MUON_NS_OK;
}

// One stack of a (possibly grouped) NS call.
struct Stack {
  Problem p;
  Layout L;
  const uint16_t* G;
  uint16_t* out;
  uint8_t* ws;  // this stack's workspace (layout L)
  uint16_t* cur;
  // Muon step, optional: the last update writes W = w_decay W - w_lrs NS(G)
  // (fp32 masters) instead of `out`, which then holds no result.
  float* W = nullptr;
  float w_decay = 1.0f, w_lrs = 0.0f;
};

// NS of several stacks, all kernels reporting to `err`.  Stacks are launched
// together, per orientation, in launches of at most kMaxGroups groups.
// `cleared`: the caller has already zeroed every stack's tickets and
// dependency counters.  `norms_ready`: the caller has already written every
// stack's norms of G (the Muon step's momentum kernel), so no norm kernel runs.
int run_ns_stacks(Stack* S, int ns, int steps, const float abc[3], float eps, int* err, int sms,
                  cudaStream_t st, bool cleared = false, bool norms_ready = false) {
  int s = MUON_NS_OK;
  if (steps == 0) {
    for (int i = 0; i < ns; ++i)
      if ((s = run_normalize(S[i].p, S[i].L, S[i].G, S[i].out, eps, S[i].ws, st)) != MUON_NS_OK)
        return s;
    return MUON_NS_OK;
  }
  // Norms only; the first step reads G itself and applies s = 1/(norm + eps)
  // in its epilogues (A0 = s^2 G G^T, X1 = s O G + s (a + D) G), so no scaled
  // copy of G is written or read.  One memset clears each stack's norm
  // tickets and its dependency counters.
  for (int i = 0; i < ns; ++i) {
    if (!cleared &&
        cudaMemsetAsync(S[i].ws + S[i].L.tickets, 0, 16 * static_cast<size_t>(S[i].p.batch), st) !=
            cudaSuccess)
      return MUON_NS_ERR_CUDA;
    if (!norms_ready &&
        (s = run_normalize(S[i].p, S[i].L, S[i].G, nullptr, eps, S[i].ws, st, false)) != MUON_NS_OK)
      return s;
  }
  StepIO io[mns::kMaxGroups];
  int members[mns::kMaxGroups];
  for (int k = 0; k < steps; ++k) {
    for (int cls = 0; cls < 2; ++cls) {  // wide stacks, then tall stacks
      int i = 0;
      while (i < ns) {
        int ng = 0;
        for (; i < ns && ng < mns::kMaxGroups; ++i) {
          if (static_cast<int>(S[i].p.T) != cls) continue;
          Stack& t = S[i];
          uint16_t* wsx = reinterpret_cast<uint16_t*>(t.ws + t.L.x);
          // Iterates alternate between the workspace and `out` so that the
          // last lands in `out`; in place (out == G) the first iterate must
          // not overwrite G while step 1 still reads it.
          uint16_t* nxt;
          if (k == 0)
            nxt = (t.out == t.G || steps % 2 == 0) ? wsx : t.out;
          else
            nxt = (t.cur == t.out) ? wsx : t.out;
          StepIO& e = io[ng];
          e = StepIO{};  // every optional field (norms, Xt) starts null
          e.p = t.p;
          e.X = (k == 0) ? t.G : t.cur;
          e.A = reinterpret_cast<uint16_t*>(t.ws + t.L.a);
          e.B = reinterpret_cast<uint16_t*>(t.ws + t.L.b);
          e.D = reinterpret_cast<float*>(t.ws + t.L.diag);
          e.norms = (k == 0) ? reinterpret_cast<const float*>(t.ws + t.L.norms) : nullptr;
          e.Xn = nxt;
          if (t.W != nullptr && k + 1 == steps) {
            // The Muon step's last update writes the masters; Xn only
            // names a valid buffer for the output tensor map.
            e.W = t.W;
            e.w_decay = t.w_decay;
            e.w_lrs = t.w_lrs;
          }
          e.half = MNS_HALF_SYM && !t.p.f32;
          e.step = k;
          // A single matrix gains nothing (its next product needs all of
          // it).  Counters stay far below 2^31 for any realistic step count;
          // past that, products wait for whole kernels.
          const long long peak = static_cast<long long>(steps) *
                                 std::max(dep_per_step_sym(t.p), dep_per_step_update(t.p));
          if (MNS_DEP_FLAGS && !t.p.f32 && t.p.batch > 1 && peak < (1LL << 30))
            e.dep = reinterpret_cast<int*>(t.ws + t.L.deps);
          members[ng++] = i;
        }
        if (ng == 0) continue;
        // Each product runs as one launch per contraction regime: stacks with
        // short contractions (K <= kShortK) and long ones take different pair
        // modes and epilogues, and sharing a launch would give one of them
        // the other's.
        StepIO sub[mns::kMaxGroups];
        auto split = [&](auto run, auto contraction) {
          for (int longk = 0; longk < 2; ++longk) {
            int n = 0;
            for (int j = 0; j < ng; ++j)
              if ((contraction(io[j].p) > mns::kShortK) == (longk != 0)) sub[n++] = io[j];
            if (n == 0) continue;
            const int r = run(sub, n);
            if (r != MUON_NS_OK) return r;
          }
          return static_cast<int>(MUON_NS_OK);
        };
        auto K_n = [](const Problem& q) { return q.n; };
        auto K_m = [](const Problem& q) { return q.m; };
        if ((s = split([&](const StepIO* v, int n) { return run_gram(v, n, eps, err, sms, st); }, K_n)) !=
            MUON_NS_OK)
          return s;
        if ((s = split([&](const StepIO* v, int n) { return run_poly(v, n, abc[1], abc[2], err, sms, st); },
                       K_m)) != MUON_NS_OK)
          return s;
        if ((s = split([&](const StepIO* v, int n) {
               return run_update(v, n, abc[0], eps, k + 1 < steps, err, sms, st);
             }, K_m)) != MUON_NS_OK)
          return s;
        for (int j = 0; j < ng; ++j) S[members[j]].cur = io[j].Xn;
      }
    }
  }
  for (int i = 0; i < ns; ++i)
    if (S[i].W == nullptr && S[i].cur != S[i].out &&
        cudaMemcpyAsync(S[i].out, S[i].cur, S[i].L.x_bytes, cudaMemcpyDeviceToDevice, st) !=
            cudaSuccess)
      return MUON_NS_ERR_CUDA;
  return MUON_NS_OK;
}

// fp32 NS.  The tf32 tensor-core path takes K-major operands only, so the
// iterate is kept in both orientations: W = the wide m x n copy, read by the
// Gram product A = W W^T, and Y = W^T (n x m), which the update reads as
// Y' = a Y + Y B with K-major operands and whose epilogue also writes W' = Y'^T.
// The first step gets the orientation of G it lacks from one transpose.
int run_ns_f32(const Problem& p, const Layout& L, const uint16_t* G, uint16_t* out, int steps,
               const float abc[3], float eps, uint8_t* ws, int sms, cudaStream_t st) {
  int* err = reinterpret_cast<int*>(ws + L.error);
  if (cudaMemsetAsync(ws + L.error, 0, 256, st) != cudaSuccess) return MUON_NS_ERR_CUDA;
  if (steps == 0) return run_normalize(p, L, G, out, eps, ws, st);
  int s = run_normalize(p, L, G, nullptr, eps, ws, st);
  if (s != MUON_NS_OK) return s;
  uint16_t* Y0 = reinterpret_cast<uint16_t*>(ws + L.x);
  uint16_t* Y1 = reinterpret_cast<uint16_t*>(ws + L.y2);
  uint16_t* W = reinterpret_cast<uint16_t*>(ws + L.w);
  const bool wide = !p.T;
  // G^T into the orientation G lacks.
  {
    const dim3 grid(static_cast<unsigned>((p.C + 31) / 32), static_cast<unsigned>((p.R + 31) / 32),
                    static_cast<unsigned>(p.batch < 65535 ? p.batch : 65535));
    if (mns::launch_pdl(mns::ns_transpose_f32, grid, dim3(32, 8), 0, st,
                        reinterpret_cast<const float*>(G), reinterpret_cast<float*>(wide ? Y0 : W),
                        static_cast<int>(p.R), static_cast<int>(p.C), static_cast<int>(p.batch)) != cudaSuccess)
      return MUON_NS_ERR_CUDA;
  }
  Problem pw = p;  // the Gram sees W: m x n, wide
  pw.R = p.m;
  pw.C = p.n;
  pw.T = false;
  Problem py = p;  // the update sees Y: n x m, tall
  py.R = p.n;
  py.C = p.m;
  py.T = true;
  const uint16_t* wsrc = wide ? G : W;
  const uint16_t* ysrc = wide ? Y0 : G;
  uint16_t* A = reinterpret_cast<uint16_t*>(ws + L.a);
  uint16_t* B = reinterpret_cast<uint16_t*>(ws + L.b);
  float* D = reinterpret_cast<float*>(ws + L.diag);
  const float* norms = reinterpret_cast<const float*>(ws + L.norms);
  for (int k = 0; k < steps; ++k) {
    const bool last = k + 1 == steps;
    StepIO g = {};
    g.p = pw;
    g.X = wsrc;
    g.A = A;
    g.norms = k == 0 ? norms : nullptr;
    if ((s = run_gram(&g, 1, eps, err, sms, st)) != MUON_NS_OK) return s;
    StepIO q = {};
    q.p = pw;
    q.A = A;
    q.B = B;
    q.D = D;
    if ((s = run_poly(&q, 1, abc[1], abc[2], err, sms, st)) != MUON_NS_OK) return s;
    // Y' never overwrites the Y it reads; for a tall input the last Y' is the
    // result (straight into out unless out is G, still read in step 1).
    uint16_t* ynext = (ysrc == Y0) ? Y1 : Y0;
    if (last && !wide && (out != G || k > 0)) ynext = out;
    StepIO u = {};
    u.p = py;
    u.X = ysrc;
    u.B = B;
    u.D = D;
    u.norms = k == 0 ? norms : nullptr;
    u.Xn = ynext;
    u.Xt = last ? (wide ? out : nullptr) : W;
    if ((s = run_update(&u, 1, abc[0], eps, !last, err, sms, st)) != MUON_NS_OK) return s;
    ysrc = ynext;
    wsrc = W;
  }
  if (!wide && ysrc != out &&
      cudaMemcpyAsync(out, ysrc, L.x_bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MUON_NS_ERR_CUDA;
  return MUON_NS_OK;
}

int run_ns(const Problem& p, const Layout& L, const uint16_t* G, uint16_t* out, int steps,
           const float abc[3], float eps, uint8_t* ws, int sms, cudaStream_t st) {
  int* err = reinterpret_cast<int*>(ws + L.error);
  // The error word, the norm tickets and the dependency counters lie end to
  // end at the start of the workspace: one memset clears them.
  if (L.error != 0 || L.tickets != 256 || L.deps != L.tickets + 4 * static_cast<size_t>(p.batch))
    return MUON_NS_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, L.deps + 12 * static_cast<size_t>(p.batch), st) != cudaSuccess)
    return MUON_NS_ERR_CUDA;
  Stack S;
  S.p = p;
  S.L = L;
  S.G = G;
  S.out = out;
  S.ws = ws;
  S.cur = nullptr;
  return run_ns_stacks(&S, 1, steps, abc, eps, err, sms, st, true);
}

int check_scalars(int steps, const float* coeffs, float eps, float abc[3]) {
  if (steps < 0) return MUON_NS_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return MUON_NS_ERR_INVALID_ARG;
  const float* c = coeffs ? coeffs : kDefaultCoeffs;
  for (int i = 0; i < 3; ++i) {
    if (!std::isfinite(c[i])) return MUON_NS_ERR_INVALID_ARG;
    abc[i] = c[i];
  }
  return MUON_NS_OK;
}

// ----------------------------------------------------- cached workspaces --

struct Cache {
  void* ptr;
  size_t bytes;
};
std::mutex g_cache_mu;
Cache g_cache[64];

}  // namespace

extern "C" {

const char* muon_ns_version(void) { return "0.1.0"; }

const char* muon_ns_status_string(int status) {
  switch (status) {
    case MUON_NS_OK: return "ok";
    case MUON_NS_ERR_INVALID_ARG: return "invalid argument";
    case MUON_NS_ERR_ALIGNMENT: return "alignment: rows/cols must be multiples of 8 and pointers 16-byte aligned";
    case MUON_NS_ERR_UNSUPPORTED_DEVICE: return "unsupported device: compute capability 10.3 (sm_103) required";
    case MUON_NS_ERR_WORKSPACE: return "workspace missing or too small";
    case MUON_NS_ERR_CUDA: return "CUDA call failed";
    case MUON_NS_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    default: return "unknown status";
  }
}

int muon_ns_device_supported(int device) {
  int prev = -1;
  if (device >= 0) {
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
      cudaGetLastError();
      return MUON_NS_ERR_UNSUPPORTED_DEVICE;
    }
  }
  DevInfo d;
  const int s = current_device_info(&d);
  if (prev >= 0 && prev != device) cudaSetDevice(prev);
  return s;
}

int muon_ns_workspace_size(int batch, int rows, int cols, size_t* bytes) {
  if (!bytes) return MUON_NS_ERR_INVALID_ARG;
  Problem p;
  bool empty;
  const int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  *bytes = empty ? 0 : make_layout(p).total;
  return MUON_NS_OK;
}

int workspace_region(bool f32, int batch, int rows, int cols, int region, size_t* offset,
                     size_t* bytes) {
  if (!offset || !bytes) return MUON_NS_ERR_INVALID_ARG;
  Problem p;
  bool empty;
  const int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  p.f32 = f32;
  const Layout L = make_layout(p);
  switch (region) {
    case MUON_NS_WS_TOTAL: *offset = 0; *bytes = L.total; break;
    case MUON_NS_WS_ERROR: *offset = L.error; *bytes = 4; break;
    case MUON_NS_WS_NORMS: *offset = L.norms; *bytes = 4 * static_cast<size_t>(p.batch); break;
    case MUON_NS_WS_X: *offset = L.x; *bytes = L.x_bytes; break;
    case MUON_NS_WS_GRAM: *offset = L.a; *bytes = L.a_bytes; break;
    case MUON_NS_WS_POLY: *offset = L.b; *bytes = L.a_bytes; break;
    case MUON_NS_WS_DIAG: *offset = L.diag; *bytes = 4 * static_cast<size_t>(p.batch) * p.m; break;
    default: return MUON_NS_ERR_INVALID_ARG;
  }
  return MUON_NS_OK;
}

int muon_ns_workspace_region(int batch, int rows, int cols, int region, size_t* offset,
                             size_t* bytes) {
  return workspace_region(false, batch, rows, cols, region, offset, bytes);
}

int muon_ns_f32_workspace_region(int batch, int rows, int cols, int region, size_t* offset,
                                 size_t* bytes) {
  return workspace_region(true, batch, rows, cols, region, offset, bytes);
}

int muon_ns_f32_workspace_size(int batch, int rows, int cols, size_t* bytes) {
  if (!bytes) return MUON_NS_ERR_INVALID_ARG;
  Problem p;
  bool empty;
  const int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  p.f32 = true;
  *bytes = empty ? 0 : make_layout(p).total;
  return MUON_NS_OK;
}

int muon_ns_ws(const muon_bf16* G, muon_bf16* out, int batch, int rows, int cols, int steps,
               const float* coeffs, float eps, void* workspace, size_t workspace_bytes,
               cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  float abc[3];
  if ((s = check_scalars(steps, coeffs, eps, abc)) != MUON_NS_OK) return s;
  if (empty) return MUON_NS_OK;
  if (!G || !out) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(G) || !aligned16(out)) return MUON_NS_ERR_ALIGNMENT;
  const Layout L = make_layout(p);
  if (!workspace || workspace_bytes < L.total) return MUON_NS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  return run_ns(p, L, G, out, steps, abc, eps, static_cast<uint8_t*>(workspace), d.sms, stream);
}

int muon_ns_ws_f32(const float* G, float* out, int batch, int rows, int cols, int steps,
                   const float* coeffs, float eps, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  p.f32 = true;
  float abc[3];
  if ((s = check_scalars(steps, coeffs, eps, abc)) != MUON_NS_OK) return s;
  if (empty) return MUON_NS_OK;
  if (!G || !out) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(G) || !aligned16(out)) return MUON_NS_ERR_ALIGNMENT;
  const Layout L = make_layout(p);
  if (!workspace || workspace_bytes < L.total) return MUON_NS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  return run_ns_f32(p, L, reinterpret_cast<const uint16_t*>(G), reinterpret_cast<uint16_t*>(out),
                    steps, abc, eps, static_cast<uint8_t*>(workspace), d.sms, stream);
}

int muon_ns(const muon_bf16* G, muon_bf16* out, int batch, int rows, int cols, int steps,
            const float* coeffs, float eps, cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  float abc[3];
  if ((s = check_scalars(steps, coeffs, eps, abc)) != MUON_NS_OK) return s;
  if (empty) return MUON_NS_OK;
  if (!G || !out) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(G) || !aligned16(out)) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  int dev = 0;
  if ((s = current_device_info(&d, &dev)) != MUON_NS_OK) return s;
  const Layout L = make_layout(p);
  std::lock_guard<std::mutex> lock(g_cache_mu);
  Cache& c = g_cache[dev];
  if (c.bytes < L.total) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
      cudaGetLastError();
      return MUON_NS_ERR_CUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return MUON_NS_ERR_WORKSPACE;
    if (c.ptr) {
      cudaFree(c.ptr);
      c.ptr = nullptr;
      c.bytes = 0;
    }
    if (cudaMalloc(&c.ptr, L.total) != cudaSuccess) {
      cudaGetLastError();
      c.ptr = nullptr;
      return MUON_NS_ERR_CUDA;
    }
    c.bytes = L.total;
  }
  return run_ns(p, L, G, out, steps, abc, eps, static_cast<uint8_t*>(c.ptr), d.sms, stream);
}

int muon_ns_grouped_workspace_size(const muon_ns_stack* stacks, int num_stacks, size_t* bytes) {
  if (!bytes || num_stacks < 0 || num_stacks > 64 || (num_stacks > 0 && !stacks))
    return MUON_NS_ERR_INVALID_ARG;
  size_t total = 0;
  for (int i = 0; i < num_stacks; ++i) {
    Problem p;
    bool empty;
    const int s = check_shape(stacks[i].batch, stacks[i].rows, stacks[i].cols, &p, &empty);
    if (s != MUON_NS_OK) return s;
    if (!empty) total += make_layout(p).total;
  }
  *bytes = total;
  return MUON_NS_OK;
}

int muon_ns_grouped(const muon_ns_stack* stacks, int num_stacks, int steps, const float* coeffs,
                    float eps, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (num_stacks < 0 || num_stacks > 64 || (num_stacks > 0 && !stacks)) return MUON_NS_ERR_INVALID_ARG;
  float abc[3];
  int s = check_scalars(steps, coeffs, eps, abc);
  if (s != MUON_NS_OK) return s;
  Stack S[64];
  size_t offsets[64];
  int ns = 0;
  size_t off = 0;
  for (int i = 0; i < num_stacks; ++i) {
    Problem p;
    bool empty;
    if ((s = check_shape(stacks[i].batch, stacks[i].rows, stacks[i].cols, &p, &empty)) != MUON_NS_OK)
      return s;
    if (empty) continue;
    if (!stacks[i].G || !stacks[i].out) return MUON_NS_ERR_INVALID_ARG;
    if (!aligned16(stacks[i].G) || !aligned16(stacks[i].out)) return MUON_NS_ERR_ALIGNMENT;
    Stack& t = S[ns];
    t.p = p;
    t.L = make_layout(p);
    t.G = stacks[i].G;
    t.out = stacks[i].out;
    t.ws = nullptr;
    t.cur = nullptr;
    offsets[ns++] = off;
    off += t.L.total;
  }
  if (ns == 0) return MUON_NS_OK;
  if (!workspace || workspace_bytes < off) return MUON_NS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  for (int i = 0; i < ns; ++i) S[i].ws = base + offsets[i];
  int* err = reinterpret_cast<int*>(base + S[0].L.error);
  if (cudaMemsetAsync(base, 0, 256, stream) != cudaSuccess) return MUON_NS_ERR_CUDA;
  return run_ns_stacks(S, ns, steps, abc, eps, err, d.sms, stream);
}

// ------------------------------------------------------- host-held stacks --

}  // extern "C"

namespace {

// Streams and events of the host-buffer path, created once per device: one
// stream for uploads, one for downloads; per slot, the events "input
// uploaded", "chunk computed" and "output downloaded".
// Chunks in flight in a host-path call: each has its own slot of input,
// output and NS workspace, so chunk i's upload waits for chunk
// i - kHostSlots's compute and its compute for that chunk's download.
#ifndef MNS_HOST_SLOTS
#define MNS_HOST_SLOTS 2
#endif
constexpr int kHostSlots = MNS_HOST_SLOTS;

struct HostPipe {
  bool ready;
  cudaStream_t up, down;
  cudaEvent_t start, in[kHostSlots], done[kHostSlots], out[kHostSlots];
};
std::mutex g_pipe_mu;
HostPipe g_pipe[64];

int host_pipe_init(HostPipe* hp) {
  if (hp->ready) return MUON_NS_OK;
  if (cudaStreamCreateWithFlags(&hp->up, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&hp->down, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&hp->start, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    return MUON_NS_ERR_CUDA;
  }
  for (int i = 0; i < kHostSlots; ++i)
    if (cudaEventCreateWithFlags(&hp->in[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp->done[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp->out[i], cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return MUON_NS_ERR_CUDA;
    }
  hp->ready = true;
  return MUON_NS_OK;
}

// Largest chunk of a host-path call.  The default takes about 96 MiB of bf16
// input per chunk, at most half the stack so that copies overlap compute, and
// the whole stack when it holds less than 32 MiB: every chunk pays a whole
// call's chain of launches, which outweighs any overlap for small stacks.
// (Measured on GB300 with stacks of 1 MB to 940 MB, this picks the fastest of
// the swept chunk sizes for each.)
inline int host_chunk(long long batch, long long rows, long long cols, int chunk) {
  if (chunk > 0) return static_cast<int>(chunk < batch ? chunk : batch);
  const long long mat = 2 * rows * cols;
  if (batch * mat < (32LL << 20)) return static_cast<int>(batch);
  const long long by_bytes = ((96LL << 20) + mat - 1) / mat;
  const long long half = (batch + 1) / 2;
  const long long c = by_bytes < half ? by_bytes : half;
  return static_cast<int>(c < 1 ? 1 : c);
}

// Chunk plan of a host-path call with largest chunk c (sizes in matrices,
// in order; every size <= c, the sum is the batch): when the stack spans more
// than one chunk, the first and the last take ceil(c / 2) (shorter copies
// before the first compute and after the last, which nothing overlaps), the
// ones between c, the one before the last the remainder.  (Ends that ramp
// c / 8, c / 4, c / 2 were measured slower on every stack: each extra chunk
// pays a whole call's chain of launches on a GPU it does not fill.)
void host_plan(int batch, int c, std::vector<int>* plan) {
  plan->clear();
  if (batch <= 0) return;
  if (batch <= c) {
    plan->push_back(batch);
    return;
  }
  const int h = (c + 1) / 2;
  const int mid = batch - 2 * h;  // >= 0 since c < batch
  const int nmid = (mid + c - 1) / c;
  plan->push_back(h);
  for (int i = 1; i <= nmid; ++i) plan->push_back(i < nmid ? c : mid - (nmid - 1) * c);
  plan->push_back(h);
}

// Host-path workspace: the call's error word, then two slots of (input
// chunk, output chunk, NS workspace for one chunk).
struct HostLayout {
  size_t in, out, ws, slot, total;
};

HostLayout host_layout(const Problem& pc) {
  HostLayout H;
  const size_t chunk_bytes = 2 * static_cast<size_t>(pc.batch) * pc.R * pc.C;
  H.in = 0;
  H.out = round_up(chunk_bytes, 1024);
  H.ws = H.out + round_up(chunk_bytes, 1024);
  H.slot = round_up(H.ws + make_layout(pc).total, 1024);
  H.total = 1024 + kHostSlots * H.slot;
  return H;
}

}  // namespace

extern "C" {

int muon_ns_host_workspace_size(int batch, int rows, int cols, int chunk, size_t* bytes) {
  if (!bytes) return MUON_NS_ERR_INVALID_ARG;
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  if (empty) {
    *bytes = 0;
    return MUON_NS_OK;
  }
  Problem pc;
  check_shape(host_chunk(batch, rows, cols, chunk), rows, cols, &pc, &empty);
  *bytes = host_layout(pc).total;
  return MUON_NS_OK;
}

int muon_ns_host_chunk(int batch, int rows, int cols, int chunk) {
  Problem p;
  bool empty;
  if (check_shape(batch, rows, cols, &p, &empty) != MUON_NS_OK || empty) return 0;
  return host_chunk(batch, rows, cols, chunk);
}

int muon_ns_host_plan(int batch, int rows, int cols, int chunk, int* sizes, int max_chunks) {
  Problem p;
  bool empty;
  if (check_shape(batch, rows, cols, &p, &empty) != MUON_NS_OK || max_chunks < 0) return -1;
  if (empty) return 0;
  std::vector<int> plan;
  host_plan(batch, host_chunk(batch, rows, cols, chunk), &plan);
  if (sizes != nullptr)
    for (int i = 0; i < static_cast<int>(plan.size()) && i < max_chunks; ++i) sizes[i] = plan[i];
  return static_cast<int>(plan.size());
}

int muon_ns_host(const muon_bf16* G_host, muon_bf16* out_host, int batch, int rows, int cols,
                 int steps, const float* coeffs, float eps, int chunk, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  float abc[3];
  if ((s = check_scalars(steps, coeffs, eps, abc)) != MUON_NS_OK) return s;
  if (empty) return MUON_NS_OK;
  if (!G_host || !out_host) return MUON_NS_ERR_INVALID_ARG;
  const int cb = host_chunk(batch, rows, cols, chunk);
  Problem pc;
  check_shape(cb, rows, cols, &pc, &empty);
  const HostLayout H = host_layout(pc);
  if (!workspace || workspace_bytes < H.total) return MUON_NS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  int dev = 0;
  if ((s = current_device_info(&d, &dev)) != MUON_NS_OK) return s;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe& hp = g_pipe[dev];
  if ((s = host_pipe_init(&hp)) != MUON_NS_OK) return s;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  int* err = reinterpret_cast<int*>(base);
  const size_t mat = static_cast<size_t>(rows) * cols;
  auto fail = [] {
    cudaGetLastError();
    return MUON_NS_ERR_CUDA;
  };
  // The copy streams start after all work already queued on `stream` (so a
  // workspace reused from a previous call is free) and the error word is clear.
  if (cudaMemsetAsync(base, 0, 256, stream) != cudaSuccess ||
      cudaEventRecord(hp.start, stream) != cudaSuccess ||
      cudaStreamWaitEvent(hp.up, hp.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp.down, hp.start, 0) != cudaSuccess)
    return fail();
  std::vector<int> plan;
  host_plan(batch, cb, &plan);
  long long b0 = 0;
  const int nchunks = static_cast<int>(plan.size());
  for (int i = 0; i < nchunks; ++i) {
    const int nb = plan[i];
    const int sl = i % kHostSlots;
    const size_t bytes = 2 * mat * nb;
    uint8_t* slot = base + 1024 + sl * H.slot;
    uint16_t* din = reinterpret_cast<uint16_t*>(slot + H.in);
    uint16_t* dout = reinterpret_cast<uint16_t*>(slot + H.out);
    Problem pi;
    check_shape(nb, rows, cols, &pi, &empty);
    Stack S;
    S.p = pi;
    S.L = make_layout(pi);
    S.G = din;
    S.out = dout;
    S.ws = slot + H.ws;
    S.cur = nullptr;
    // Upload once the slot's previous chunk has finished reading its input;
    // then, on the same stream and so beside the previous chunk's compute,
    // clear this chunk's counters and take its norms (steps > 0), which
    // keeps both off the compute stream.
    if (i >= kHostSlots && cudaStreamWaitEvent(hp.up, hp.done[sl], 0) != cudaSuccess) return fail();
    if (cudaMemcpyAsync(din, G_host + b0 * mat, bytes, cudaMemcpyHostToDevice, hp.up) != cudaSuccess) return fail();
    if (steps > 0) {
      if (cudaMemsetAsync(S.ws + S.L.tickets, 0, 16 * static_cast<size_t>(nb), hp.up) != cudaSuccess) return fail();
      if ((s = run_normalize(pi, S.L, din, nullptr, eps, S.ws, hp.up, false)) != MUON_NS_OK) return s;
    }
    if (cudaEventRecord(hp.in[sl], hp.up) != cudaSuccess) return fail();
    // Compute once the input (and its norms) are ready and the slot's
    // previous output has been downloaded.
    if (cudaStreamWaitEvent(stream, hp.in[sl], 0) != cudaSuccess) return fail();
    if (i >= kHostSlots && cudaStreamWaitEvent(stream, hp.out[sl], 0) != cudaSuccess) return fail();
    if ((s = run_ns_stacks(&S, 1, steps, abc, eps, err, d.sms, stream, steps > 0, steps > 0)) != MUON_NS_OK)
      return s;
    if (cudaEventRecord(hp.done[sl], stream) != cudaSuccess) return fail();
    // Download once computed.
    if (cudaStreamWaitEvent(hp.down, hp.done[sl], 0) != cudaSuccess ||
        cudaMemcpyAsync(out_host + b0 * mat, dout, bytes, cudaMemcpyDeviceToHost, hp.down) != cudaSuccess ||
        cudaEventRecord(hp.out[sl], hp.down) != cudaSuccess)
      return fail();
    b0 += nb;
  }
  // `stream` completes after the last downloads.
  for (int sl = 0; sl < kHostSlots && sl < nchunks; ++sl)
    if (cudaStreamWaitEvent(stream, hp.out[sl], 0) != cudaSuccess) return fail();
  return MUON_NS_OK;
}

int muon_ns_read_error(const void* workspace, int* device_error, int clear, cudaStream_t stream) {
  if (!workspace || !device_error) return MUON_NS_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return MUON_NS_ERR_CUDA;
  }
  int v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MUON_NS_ERR_CUDA;
  }
  if (clear && v != 0 &&
      cudaMemset(const_cast<void*>(workspace), 0, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return MUON_NS_ERR_CUDA;
  }
  *device_error = v;
  return v ? MUON_NS_ERR_TIMEOUT : MUON_NS_OK;
}

int muon_ns_check(const void* workspace, int* host_word, cudaStream_t stream) {
  if (!workspace || !host_word) return MUON_NS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_NS_ERR_ALIGNMENT;
  // The word must be memory the copy engine writes without staging
  // (page-locked or registered host memory, or managed memory): a pageable
  // destination would make the copy synchronous and cannot be captured.
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host_word) != cudaSuccess) {
    cudaGetLastError();
    return MUON_NS_ERR_INVALID_ARG;
  }
  if (a.type != cudaMemoryTypeHost && a.type != cudaMemoryTypeManaged) return MUON_NS_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(host_word, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess) {
    cudaGetLastError();
    return MUON_NS_ERR_CUDA;
  }
  return MUON_NS_OK;
}

int muon_ns_cached_error(int device, int* device_error) {
  if (!device_error || device < 0 || device >= 64) return MUON_NS_ERR_INVALID_ARG;
  void* ptr;
  {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    ptr = g_cache[device].ptr;
  }
  *device_error = 0;
  if (!ptr) return MUON_NS_OK;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return MUON_NS_ERR_CUDA;
  }
  const int s = muon_ns_read_error(ptr, device_error, 0, nullptr);
  cudaSetDevice(prev);
  return s;
}

int muon_ns_set_wait_budget(long long cycles) {
  if (cycles < 0) return MUON_NS_ERR_INVALID_ARG;
  g_wait_budget.store(cycles);
  return MUON_NS_OK;
}

int muon_ns_inject_stall(int enable) {
  g_inject_stall.store(enable != 0 ? 1 : 0);
  return MUON_NS_OK;
}

int muon_ns_normalize(const muon_bf16* G, muon_bf16* X, int batch, int rows, int cols, float eps,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return MUON_NS_ERR_INVALID_ARG;
  if (empty) return MUON_NS_OK;
  if (!G) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(G) || !aligned16(X)) return MUON_NS_ERR_ALIGNMENT;
  const Layout L = make_layout(p);
  if (!workspace || workspace_bytes < L.total) return MUON_NS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  return run_normalize(p, L, G, X, eps, static_cast<uint8_t*>(workspace), stream);
}

int muon_ns_gram_ex(const muon_bf16* X, muon_bf16* A, int batch, int rows, int cols, const float* norms,
                    float eps, int flags, int* device_error, cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  if (flags & ~MUON_NS_HALF) return MUON_NS_ERR_INVALID_ARG;
  if (empty) return MUON_NS_OK;
  if (!X || !A) return MUON_NS_ERR_INVALID_ARG;
  if (norms && (!(eps >= 0.0f) || !std::isfinite(eps))) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(A)) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  StepIO io = {};
  io.p = p;
  io.X = X;
  io.A = A;
  io.norms = norms;
  io.half = (flags & MUON_NS_HALF) != 0;
  return run_gram(&io, 1, eps, device_error, d.sms, stream);
}

int muon_ns_gram(const muon_bf16* X, muon_bf16* A, int batch, int rows, int cols,
                 const float* norms, float eps, int* device_error, cudaStream_t stream) {
  return muon_ns_gram_ex(X, A, batch, rows, cols, norms, eps, 0, device_error, stream);
}

int muon_ns_poly_ex(const muon_bf16* A, muon_bf16* B, float* diag, int batch, int m, float b, float c,
                    int flags, int* device_error, cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, m, m, &p, &empty);
  if (s != MUON_NS_OK) return s;
  if (!std::isfinite(b) || !std::isfinite(c) || (flags & ~MUON_NS_HALF)) return MUON_NS_ERR_INVALID_ARG;
  if (empty) return MUON_NS_OK;
  if (!A || !B || A == B) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(diag)) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  StepIO io = {};
  io.p = p;
  io.A = const_cast<uint16_t*>(A);
  io.B = B;
  io.D = diag;
  io.half = (flags & MUON_NS_HALF) != 0;
  return run_poly(&io, 1, b, c, device_error, d.sms, stream);
}

int muon_ns_poly(const muon_bf16* A, muon_bf16* B, float* diag, int batch, int m, float b,
                 float c, int* device_error, cudaStream_t stream) {
  return muon_ns_poly_ex(A, B, diag, batch, m, b, c, 0, device_error, stream);
}

int muon_ns_update_ex(const muon_bf16* X, const muon_bf16* B, const float* diag, muon_bf16* Xn, int batch,
                      int rows, int cols, float a, const float* norms, float eps, int flags, int* device_error,
                      cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  if (!std::isfinite(a) || (flags & ~MUON_NS_HALF)) return MUON_NS_ERR_INVALID_ARG;
  if (norms && (!(eps >= 0.0f) || !std::isfinite(eps))) return MUON_NS_ERR_INVALID_ARG;
  if (empty) return MUON_NS_OK;
  if (!X || !B || !Xn || Xn == X || Xn == B) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(B) || !aligned16(Xn) || !aligned16(diag))
    return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  StepIO io = {};
  io.p = p;
  io.X = X;
  io.B = const_cast<uint16_t*>(B);
  io.D = const_cast<float*>(diag);
  io.norms = norms;
  io.Xn = Xn;
  io.half = (flags & MUON_NS_HALF) != 0;
  return run_update(&io, 1, a, eps, false, device_error, d.sms, stream);
}

int muon_ns_update(const muon_bf16* X, const muon_bf16* B, const float* diag, muon_bf16* Xn,
                   int batch, int rows, int cols, float a, const float* norms, float eps,
                   int* device_error, cudaStream_t stream) {
  return muon_ns_update_ex(X, B, diag, Xn, batch, rows, cols, a, norms, eps, 0, device_error, stream);
}

}  // extern "C"

// ------------------------------------------------------------- Muon step --

namespace {

// decay = 1 - lr wd and lrs = lr scale, in fp32, from finite hyperparameters.
int check_hparams(const muon_step_hparams* hp, float* decay, float* lrs) {
  if (!hp) return MUON_NS_ERR_INVALID_ARG;
  if (!std::isfinite(hp->lr) || !std::isfinite(hp->momentum) || !std::isfinite(hp->weight_decay) ||
      !std::isfinite(hp->scale))
    return MUON_NS_ERR_INVALID_ARG;
  *decay = 1.0f - hp->lr * hp->weight_decay;
  *lrs = hp->lr * hp->scale;
  return MUON_NS_OK;
}

// A Muon-step workspace is the NS workspace of the stack followed by the
// bf16 NS input U [batch][rows][cols].
size_t step_u_offset(const Layout& L) { return round_up(L.total, 1024); }
size_t step_ws_total(const Problem& p, const Layout& L) {
  return step_u_offset(L) + round_up(2 * static_cast<size_t>(p.batch) * p.R * p.C, 1024);
}

// The momentum kernel over the stack; tickets must be zero (it writes the
// norms of U into the workspace's norm region).
int launch_momentum(const Problem& p, const Layout& L, const float* G, float* M, uint16_t* U, float mu,
                    int nesterov, uint8_t* ws, cudaStream_t st) {
  const long long vec = p.R * p.C / 8;
  return to_status(mns::launch_pdl(mns::muon_momentum_norm, batch_grid(L.chunks, p.batch), dim3(mns::kNormThreads), 0,
                                   st, reinterpret_cast<const float4*>(G), reinterpret_cast<float4*>(M),
                                   reinterpret_cast<uint4*>(U), vec, L.chunks, static_cast<int>(p.batch), mu,
                                   nesterov ? 1 : 0,
                                   reinterpret_cast<float*>(ws + L.partials),
                                   reinterpret_cast<unsigned int*>(ws + L.tickets),
                                   reinterpret_cast<float*>(ws + L.norms)));
}

// W = decay W - lrs O over n elements (a multiple of 8), grid-stride with at
// most 8 CTAs of 256 threads per SM.
int launch_apply(float* W, const uint16_t* O, long long n, float decay, float lrs, int sms, cudaStream_t st) {
  const long long n8 = n / 8;
  const long long want = (n8 + 255) / 256;
  const long long cap = 8LL * sms;
  const unsigned blocks = static_cast<unsigned>(std::max(1LL, std::min(want, cap)));
  return to_status(mns::launch_pdl(mns::muon_apply, dim3(blocks), dim3(256), 0, st, reinterpret_cast<float4*>(W),
                                   reinterpret_cast<const uint4*>(O), n8, decay, lrs));
}

bool overlap(const void* a, const void* b, size_t bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bytes && y < x + bytes;
}

}  // namespace

extern "C" {

int muon_step_workspace_size(int batch, int rows, int cols, size_t* bytes) {
  if (!bytes) return MUON_NS_ERR_INVALID_ARG;
  Problem p;
  bool empty;
  const int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  *bytes = empty ? 0 : step_ws_total(p, make_layout(p));
  return MUON_NS_OK;
}

int muon_step_ws(float* W, float* M, const float* G, int batch, int rows, int cols,
                 const muon_step_hparams* hp, int steps, const float* coeffs, float eps, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  float abc[3], decay, lrs;
  if ((s = check_scalars(steps, coeffs, eps, abc)) != MUON_NS_OK) return s;
  if ((s = check_hparams(hp, &decay, &lrs)) != MUON_NS_OK) return s;
  if (empty) return MUON_NS_OK;
  if (!W || !M || !G) return MUON_NS_ERR_INVALID_ARG;
  const size_t fbytes = 4 * static_cast<size_t>(p.batch) * p.R * p.C;
  if (overlap(W, M, fbytes) || overlap(W, G, fbytes) || overlap(M, G, fbytes)) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(M) || !aligned16(G)) return MUON_NS_ERR_ALIGNMENT;
  const Layout L = make_layout(p);
  if (!workspace || workspace_bytes < step_ws_total(p, L)) return MUON_NS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* U = reinterpret_cast<uint16_t*>(ws + step_u_offset(L));
  // Error word, norm tickets and dependency counters in one memset.
  if (cudaMemsetAsync(ws, 0, L.deps + 12 * static_cast<size_t>(p.batch), stream) != cudaSuccess)
    return MUON_NS_ERR_CUDA;
  if ((s = launch_momentum(p, L, G, M, U, hp->momentum, hp->nesterov, ws, stream)) != MUON_NS_OK) return s;
  if (steps == 0) {
    // O = U / (||U||_F + eps) into the iterate region, then the update.
    uint16_t* O = reinterpret_cast<uint16_t*>(ws + L.x);
    if (mns::launch_pdl(mns::ns_scale<false>, batch_grid(L.chunks, p.batch), dim3(mns::kNormThreads), 0, stream,
                        reinterpret_cast<const uint4*>(U), reinterpret_cast<uint4*>(O), p.R * p.C / 8,
                        static_cast<int>(p.batch), reinterpret_cast<const float*>(ws + L.norms), eps) != cudaSuccess)
      return MUON_NS_ERR_CUDA;
    return launch_apply(W, O, p.batch * p.R * p.C, decay, lrs, d.sms, stream);
  }
  Stack S;
  S.p = p;
  S.L = L;
  S.G = U;
  S.out = U;  // in place: U is dead once step 1 has read it
  S.ws = ws;
  S.cur = nullptr;
  S.W = W;
  S.w_decay = decay;
  S.w_lrs = lrs;
  return run_ns_stacks(&S, 1, steps, abc, eps, reinterpret_cast<int*>(ws + L.error), d.sms, stream, true, true);
}

namespace {

// One stack of a grouped Muon step, checked: its shape, scalars and layout.
struct StepStack {
  Problem p;
  Layout L;
  float decay, lrs;
  size_t offset;  // of this stack's step workspace in the call's workspace
};

int check_step_stacks(const muon_step_stack* stacks, int num_stacks, StepStack* out, int* n_out, size_t* bytes) {
  if (num_stacks < 0 || num_stacks > 64 || (num_stacks > 0 && !stacks)) return MUON_NS_ERR_INVALID_ARG;
  int n = 0;
  size_t off = 0;
  for (int i = 0; i < num_stacks; ++i) {
    const muon_step_stack& st = stacks[i];
    StepStack& t = out[n];
    bool empty;
    int s = check_shape(st.batch, st.rows, st.cols, &t.p, &empty);
    if (s != MUON_NS_OK) return s;
    if ((s = check_hparams(&st.hp, &t.decay, &t.lrs)) != MUON_NS_OK) return s;
    if (empty) continue;
    if (!st.W || !st.M || !st.G) return MUON_NS_ERR_INVALID_ARG;
    if (!aligned16(st.W) || !aligned16(st.M) || !aligned16(st.G)) return MUON_NS_ERR_ALIGNMENT;
    t.L = make_layout(t.p);
    t.offset = off;
    off += step_ws_total(t.p, t.L);
    ++n;
  }
  // W and M are written: neither may overlap any stack's W, M or G (its own
  // W and M excepted, which are the same buffer).
  auto range = [&](int i, int a, uintptr_t* lo, uintptr_t* hi) {
    const void* ptr[3] = {stacks[i].W, stacks[i].M, stacks[i].G};
    *lo = reinterpret_cast<uintptr_t>(ptr[a]);
    *hi = *lo + 4 * static_cast<size_t>(stacks[i].batch) * stacks[i].rows * stacks[i].cols;
  };
  for (int i = 0; i < num_stacks; ++i) {
    for (int a = 0; a < 2; ++a) {
      uintptr_t lo, hi;
      range(i, a, &lo, &hi);
      if (lo == hi) continue;
      for (int j = 0; j < num_stacks; ++j) {
        for (int c = 0; c < 3; ++c) {
          if (i == j && a == c) continue;
          uintptr_t lo2, hi2;
          range(j, c, &lo2, &hi2);
          if (lo2 != hi2 && lo < hi2 && lo2 < hi) return MUON_NS_ERR_INVALID_ARG;
        }
      }
    }
  }
  *n_out = n;
  *bytes = off;
  return MUON_NS_OK;
}

}  // namespace

int muon_step_grouped_workspace_size(const muon_step_stack* stacks, int num_stacks, size_t* bytes) {
  if (!bytes) return MUON_NS_ERR_INVALID_ARG;
  StepStack S[64];
  int n = 0;
  return check_step_stacks(stacks, num_stacks, S, &n, bytes);
}

int muon_step_grouped(const muon_step_stack* stacks, int num_stacks, int steps, const float* coeffs, float eps,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  float abc[3];
  int s = check_scalars(steps, coeffs, eps, abc);
  if (s != MUON_NS_OK) return s;
  StepStack T[64];
  int n = 0;
  size_t need = 0;
  if ((s = check_step_stacks(stacks, num_stacks, T, &n, &need)) != MUON_NS_OK) return s;
  if (n == 0) return MUON_NS_OK;
  if (!workspace || workspace_bytes < need) return MUON_NS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  Stack S[64];
  int k = 0;
  for (int i = 0; i < num_stacks; ++i) {
    const muon_step_stack& st = stacks[i];
    if (st.batch == 0 || st.rows == 0 || st.cols == 0) continue;
    const StepStack& t = T[k];
    uint8_t* ws = base + t.offset;
    uint16_t* U = reinterpret_cast<uint16_t*>(ws + step_u_offset(t.L));
    // This stack's error word, tickets and counters in one memset.
    if (cudaMemsetAsync(ws, 0, t.L.deps + 12 * static_cast<size_t>(t.p.batch), stream) != cudaSuccess)
      return MUON_NS_ERR_CUDA;
    if ((s = launch_momentum(t.p, t.L, st.G, st.M, U, st.hp.momentum, st.hp.nesterov, ws, stream)) != MUON_NS_OK)
      return s;
    if (steps == 0) {
      uint16_t* O = reinterpret_cast<uint16_t*>(ws + t.L.x);
      if (mns::launch_pdl(mns::ns_scale<false>, batch_grid(t.L.chunks, t.p.batch), dim3(mns::kNormThreads), 0,
                          stream, reinterpret_cast<const uint4*>(U), reinterpret_cast<uint4*>(O), t.p.R * t.p.C / 8,
                          static_cast<int>(t.p.batch), reinterpret_cast<const float*>(ws + t.L.norms),
                          eps) != cudaSuccess)
        return MUON_NS_ERR_CUDA;
      if ((s = launch_apply(st.W, O, t.p.batch * t.p.R * t.p.C, t.decay, t.lrs, d.sms, stream)) != MUON_NS_OK)
        return s;
    }
    Stack& q = S[k];
    q.p = t.p;
    q.L = t.L;
    q.G = U;
    q.out = U;
    q.ws = ws;
    q.cur = nullptr;
    q.W = st.W;
    q.w_decay = t.decay;
    q.w_lrs = t.lrs;
    ++k;
  }
  if (steps == 0) return MUON_NS_OK;
  // Every kernel reports to the first stack's error word.
  return run_ns_stacks(S, k, steps, abc, eps, reinterpret_cast<int*>(base + T[0].offset + T[0].L.error), d.sms,
                       stream, true, true);
}

int muon_momentum(float* M, const float* G, muon_bf16* U, int batch, int rows, int cols, float momentum,
                  int nesterov, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  if (!std::isfinite(momentum)) return MUON_NS_ERR_INVALID_ARG;
  if (empty) return MUON_NS_OK;
  if (!M || !G || !U) return MUON_NS_ERR_INVALID_ARG;
  if (overlap(M, G, 4 * static_cast<size_t>(p.batch) * p.R * p.C)) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(M) || !aligned16(G) || !aligned16(U)) return MUON_NS_ERR_ALIGNMENT;
  const Layout L = make_layout(p);
  if (!workspace || workspace_bytes < L.total) return MUON_NS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (cudaMemsetAsync(ws + L.tickets, 0, 4 * static_cast<size_t>(p.batch), stream) != cudaSuccess)
    return MUON_NS_ERR_CUDA;
  return launch_momentum(p, L, G, M, U, momentum, nesterov, ws, stream);
}

int muon_apply(float* W, const muon_bf16* O, int batch, int rows, int cols, const muon_step_hparams* hp,
               cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  float decay, lrs;
  if ((s = check_hparams(hp, &decay, &lrs)) != MUON_NS_OK) return s;
  if (empty) return MUON_NS_OK;
  if (!W || !O) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(O)) return MUON_NS_ERR_ALIGNMENT;
  DevInfo d;
  if ((s = current_device_info(&d)) != MUON_NS_OK) return s;
  return launch_apply(W, O, p.batch * p.R * p.C, decay, lrs, d.sms, stream);
}

int muon_step_launches(int steps) { return steps < 0 ? -1 : (steps == 0 ? 3 : 1 + 3 * steps); }

int muon_ns_launches_per_call(int steps) {
  return steps < 0 ? -1 : (steps == 0 ? 2 : 1 + 3 * steps);
}

long long muon_ns_tile_count(int kind, int batch, int M, int N) {
  if (kind < 0 || kind > 3 || batch < 0 || M < 0 || N < 0) return -1;
  if ((kind & 1) == 0 && M != N) return -1;
  return mns::make_tile_space((kind & 1) == 0 ? 1 : 0, batch, M, N, kind >> 1).total;
}

int muon_ns_tile_coords(int kind, int batch, int M, int N, long long tile, int* matrix,
                        int* row_tile, int* col_tile) {
  if (!matrix || !row_tile || !col_tile) return MUON_NS_ERR_INVALID_ARG;
  const long long total = muon_ns_tile_count(kind, batch, M, N);
  if (total < 0 || tile < 0 || tile >= total) return MUON_NS_ERR_INVALID_ARG;
  const mns::TileSpace sp = mns::make_tile_space((kind & 1) == 0 ? 1 : 0, batch, M, N, kind >> 1);
  mns::tile_decode(sp, tile, matrix, row_tile, col_tile);
  return MUON_NS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Normalisation without any allocation.
//
// Some callers cannot allocate device memory: a plugin that a host program
// hands only its input and output buffers, a framework whose caching
// allocator owns all device memory and forbids direct cudaMalloc, or a
// latency-bound loop that cannot afford cudaMalloc's implicit device
// synchronisation.  muon_ns_normalize_static() serves them: the norm kernel's
// scratch (per-matrix tickets, per-chunk partial sums and the norms) lives in
// the fixed array below, which every GPU that loads this library holds until
// the process exits.
// ---------------------------------------------------------------------------

namespace {
constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB
std::mutex g_static_mu;
void* g_static_addr[64];
}  // namespace

static __device__ __align__(256) unsigned char g_ns_static_scratch[kStaticScratchBytes];

namespace {

// Device address of the static scratch on the current device `dev`, looked up
// once per device (the array's name is only a host-side stand-in in host code).
int static_scratch_address(int dev, uint8_t** out) {
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_ns_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MUON_NS_ERR_CUDA;
    }
    g_static_addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_static_addr[dev]);
  return MUON_NS_OK;
}

}  // namespace

extern "C" int muon_ns_normalize_static(const muon_bf16* G, muon_bf16* X, int batch, int rows,
                                        int cols, float eps, cudaStream_t stream) {
  Problem p;
  bool empty;
  int s = check_shape(batch, rows, cols, &p, &empty);
  if (s != MUON_NS_OK) return s;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return MUON_NS_ERR_INVALID_ARG;
  if (empty) return MUON_NS_OK;
  if (!G || !X) return MUON_NS_ERR_INVALID_ARG;
  if (!aligned16(G) || !aligned16(X)) return MUON_NS_ERR_ALIGNMENT;
  // Scratch layout inside the static array: tickets, partial sums, norms.
  Layout L = make_layout(p);
  L.error = 0;
  L.tickets = 0;
  L.partials = round_up(4 * static_cast<size_t>(p.batch), 256);
  L.norms = round_up(L.partials + 4 * static_cast<size_t>(p.batch) * L.chunks, 256);
  if (L.norms + 4 * static_cast<size_t>(p.batch) > kStaticScratchBytes) return MUON_NS_ERR_WORKSPACE;
  DevInfo d;
  int dev = 0;
  if ((s = current_device_info(&d, &dev)) != MUON_NS_OK) return s;
  uint8_t* scratch = nullptr;
  if ((s = static_scratch_address(dev, &scratch)) != MUON_NS_OK) return s;
  // The tickets are zeroed by run_normalize on `stream`; partials and norms
  // are overwritten.
  return run_normalize(p, L, G, X, eps, scratch, stream);
}
