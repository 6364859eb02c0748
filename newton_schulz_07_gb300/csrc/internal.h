// Internal interface between the C-ABI host code and the kernel translation
// units (one per group of tensor-core kernel instantiations, built in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "tile_sched.h"

namespace mns {

struct GemmParams;

// How a product launch pairs its CTAs.  The host builds the tile space and
// the B-operand tensor maps from the mode, and the launcher instantiates the
// kernel for it.
enum PairMode : int {
  kSingle = 0,     // one CTA per 128 x 256 tile
  kMulticast = 1,  // clusters of two CTAs (row tiles 2p, 2p + 1) sharing a multicast B panel
  kPairMma = 2,    // clusters of two CTAs running 2-SM MMAs (M = 256)
};

// 2-SM MMAs for contractions longer than 1024; shorter ones leave the
// epilogue as long as the main loop, and a 2-SM pair must wait for both
// CTAs' epilogues before reusing an accumulator (measured on GB300: K = 768
// bf16 products 3-8 % slower with 2-SM MMAs, K >= 1536 products 2-11 %
// faster).  Short bf16 products use multicast pairs; short fp32 products run
// single CTAs (multicast pairs measured slightly slower for them).
// MNS_PAIR_MMA=0 turns 2-SM MMAs off.
#ifndef MNS_PAIR_MMA
#define MNS_PAIR_MMA 1
#endif
constexpr int kShortK = 1024;  // contractions up to this are "short"
inline PairMode pair_mode(bool f32, int max_k) {
  if (MNS_PAIR_MMA && max_k > kShortK) return kPairMma;
  return f32 ? kSingle : kMulticast;
}

// Epilogue warps of a bf16 update launch: 8 for short contractions on
// multicast pairs, 4 otherwise.  The 4-warp bf16 update writes its output in
// 32 x 64 boxes (128-byte rows, 128-byte swizzle); every other product writes
// 32 x 32 chunks.  The launcher instantiates, and the host builds the output
// tensor map, from this one function.
inline int update_epi_warps(PairMode mode, int max_k) {
  return (mode != kPairMma && max_k <= kShortK) ? 8 : 4;
}

// `max_k` is the largest contraction of the launch's groups: short
// contractions use 8 epilogue warps in the update.
// Gram / polynomial products: lower-triangle tiles, mirrored stores.
cudaError_t launch_sym_kk(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream);    // K-major operands
cudaError_t launch_sym_mnmn(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream);  // MN-major operands
// Update products: full output grid.
cudaError_t launch_full_kmn(const GemmParams& p, PairMode mode, int max_k, int grid, cudaStream_t stream);
cudaError_t launch_full_kk(const GemmParams& p, PairMode mode, int max_k, int grid, cudaStream_t stream);

// The last update of a Muon step (GroupArgs::w_out): bf16 update products
// whose epilogue writes the fp32 master weights; always 4 epilogue warps.
// The factors are GemmParams::w_decay / w_lrs for every group, or with
// `per_group` each group's GemmParams::w_decay_g / w_lrs_g.
cudaError_t launch_full_kmn_w(const GemmParams& p, PairMode mode, int grid, bool per_group, cudaStream_t stream);
cudaError_t launch_full_kk_w(const GemmParams& p, PairMode mode, int grid, bool per_group, cudaStream_t stream);
// The per-group instantiations (gemm_wout_grp.cu).
cudaError_t launch_full_kmn_wg(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream);
cudaError_t launch_full_kk_wg(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream);

// The same for fp32 operands and outputs (tf32 tensor cores).
cudaError_t launch_sym_kk_f32(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream);
cudaError_t launch_sym_mnmn_f32(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream);
cudaError_t launch_full_kmn_f32(const GemmParams& p, PairMode mode, int max_k, int grid, cudaStream_t stream);
cudaError_t launch_full_kk_f32(const GemmParams& p, PairMode mode, int max_k, int grid, cudaStream_t stream);

}  // namespace mns
