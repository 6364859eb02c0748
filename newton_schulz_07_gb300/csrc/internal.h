// Internal interface between the C-ABI host code and the kernel translation
// units (one per group of tensor-core kernel instantiations, built in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "tile_sched.h"

namespace mns {

struct GemmParams;

// CTAs per cluster of the bf16 products (1, or 2 for pairs of row tiles that
// share their B-operand panel through TMA multicast).  The host builds the
// tile spaces and the B-operand tensor maps to match.  The fp32 products run
// without clusters.
#ifndef MNS_CLUSTER_SYM
#define MNS_CLUSTER_SYM 2
#endif
#ifndef MNS_CLUSTER_FULL
#define MNS_CLUSTER_FULL 2
#endif
// bf16 pairs run 2-SM MMAs when the launch's longest contraction exceeds
// kPairMmaMinK - 1, and single-CTA MMAs on a multicast B panel otherwise:
// short contractions leave the epilogue as long as the main loop, and a 2-SM
// pair must wait for both CTAs' epilogues before reusing an accumulator
// (measured on GB300: K = 768 products 3-8 % slower with 2-SM MMAs, K >= 1536
// products 2-11 % faster).  MNS_PAIR_MMA=0 disables 2-SM MMAs.
#ifndef MNS_PAIR_MMA
#define MNS_PAIR_MMA 1
#endif
constexpr int kClusterSym = MNS_CLUSTER_SYM;
constexpr int kClusterFull = MNS_CLUSTER_FULL;
constexpr int kPairMmaMinK = MNS_PAIR_MMA ? 1025 : 0x7FFFFFFF;

// `max_k` is the largest contraction of the launch's groups: short
// contractions use 8 epilogue warps in the update and no 2-SM MMAs.
// Gram / polynomial products: lower-triangle tiles, mirrored stores.
cudaError_t launch_sym_kk(const GemmParams& p, int max_k, int grid, cudaStream_t stream);    // K-major operands
cudaError_t launch_sym_mnmn(const GemmParams& p, int max_k, int grid, cudaStream_t stream);  // MN-major operands
// Update products: full output grid.
cudaError_t launch_full_kmn(const GemmParams& p, int max_k, int grid, cudaStream_t stream);
cudaError_t launch_full_kk(const GemmParams& p, int max_k, int grid, cudaStream_t stream);

// The same for fp32 operands and outputs (tf32 tensor cores).
cudaError_t launch_sym_kk_f32(const GemmParams& p, int grid, cudaStream_t stream);
cudaError_t launch_sym_mnmn_f32(const GemmParams& p, int grid, cudaStream_t stream);
cudaError_t launch_full_kmn_f32(const GemmParams& p, int max_k, int grid, cudaStream_t stream);
cudaError_t launch_full_kk_f32(const GemmParams& p, int max_k, int grid, cudaStream_t stream);

}  // namespace mns
