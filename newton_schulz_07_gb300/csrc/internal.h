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
constexpr int kClusterSym = MNS_CLUSTER_SYM;
constexpr int kClusterFull = MNS_CLUSTER_FULL;

// Gram / polynomial products: lower-triangle tiles, mirrored stores.
cudaError_t launch_sym_kk(const GemmParams& p, int grid, cudaStream_t stream);    // K-major operands
cudaError_t launch_sym_mnmn(const GemmParams& p, int grid, cudaStream_t stream);  // MN-major operands
// Update products: full output grid.  `max_k` is the largest contraction of
// the launch's groups (short contractions use 8 epilogue warps).
cudaError_t launch_full_kmn(const GemmParams& p, int max_k, int grid, cudaStream_t stream);
cudaError_t launch_full_kk(const GemmParams& p, int max_k, int grid, cudaStream_t stream);

// The same for fp32 operands and outputs (tf32 tensor cores).
cudaError_t launch_sym_kk_f32(const GemmParams& p, int grid, cudaStream_t stream);
cudaError_t launch_sym_mnmn_f32(const GemmParams& p, int grid, cudaStream_t stream);
cudaError_t launch_full_kmn_f32(const GemmParams& p, int max_k, int grid, cudaStream_t stream);
cudaError_t launch_full_kk_f32(const GemmParams& p, int max_k, int grid, cudaStream_t stream);

}  // namespace mns
