// Internal interface between the C-ABI host code and the kernel translation
// units (one per group of tensor-core kernel instantiations, built in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "tile_sched.h"

namespace mns {

struct GemmParams;

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
