// Internal interface between the C-ABI host code and the kernel translation
// units (one per group of tensor-core kernel instantiations, built in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "tile_sched.h"

namespace mns {

struct GemmArgs;

// Tensor maps: a, b = operands; o = output (32 x 32 boxes, 64-byte swizzle).
// Gram / polynomial products: lower-triangle tiles, mirrored stores.
cudaError_t launch_sym_kk(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                          const GemmArgs& args,
                          int grid, cudaStream_t stream);  // both operands K-major
cudaError_t launch_sym_mnmn(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                          const GemmArgs& args,
                            int grid, cudaStream_t stream);  // both operands MN-major
// Update products: full output grid.
cudaError_t launch_full_kmn(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                          const GemmArgs& args,
                            int grid, cudaStream_t stream);  // B operand MN-major
cudaError_t launch_full_kk(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o,
                          const GemmArgs& args,
                           int grid, cudaStream_t stream);  // both operands K-major

}  // namespace mns
