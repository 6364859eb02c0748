// Instantiations of the tensor-core kernel for the update products
// (a X + B X, and a Y + Y B for inputs kept in their tall orientation).
#include "gemm_launch.cuh"

namespace mns {

constexpr bool kFullPairs = kClusterFull == 2;

// Short contractions: 8 epilogue warps, no 2-SM MMAs; long ones: 4 epilogue
// warps, 2-SM MMAs for CTA pairs.
cudaError_t launch_full_kmn(const GemmParams& p, int max_k, int grid, cudaStream_t stream) {
  if (max_k <= 1024) return launch_tc_gemm<false, true, false, 8, false, kClusterFull, false>(p, grid, stream);
  return max_k >= kPairMmaMinK
             ? launch_tc_gemm<false, true, false, 4, false, kClusterFull, kFullPairs>(p, grid, stream)
             : launch_tc_gemm<false, true, false, 4, false, kClusterFull, false>(p, grid, stream);
}

cudaError_t launch_full_kk(const GemmParams& p, int max_k, int grid, cudaStream_t stream) {
  if (max_k <= 1024) return launch_tc_gemm<false, false, false, 8, false, kClusterFull, false>(p, grid, stream);
  return max_k >= kPairMmaMinK
             ? launch_tc_gemm<false, false, false, 4, false, kClusterFull, kFullPairs>(p, grid, stream)
             : launch_tc_gemm<false, false, false, 4, false, kClusterFull, false>(p, grid, stream);
}

}  // namespace mns
