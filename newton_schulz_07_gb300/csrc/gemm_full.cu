// Instantiations of the tensor-core kernel for the update products
// (a X + B X, and a Y + Y B for inputs kept in their tall orientation).
#include "gemm_launch.cuh"

namespace mns {

cudaError_t launch_full_kmn(const GemmParams& p, int max_k, int grid, cudaStream_t stream) {
  return max_k <= 1024 ? launch_tc_gemm<false, true, false, 8, false, kClusterFull>(p, grid, stream)
                       : launch_tc_gemm<false, true, false, 4, false, kClusterFull>(p, grid, stream);
}

cudaError_t launch_full_kk(const GemmParams& p, int max_k, int grid, cudaStream_t stream) {
  return max_k <= 1024 ? launch_tc_gemm<false, false, false, 8, false, kClusterFull>(p, grid, stream)
                       : launch_tc_gemm<false, false, false, 4, false, kClusterFull>(p, grid, stream);
}

}  // namespace mns
