// Instantiations of the tensor-core kernel for the symmetric products
// (Gram X X^T or Y^T Y, and b A + c A A).
#include "gemm_launch.cuh"

namespace mns {

cudaError_t launch_sym_kk(const GemmParams& p, int grid, cudaStream_t stream) {
  return launch_tc_gemm<false, false, true, 8, false, kClusterSym>(p, grid, stream);
}

cudaError_t launch_sym_mnmn(const GemmParams& p, int grid, cudaStream_t stream) {
  return launch_tc_gemm<true, true, true, 8, false, kClusterSym>(p, grid, stream);
}

}  // namespace mns
