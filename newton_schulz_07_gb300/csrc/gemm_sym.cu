// Instantiations of the tensor-core kernel for the symmetric products
// (Gram X X^T or Y^T Y, and b A + c A A).
#include "gemm_launch.cuh"

namespace mns {

constexpr bool kSymPairs = kClusterSym == 2;

cudaError_t launch_sym_kk(const GemmParams& p, int max_k, int grid, cudaStream_t stream) {
  return (kSymPairs && max_k >= kPairMmaMinK)
             ? launch_tc_gemm<false, false, true, 8, false, kClusterSym, kSymPairs>(p, grid, stream)
             : launch_tc_gemm<false, false, true, 8, false, kClusterSym, false>(p, grid, stream);
}

cudaError_t launch_sym_mnmn(const GemmParams& p, int max_k, int grid, cudaStream_t stream) {
  return (kSymPairs && max_k >= kPairMmaMinK)
             ? launch_tc_gemm<true, true, true, 8, false, kClusterSym, kSymPairs>(p, grid, stream)
             : launch_tc_gemm<true, true, true, 8, false, kClusterSym, false>(p, grid, stream);
}

}  // namespace mns
