// Instantiations of the tensor-core kernel for the symmetric products
// (Gram X X^T or Y^T Y, and b A + c A A).
#include "gemm_launch.cuh"

namespace mns {

cudaError_t launch_sym_kk(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o, const GemmArgs& args,
                          int grid, cudaStream_t stream) {
  return launch_tc_gemm<false, false, true, 8>(a, b, o, args, grid, stream);
}

cudaError_t launch_sym_mnmn(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o, const GemmArgs& args,
                            int grid, cudaStream_t stream) {
  return launch_tc_gemm<true, true, true, 8>(a, b, o, args, grid, stream);
}

}  // namespace mns
