// Instantiations of the tensor-core kernel for the update products
// (a X + B X, and a Y + Y B for inputs kept in their tall orientation).
#include "gemm_launch.cuh"

namespace mns {

cudaError_t launch_full_kmn(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o, const GemmArgs& args,
                            int grid, cudaStream_t stream) {
  return args.K <= 1024 ? launch_tc_gemm<false, true, false, 8>(a, b, o, args, grid, stream)
                        : launch_tc_gemm<false, true, false, 4>(a, b, o, args, grid, stream);
}

cudaError_t launch_full_kk(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o, const GemmArgs& args,
                           int grid, cudaStream_t stream) {
  return args.K <= 1024 ? launch_tc_gemm<false, false, false, 8>(a, b, o, args, grid, stream)
                        : launch_tc_gemm<false, false, false, 4>(a, b, o, args, grid, stream);
}

}  // namespace mns
