// Instantiations of the tensor-core kernel for fp32 operands (tf32 tensor
// cores, fp32 storage of the iterate and of A and B).
#include "gemm_launch.cuh"

namespace mns {

cudaError_t launch_sym_kk_f32(const GemmParams& p, int grid, cudaStream_t stream) {
  return launch_tc_gemm<false, false, true, 8, true>(p, grid, stream);
}

cudaError_t launch_sym_mnmn_f32(const GemmParams& p, int grid, cudaStream_t stream) {
  return launch_tc_gemm<true, true, true, 8, true>(p, grid, stream);
}

cudaError_t launch_full_kmn_f32(const GemmParams& p, int max_k, int grid, cudaStream_t stream) {
  return max_k <= 1024 ? launch_tc_gemm<false, true, false, 8, true>(p, grid, stream)
                       : launch_tc_gemm<false, true, false, 4, true>(p, grid, stream);
}

cudaError_t launch_full_kk_f32(const GemmParams& p, int max_k, int grid, cudaStream_t stream) {
  return max_k <= 1024 ? launch_tc_gemm<false, false, false, 8, true>(p, grid, stream)
                       : launch_tc_gemm<false, false, false, 4, true>(p, grid, stream);
}

}  // namespace mns
