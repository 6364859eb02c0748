// Instantiations of the tensor-core kernel for the update products
// (a X + B X, and a Y + Y B for inputs kept in their tall orientation), bf16
// operands.  Short contractions (K <= 1024) on multicast pairs take 8
// epilogue warps, the rest 4 (update_epi_warps; measured on GB300).
#include "gemm_launch.cuh"

namespace mns {

// bf16 products always run on CTA pairs (pair_mode never picks kSingle).
template <bool B_MN>
cudaError_t launch_full(const GemmParams& p, PairMode mode, int max_k, int grid, cudaStream_t stream) {
  if (mode == kSingle) return cudaErrorInvalidValue;
  if (mode == kPairMma) return launch_tc_gemm<false, B_MN, false, 4, false, 2, true>(p, grid, stream);
  return update_epi_warps(mode, max_k) == 8
             ? launch_tc_gemm<false, B_MN, false, 8, false, 2, false>(p, grid, stream)
             : launch_tc_gemm<false, B_MN, false, 4, false, 2, false>(p, grid, stream);
}

cudaError_t launch_full_kmn(const GemmParams& p, PairMode mode, int max_k, int grid, cudaStream_t stream) {
  return launch_full<true>(p, mode, max_k, grid, stream);
}

cudaError_t launch_full_kk(const GemmParams& p, PairMode mode, int max_k, int grid, cudaStream_t stream) {
  return launch_full<false>(p, mode, max_k, grid, stream);
}

}  // namespace mns
