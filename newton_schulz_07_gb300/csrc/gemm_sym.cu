// Instantiations of the tensor-core kernel for the symmetric products
// (Gram X X^T or Y^T Y, and b A + c A A), bf16 operands.
#include "gemm_launch.cuh"

namespace mns {

// bf16 products always run on CTA pairs (pair_mode never picks kSingle).
template <bool MN>
cudaError_t launch_sym(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream) {
  if (mode == kSingle) return cudaErrorInvalidValue;
  return mode == kPairMma ? launch_tc_gemm<MN, MN, true, 8, false, 2, true>(p, grid, stream)
                          : launch_tc_gemm<MN, MN, true, 8, false, 2, false>(p, grid, stream);
}

cudaError_t launch_sym_kk(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream) {
  return launch_sym<false>(p, mode, grid, stream);
}

cudaError_t launch_sym_mnmn(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream) {
  return launch_sym<true>(p, mode, grid, stream);
}

}  // namespace mns
