// Instantiations of the tensor-core kernel for fp32 operands (tf32 tensor
// cores, fp32 storage of the iterate and of A and B).  Every fp32 operand is
// K-major; long contractions run on CTA pairs with 2-SM MMAs, short ones on
// single CTAs.
#include "gemm_launch.cuh"

namespace mns {

template <bool MN>
cudaError_t launch_sym_f32(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream) {
  return mode == kPairMma ? launch_tc_gemm<MN, MN, true, 8, true, 2, true>(p, grid, stream)
                          : launch_tc_gemm<MN, MN, true, 8, true, 1, false>(p, grid, stream);
}

cudaError_t launch_sym_kk_f32(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream) {
  return launch_sym_f32<false>(p, mode, grid, stream);
}

cudaError_t launch_sym_mnmn_f32(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream) {
  return launch_sym_f32<true>(p, mode, grid, stream);
}

template <bool B_MN>
cudaError_t launch_full_f32(const GemmParams& p, PairMode mode, int max_k, int grid, cudaStream_t stream) {
  if (mode == kPairMma) return launch_tc_gemm<false, B_MN, false, 4, true, 2, true>(p, grid, stream);
  return max_k <= kShortK ? launch_tc_gemm<false, B_MN, false, 8, true, 1, false>(p, grid, stream)
                       : launch_tc_gemm<false, B_MN, false, 4, true, 1, false>(p, grid, stream);
}

cudaError_t launch_full_kmn_f32(const GemmParams& p, PairMode mode, int max_k, int grid, cudaStream_t stream) {
  return launch_full_f32<true>(p, mode, max_k, grid, stream);
}

cudaError_t launch_full_kk_f32(const GemmParams& p, PairMode mode, int max_k, int grid, cudaStream_t stream) {
  return launch_full_f32<false>(p, mode, max_k, grid, stream);
}

}  // namespace mns
