// The last-update kernels of a grouped Muon step whose stacks differ in
// learning rate, weight decay or shape scale: as in gemm_wout.cu, but the
// epilogue takes each group's factors (WOUT = 2).
#include "gemm_launch.cuh"
#include "internal.h"

namespace mns {

template <bool B_MN>
cudaError_t launch_full_wg(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream) {
  if (mode == kSingle) return cudaErrorInvalidValue;
  return mode == kPairMma ? launch_tc_gemm<false, B_MN, false, 4, false, 2, true, 2>(p, grid, stream)
                          : launch_tc_gemm<false, B_MN, false, 4, false, 2, false, 2>(p, grid, stream);
}

cudaError_t launch_full_kmn_wg(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream) {
  return launch_full_wg<true>(p, mode, grid, stream);
}

cudaError_t launch_full_kk_wg(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream) {
  return launch_full_wg<false>(p, mode, grid, stream);
}

}  // namespace mns
