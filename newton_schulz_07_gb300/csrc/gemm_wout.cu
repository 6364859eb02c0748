// Instantiations of the tensor-core kernel for the last update product of a
// Muon step (a X + B X, or a Y + Y B for tall inputs, bf16 operands), whose
// epilogue writes W = (1 - lr wd) W - lr scale bf16(X') into the fp32 master
// weights instead of storing X'.  Always 4 epilogue warps: the prefetched
// master-weight rows need the registers that 8 warps would not leave.  This
// unit holds the kernels whose factors are the launch's (WOUT = 1); those
// with each group's own factors (WOUT = 2) are in gemm_wout_grp.cu, compiled
// in parallel.
#include "gemm_launch.cuh"
#include "internal.h"

namespace mns {

template <bool B_MN>
cudaError_t launch_full_w(const GemmParams& p, PairMode mode, int grid, cudaStream_t stream) {
  if (mode == kSingle) return cudaErrorInvalidValue;
  return mode == kPairMma ? launch_tc_gemm<false, B_MN, false, 4, false, 2, true, 1>(p, grid, stream)
                          : launch_tc_gemm<false, B_MN, false, 4, false, 2, false, 1>(p, grid, stream);
}

cudaError_t launch_full_kmn_w(const GemmParams& p, PairMode mode, int grid, bool per_group, cudaStream_t stream) {
  return per_group ? launch_full_kmn_wg(p, mode, grid, stream) : launch_full_w<true>(p, mode, grid, stream);
}

cudaError_t launch_full_kk_w(const GemmParams& p, PairMode mode, int grid, bool per_group, cudaStream_t stream) {
  return per_group ? launch_full_kk_wg(p, mode, grid, stream) : launch_full_w<false>(p, mode, grid, stream);
}

}  // namespace mns
