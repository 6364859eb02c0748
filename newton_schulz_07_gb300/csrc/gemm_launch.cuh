// Launch helper for one instantiation of the tensor-core product kernel.
#pragma once

#include <atomic>
#include <utility>

#include "gemm_tc.cuh"
#include "internal.h"

namespace mns {

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel in the stream finishes, and waits for it with
// griddepcontrol.wait before touching its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <bool A_MN, bool B_MN, bool SYM, int EPI_WARPS, bool F32 = false>
cudaError_t launch_tc_gemm(const GemmParams& p, int grid, cudaStream_t stream) {
  constexpr int kSmem = Staging<SYM, EPI_WARPS, F32>::kSmemBytes;
  // The dynamic shared-memory limit is raised once per device.
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(ns_tc_gemm<A_MN, B_MN, SYM, EPI_WARPS, F32>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  return launch_pdl(ns_tc_gemm<A_MN, B_MN, SYM, EPI_WARPS, F32>, dim3(grid), dim3(Epi<EPI_WARPS>::kCtaThreads),
                    kSmem, stream, p);
}

}  // namespace mns
