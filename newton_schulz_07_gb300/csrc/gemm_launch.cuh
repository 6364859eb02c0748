// Launch helper for one instantiation of the tensor-core product kernel.
#pragma once

#include <atomic>

#include "gemm_tc.cuh"
#include "internal.h"

namespace mns {

template <bool A_MN, bool B_MN, bool SYM>
cudaError_t launch_tc_gemm(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& args,
                           int grid, cudaStream_t stream) {
  // The dynamic shared-memory limit is raised once per device.
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(ns_tc_gemm<A_MN, B_MN, SYM>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  ns_tc_gemm<A_MN, B_MN, SYM><<<grid, Epi<SYM>::kCtaThreads, kSmemBytes, stream>>>(a, b, args);
  return cudaGetLastError();
}

}  // namespace mns
