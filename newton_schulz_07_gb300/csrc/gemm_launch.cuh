// Launch helper for one instantiation of the tensor-core product kernel.
#pragma once

#include <atomic>
#include <utility>

#include "gemm_tc.cuh"
#include "internal.h"

namespace mns {

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel in the stream finishes, and waits for it with
// griddepcontrol.wait before touching its results (or, the products of a
// whole NS call, through per-matrix completion counters, with the wait moved
// to just before exit).  `cluster_x` > 1 launches clusters of that many CTAs
// along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  return launch_pdl_cluster(kernel, grid, block, smem, stream, 1, std::forward<Args>(args)...);
}

// `grid`: CTAs wanted (CL == 1) or clusters wanted (CL == 2), at most one per
// unit of the tile space.  Clusters are further limited to the number that
// can be resident at once (the kernel is persistent).
template <bool A_MN, bool B_MN, bool SYM, int EPI_WARPS, bool F32 = false, int CL = 1,
          bool SM2 = false, int WOUT = 0>
cudaError_t launch_tc_gemm(const GemmParams& p, int grid, cudaStream_t stream) {
  constexpr int kSmem = Smem<SYM, EPI_WARPS, F32, SM2>::kSmemBytes;
  constexpr int kThreads = Epi<EPI_WARPS>::kCtaThreads;
  auto kernel = ns_tc_gemm<A_MN, B_MN, SYM, EPI_WARPS, F32, CL, SM2, WOUT>;
  // Set up once per device: the dynamic shared-memory limit, and for
  // clusters the number of clusters that fit on the GPU at once.
  static std::atomic<unsigned long long> configured{0};
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (CL > 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(CL);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = CL;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
      if (e != cudaSuccess) return e;
      if (n < 1) return cudaErrorInvalidConfiguration;
      max_clusters[dev & 63].store(n);
    }
    configured.fetch_or(bit);
  }
  if (CL > 1) {
    const int mc = max_clusters[dev & 63].load();
    const int clusters = grid < mc ? grid : mc;
    return launch_pdl_cluster(kernel, dim3(CL * clusters), dim3(kThreads), kSmem, stream, CL, p);
  }
  return launch_pdl(kernel, dim3(grid), dim3(kThreads), kSmem, stream, p);
}

}  // namespace mns
