// Kernel launch with programmatic dependent launch (host side).
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>
#include <utility>

namespace fp8fg {

// Programmatic dependent launch is on unless FP8FG_PDL=0 (an A/B switch for
// timing); the kernels call grid_dependency_sync() either way.
inline bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("FP8FG_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

// Launch `kernel` on `stream`; with programmatic stream serialization the
// kernel may begin (up to its grid_dependency_sync) while the previous
// kernel on the stream is still running.
template <typename... KParams, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KParams...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same, in clusters of `cluster_x` CTAs along x (grid.x a multiple of
// it).
template <typename... KParams, typename... Args>
cudaError_t launch_kernel_cluster(void (*kernel)(KParams...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace fp8fg
