// launch.h -- host-side launchers of the templated kernels (one translation
// unit per kernel family keeps the build parallel).
#pragma once

#include <map>
#include <mutex>
#include <utility>

#include "attention.cuh"
#include "gemm.cuh"
#include "persistent.cuh"

namespace vsd {

// Opts kernel `k` in to at least `bytes` of dynamic shared memory on the
// current device.  The attribute is one value per (kernel, device) that
// every later launch is checked against, so it only ever grows: a smaller
// request after a larger one keeps the larger limit.  Thread-safe.
inline cudaError_t ensure_smem_opt_in(const void* k, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> limit;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(k, dev);
  const auto it = limit.find(key);
  if (it != limit.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) limit[key] = bytes;
  return e;
}

// Launches gemm_kernel<wf, epi> on `grid` persistent CTAs; programmatic
// dependent launch when pdl is set.
// Launches gemm_kernel<wf, epi> as a.cs-CTA clusters; `grid` is a multiple of
// a.cs and is clamped to the clusters that can be resident at once.
// Clusters of `cs` GEMM CTAs (full shared memory each) that can be resident at once.
int gemm_max_clusters(int cs);
cudaError_t launch_gemm(int wf, int epi, const CUtensorMap& tm_act, const GemmArgs& a, int grid, cudaStream_t st,
                        bool pdl);
cudaError_t launch_attn(int hd, const CUtensorMap& tm_q, const CUtensorMap& tm_kc, const CUtensorMap& tm_vc,
                        const CUtensorMap& tm_kn, const CUtensorMap& tm_vn, const AttnArgs& a, dim3 grid,
                        cudaStream_t st, bool pdl);

// Launches the persistent step kernel (head_dim 64 or 128) on `grid` CTAs, one per SM.
cudaError_t launch_step(int hd, const MkParams& p, int grid, cudaStream_t st);

template <typename... KArgs, typename... Args>
cudaError_t launch_ex_cluster(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster, cudaStream_t st,
                              bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeClusterDimension;
  attr[n].val.clusterDim.x = cluster;
  attr[n].val.clusterDim.y = 1;
  attr[n].val.clusterDim.z = 1;
  ++n;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

// `cooperative`: the CTAs of the grid wait on one another, so the launch
// must guarantee that they are all resident at once.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                      bool cooperative, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

}  // namespace vsd
