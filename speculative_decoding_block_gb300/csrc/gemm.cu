// gemm.cu -- instantiations and launcher of the weight-streaming GEMM.
#include <algorithm>
#include <utility>

#include "launch.h"

namespace vsd {

template <int WF, int EPI>
static cudaError_t launch_one(const CUtensorMap& tm_act, const GemmArgs& a, int grid,
                              cudaStream_t st, bool pdl) {
  const uint32_t smem = gemm_smem_bytes(WF, a.n_tok, a.rd, a.da, a.db, a.cs, a.act_lo_rows > 0, a.r_alias != 0);
  const cudaError_t e = ensure_smem_opt_in(reinterpret_cast<const void*>(gemm_kernel<WF, EPI>), 232448);
  if (e != cudaSuccess) return e;
  if (a.cs > 1) {
    // no more clusters than can be resident together (the CTAs loop over items)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = a.cs;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, gemm_kernel<WF, EPI>, &cfg) == cudaSuccess && max_clusters > 0)
      grid = std::min(grid, max_clusters * a.cs);
    return launch_ex_cluster(gemm_kernel<WF, EPI>, dim3(grid), dim3(kGemmThreads), smem, a.cs, st, pdl, tm_act, a);
  }
  return launch_ex(gemm_kernel<WF, EPI>, dim3(grid), dim3(kGemmThreads), smem, st, pdl, false, tm_act, a);
}

template <int WF>
static cudaError_t launch_fmt(int epi, const CUtensorMap& tm_act, const GemmArgs& a,
                              int grid, cudaStream_t st, bool pdl) {
  switch (epi) {
    case EPI_STORE: return launch_one<WF, EPI_STORE>(tm_act, a, grid, st, pdl);
    case EPI_RESID: return launch_one<WF, EPI_RESID>(tm_act, a, grid, st, pdl);
    case EPI_QKV: return launch_one<WF, EPI_QKV>(tm_act, a, grid, st, pdl);
    case EPI_SILU: return launch_one<WF, EPI_SILU>(tm_act, a, grid, st, pdl);
    case EPI_ARGMAX: return launch_one<WF, EPI_ARGMAX>(tm_act, a, grid, st, pdl);
    case EPI_SAMPLE:
      if constexpr (WF == W_BF16) return launch_one<WF, EPI_SAMPLE>(tm_act, a, grid, st, pdl);
      return cudaErrorInvalidValue;  // the head is a 16-bit matrix
  }
  return cudaErrorInvalidValue;
}

int gemm_max_clusters(int cs) {
  if (cs <= 1) {
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
  }
  auto k = gemm_kernel<W_FP8, EPI_RESID>;
  if (ensure_smem_opt_in(reinterpret_cast<const void*>(k), 232448) != cudaSuccess) return 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs * 64);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = 232448;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = cs;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n < 1) return 1;
  return n;
}

cudaError_t launch_gemm(int wf, int epi, const CUtensorMap& tm_act, const GemmArgs& a,
                        int grid, cudaStream_t st, bool pdl) {
  switch (wf) {
    case W_BF16: return launch_fmt<W_BF16>(epi, tm_act, a, grid, st, pdl);
    case W_FP8: return launch_fmt<W_FP8>(epi, tm_act, a, grid, st, pdl);
    case W_NVFP4: return launch_fmt<W_NVFP4>(epi, tm_act, a, grid, st, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace vsd
