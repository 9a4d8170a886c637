// gemm.cu -- instantiations and launcher of the weight-streaming GEMM.
#include <utility>

#include "launch.h"

namespace vsd {

template <int WF, int EPI>
static cudaError_t launch_one(const CUtensorMap& tm_act, const CUtensorMap& tm_w, const GemmArgs& a, int grid,
                              cudaStream_t st, bool pdl) {
  const uint32_t smem = gemm_smem_bytes(WF, a.n_tok, a.stages);
  static uint32_t configured = 0;  // largest dynamic shared memory set so far
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<WF, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    configured = 232448;
  }
  return launch_ex(gemm_kernel<WF, EPI>, dim3(grid), dim3(kGemmThreads), smem, st, pdl, tm_act, tm_w, a);
}

template <int WF>
static cudaError_t launch_fmt(int epi, const CUtensorMap& tm_act, const CUtensorMap& tm_w, const GemmArgs& a,
                              int grid, cudaStream_t st, bool pdl) {
  switch (epi) {
    case EPI_STORE: return launch_one<WF, EPI_STORE>(tm_act, tm_w, a, grid, st, pdl);
    case EPI_RESID: return launch_one<WF, EPI_RESID>(tm_act, tm_w, a, grid, st, pdl);
    case EPI_QKV: return launch_one<WF, EPI_QKV>(tm_act, tm_w, a, grid, st, pdl);
    case EPI_SILU: return launch_one<WF, EPI_SILU>(tm_act, tm_w, a, grid, st, pdl);
    case EPI_ARGMAX: return launch_one<WF, EPI_ARGMAX>(tm_act, tm_w, a, grid, st, pdl);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(int wf, int epi, const CUtensorMap& tm_act, const CUtensorMap& tm_w, const GemmArgs& a,
                        int grid, cudaStream_t st, bool pdl) {
  switch (wf) {
    case W_BF16: return launch_fmt<W_BF16>(epi, tm_act, tm_w, a, grid, st, pdl);
    case W_FP8: return launch_fmt<W_FP8>(epi, tm_act, tm_w, a, grid, st, pdl);
    case W_NVFP4: return launch_fmt<W_NVFP4>(epi, tm_act, tm_w, a, grid, st, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace vsd
