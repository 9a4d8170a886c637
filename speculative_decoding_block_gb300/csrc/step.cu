// step.cu -- instantiations and launcher of the persistent step kernel.
#include "launch.h"

namespace vsd {

template <int HD>
static cudaError_t launch_step_hd(const MkParams& p, int grid, cudaStream_t st) {
  const uint32_t smem = MkCfg<HD>::SMEM;
  const cudaError_t e = ensure_smem_opt_in(reinterpret_cast<const void*>(step_kernel<HD>), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // cooperative: the CTAs wait on one another between phases, so the whole
  // grid must be resident at once (the launch fails otherwise)
  return launch_ex(step_kernel<HD>, dim3(grid), dim3(kMkThreads), smem, st, false, true, p);
}

cudaError_t launch_step(int hd, const MkParams& p, int grid, cudaStream_t st) {
  if (hd == 64) return launch_step_hd<64>(p, grid, st);
  if (hd == 128) return launch_step_hd<128>(p, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace vsd
