// attention.cu -- instantiations and launcher of the verify attention.
#include <utility>

#include "launch.h"

namespace vsd {

template <int HD>
static cudaError_t launch_hd(const CUtensorMap& tm_q, const CUtensorMap& tm_kc, const CUtensorMap& tm_vc,
                             const CUtensorMap& tm_kn, const CUtensorMap& tm_vn, const AttnArgs& a, dim3 grid,
                             cudaStream_t st, bool pdl) {
  const uint32_t smem = attn_smem_bytes(HD);
  const cudaError_t e = ensure_smem_opt_in(reinterpret_cast<const void*>(attn_kernel<HD>), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // cooperative: the splits of a request wait for one another before merging
  return launch_ex(attn_kernel<HD>, grid, dim3(kAttnThreads), smem, st, pdl, true, tm_q, tm_kc, tm_vc, tm_kn, tm_vn,
                   a);
}

cudaError_t launch_attn(int hd, const CUtensorMap& tm_q, const CUtensorMap& tm_kc, const CUtensorMap& tm_vc,
                        const CUtensorMap& tm_kn, const CUtensorMap& tm_vn, const AttnArgs& a, dim3 grid,
                        cudaStream_t st, bool pdl) {
  if (hd == 64) return launch_hd<64>(tm_q, tm_kc, tm_vc, tm_kn, tm_vn, a, grid, st, pdl);
  if (hd == 128) return launch_hd<128>(tm_q, tm_kc, tm_vc, tm_kn, tm_vn, a, grid, st, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace vsd
