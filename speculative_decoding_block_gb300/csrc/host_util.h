// host_util.h -- host-side helpers shared by the library's translation
// units: the thread's last error message, the CUDA-call check and device
// allocation.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/vsd.h"

namespace vsd {

// Records the message (returned by vsd_last_error) and returns s.
vsd_status fail(vsd_status s, const char* fmt, ...);

#define CK(call)                                                                                     \
  do {                                                                                               \
    cudaError_t e_ = (call);                                                                         \
    if (e_ != cudaSuccess)                                                                           \
      return ::vsd::fail(e_ == cudaErrorMemoryAllocation ? VSD_ERR_OOM : VSD_ERR_CUDA, "%s: %s (%s:%d)", #call, \
                         cudaGetErrorString(e_), __FILE__, __LINE__);                                \
  } while (0)

template <typename T>
vsd_status dalloc(T** p, size_t count, bool zero = true) {
  *p = nullptr;
  if (count == 0) count = 1;
  CK(cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T)));
  if (zero) CK(cudaMemset(*p, 0, count * sizeof(T)));
  return VSD_OK;
}

inline int ceil_div_h(int x, int m) { return (x + m - 1) / m; }

// Programmatic dependent launch is used on explicit streams only (the
// legacy default stream keeps plain stream ordering).
inline bool use_pdl(cudaStream_t st) { return st != nullptr; }

}  // namespace vsd
