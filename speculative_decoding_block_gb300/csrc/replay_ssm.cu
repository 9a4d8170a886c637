// replay_ssm.cu -- host side of the recurrent-state rollback (vsd_ssm_*):
// the state object, its buffers and the launches of the kernels in
// replay_ssm.cuh.
#include <algorithm>

#include "host_util.h"
#include "launch.h"
#include "replay_ssm.cuh"

using namespace vsd;

struct vsd_ssm {
  int max_batch = 0, heads = 0, d = 0, window = 0, sms = 1;
  uint8_t *ckpt = nullptr, *buf_k = nullptr;  // row images (replay_ssm.cuh)
  int *ckpt_exp = nullptr, *buf_kexp = nullptr;
  float* buf_u = nullptr;
  double* buf_L = nullptr;
  int* ptr = nullptr;
  int* status = nullptr;
};

namespace {
template <int D>
vsd_status ssm_opt_in(uint32_t verify_smem, uint32_t fold_smem) {
  cudaError_t e;
  if ((e = ensure_smem_opt_in(reinterpret_cast<const void*>(ssm_verify_kernel<D>), static_cast<int>(verify_smem))) ||
      (e = ensure_smem_opt_in(reinterpret_cast<const void*>(ssm_flush_kernel<D>), static_cast<int>(fold_smem))) ||
      (e = ensure_smem_opt_in(reinterpret_cast<const void*>(ssm_state_kernel<D>), static_cast<int>(fold_smem))) ||
      (e = ensure_smem_opt_in(reinterpret_cast<const void*>(ssm_set_kernel<D>), static_cast<int>(fold_smem))))
    return fail(VSD_ERR_CUDA, "shared-memory opt-in: %s", cudaGetErrorString(e));
  return VSD_OK;
}

SsmArgs ssm_args(const vsd_ssm* s, int batch) {
  SsmArgs a{};
  a.heads = s->heads;
  a.d = s->d;
  a.window = s->window;
  a.batch = batch;
  a.ckpt = s->ckpt;
  a.ckpt_exp = s->ckpt_exp;
  a.buf_k = s->buf_k;
  a.buf_kexp = s->buf_kexp;
  a.buf_u = s->buf_u;
  a.buf_L = s->buf_L;
  a.ptr = s->ptr;
  a.status = s->status;
  return a;
}
}  // namespace

vsd_status vsd_ssm_create(int32_t max_batch, int32_t heads, int32_t d, int32_t window, vsd_ssm** out) {
  if (!out) return fail(VSD_ERR_ARG, "NULL pointer");
  *out = nullptr;
  if (max_batch < 1 || heads < 1 || window < kRows || window > kSsmMaxWindow)
    return fail(VSD_ERR_ARG, "max_batch, heads >= 1 and window in [17, %d]", kSsmMaxWindow);
  if (d != 64 && d != 128) return fail(VSD_ERR_UNSUPPORTED, "state dimension d must be 64 or 128");
  if (window > ssm_max_window(d))
    return fail(VSD_ERR_UNSUPPORTED, "window %d above %d for d = %d (shared memory)", window, ssm_max_window(d), d);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(VSD_ERR_CUDA, "no CUDA device");
  const uint32_t vsmem = ssm_verify_layout(d, window).total, fsmem = ssm_fold_smem_bytes(d, window);
  vsd_status st = d == 64 ? ssm_opt_in<64>(vsmem, fsmem) : ssm_opt_in<128>(vsmem, fsmem);
  if (st) return st;
  int sms = 1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return fail(VSD_ERR_CUDA, "SM count");
  vsd_ssm* s = new vsd_ssm();
  s->max_batch = max_batch;
  s->heads = heads;
  s->d = d;
  s->window = window;
  s->sms = sms;
  const size_t hb = static_cast<size_t>(max_batch) * heads;
  if ((st = dalloc(&s->ckpt, hb * d * d * 4)) || (st = dalloc(&s->ckpt_exp, hb * d)) ||
      (st = dalloc(&s->buf_k, hb * window * d * 4)) || (st = dalloc(&s->buf_kexp, hb * ssm_exp_stride(window))) ||
      (st = dalloc(&s->buf_u, hb * window * d)) || (st = dalloc(&s->buf_L, hb * window)) ||
      (st = dalloc(&s->ptr, max_batch)) || (st = dalloc(&s->status, 1))) {
    vsd_ssm_destroy(s);
    return st;
  }
  *out = s;
  return VSD_OK;
}

void vsd_ssm_destroy(vsd_ssm* s) {
  if (!s) return;
  void* ptrs[] = {s->ckpt, s->ckpt_exp, s->buf_k, s->buf_kexp, s->buf_u, s->buf_L, s->ptr, s->status};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  delete s;
}

vsd_status vsd_ssm_set_state(vsd_ssm* s, int32_t req, const float* state, vsd_stream stream) {
  if (!s || !state) return fail(VSD_ERR_ARG, "NULL pointer");
  if (req < 0 || req >= s->max_batch) return fail(VSD_ERR_ARG, "request %d outside [0, %d)", req, s->max_batch);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  SsmArgs a = ssm_args(s, 0);
  a.state_in = state;
  a.req = req;
  const uint32_t smem = ssm_fold_smem_bytes(s->d, s->window);
  if (s->d == 64) ssm_set_kernel<64><<<s->heads, kSsmThreads, smem, st>>>(a);
  else ssm_set_kernel<128><<<s->heads, kSsmThreads, smem, st>>>(a);
  CK(cudaGetLastError());
  CK(cudaMemsetAsync(s->ptr + req, 0, sizeof(int), st));
  return VSD_OK;
}

vsd_status vsd_ssm_get_state(vsd_ssm* s, int32_t req, float* state, vsd_stream stream) {
  if (!s || !state) return fail(VSD_ERR_ARG, "NULL pointer");
  if (req < 0 || req >= s->max_batch) return fail(VSD_ERR_ARG, "request %d outside [0, %d)", req, s->max_batch);
  SsmArgs a = ssm_args(s, 0);
  a.state_out = state;
  a.req = req;
  const uint32_t smem = ssm_fold_smem_bytes(s->d, s->window);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (s->d == 64) ssm_state_kernel<64><<<s->heads, kSsmThreads, smem, st>>>(a);
  else ssm_state_kernel<128><<<s->heads, kSsmThreads, smem, st>>>(a);
  CK(cudaGetLastError());
  return VSD_OK;
}

vsd_status vsd_ssm_verify(vsd_ssm* s, int32_t batch, const float* q, const float* k, const float* v,
                          const float* alpha, const float* beta, float* out, vsd_stream stream) {
  if (!s || !q || !k || !v || !alpha || !beta || !out) return fail(VSD_ERR_ARG, "NULL pointer");
  if (batch < 1 || batch > s->max_batch) return fail(VSD_ERR_ARG, "batch %d outside [1, %d]", batch, s->max_batch);
  for (const void* x : {static_cast<const void*>(q), static_cast<const void*>(k), static_cast<const void*>(v),
                        static_cast<const void*>(out)})
    if (reinterpret_cast<uintptr_t>(x) % 16) return fail(VSD_ERR_ARG, "q, k, v and out must be 16-byte aligned");
  SsmArgs a = ssm_args(s, batch);
  a.q = q;
  a.k = k;
  a.v = v;
  a.alpha = alpha;
  a.beta = beta;
  a.out = out;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const uint32_t smem = ssm_verify_layout(s->d, s->window).total;
  const dim3 grid(std::min(s->heads * batch, s->sms));  // persistent over the (request, head) items
  const cudaError_t e = s->d == 64 ? launch_ex(ssm_verify_kernel<64>, grid, dim3(kSsmThreads), smem, st, use_pdl(st), false, a)
                                   : launch_ex(ssm_verify_kernel<128>, grid, dim3(kSsmThreads), smem, st, use_pdl(st), false, a);
  if (e != cudaSuccess) return fail(VSD_ERR_CUDA, "replay verify launch: %s", cudaGetErrorString(e));
  return VSD_OK;
}

vsd_status vsd_ssm_commit(vsd_ssm* s, int32_t batch, const int32_t* accepted, vsd_stream stream) {
  if (!s || !accepted) return fail(VSD_ERR_ARG, "NULL pointer");
  if (batch < 1 || batch > s->max_batch) return fail(VSD_ERR_ARG, "batch %d outside [1, %d]", batch, s->max_batch);
  SsmArgs a = ssm_args(s, batch);
  a.accepted = accepted;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const uint32_t smem = ssm_fold_smem_bytes(s->d, s->window);
  const dim3 grid(s->heads, batch);
  cudaError_t e = s->d == 64 ? launch_ex(ssm_flush_kernel<64>, grid, dim3(kSsmThreads), smem, st, use_pdl(st), false, a)
                             : launch_ex(ssm_flush_kernel<128>, grid, dim3(kSsmThreads), smem, st, use_pdl(st), false, a);
  if (e == cudaSuccess)
    e = launch_ex(ssm_pointer_kernel, dim3(ceil_div_h(batch, 128)), dim3(128), 0, st, use_pdl(st), false, a);
  if (e != cudaSuccess) return fail(VSD_ERR_CUDA, "replay commit launch: %s", cudaGetErrorString(e));
  return VSD_OK;
}

vsd_status vsd_ssm_get_device_status(vsd_ssm* s, vsd_stream stream, int32_t* out) {
  if (!s || !out) return fail(VSD_ERR_ARG, "NULL pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  CK(cudaMemcpyAsync(&v, s->status, 4, cudaMemcpyDeviceToHost, st));
  CK(cudaMemsetAsync(s->status, 0, 4, st));
  CK(cudaStreamSynchronize(st));
  *out = v;
  return VSD_OK;
}
