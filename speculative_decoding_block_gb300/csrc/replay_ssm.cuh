// replay_ssm.cuh -- ReplaySSM-style verification and rollback of a recurrent
// (gated delta rule) layer under block speculative decoding.
//
// "The Inference Stack Behind OCRia", section "Make speculative verification
// cheaper": a GDN layer's fixed-size state is kept as a checkpoint plus a
// small buffer of recent inputs; outputs are computed from the checkpoint and
// the buffered inputs, the checkpoint is rewritten only at periodic flushes,
// and rejected drafts are rolled back by moving the buffer pointer.  The
// pages give no update rule; the gated delta rule of Gated DeltaNet is used:
//     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
//     o_t = S_t q_t,
// per request and head, S of d x d (d_k = d_v = d).  Computed per thread as
// u = S k, S <- alpha S + beta (v - alpha u) k^T, o = S q.
//
// The rows of S update independently (row i needs only S[i,:], k, v_i and the
// gates), so a CTA of 256 threads takes 64 rows of one (head, request): four
// adjacent lanes share a row, each holding d / 4 of its columns in registers.
// Every input of the replay is staged in shared memory first, so the token
// loop needs no block-wide barrier (a row's dot products reduce across its
// four lanes).  grid (H, B, d / 64).
#pragma once

#include "vsd_common.cuh"

namespace vsd {

constexpr int kSsmThreads = 256;
constexpr int kSsmTpr = 4;                          // lanes per state row
constexpr int kSsmRowsPerCta = kSsmThreads / kSsmTpr;  // 64
constexpr int kSsmMaxWindow = 128;

struct SsmArgs {
  int heads, d, window, batch;
  // a verify block [B][H][17][d] (q, k, v) and [B][H][17] (alpha, beta)
  const float *q, *k, *v, *alpha, *beta;
  float* out;                        // [B][H][17][d]
  float* ckpt;                       // [max_batch][H][d][d]
  float *buf_k, *buf_v, *buf_ab;     // [max_batch][H][window][d], same, [..][window][2]
  int* ptr;                          // [max_batch] retained buffered tokens
  const int* accepted;               // [B] commit: accepted drafts a (-1: rejected)
  float* state_out;                  // [H][d][d] effective state of one request
  int req;                           // its request
  int* status;
};

__host__ __device__ inline uint32_t ssm_smem_bytes(int d, int window) {
  return static_cast<uint32_t>(window * (2 * d + 2) + kRows * d) * 4u;
}

// The thread's d / TPR columns of its row (lane c0 of the row holds the
// float4 chunks c0, c0 + TPR, c0 + 2 TPR, ...: the row's four lanes read
// consecutive 16-byte pieces, free of bank conflicts) through `n` staged
// tokens; with q
// given, the outputs of tokens n_out_from.. are written to out (row t of out
// for token n_out_from + t).
template <int D>
__device__ __forceinline__ void ssm_replay(float* S, const float* sk, const float* sv, const float* sab, int n,
                                           const float* sq, int n_out_from, float* out, int row, int c0) {
  constexpr int TPR = kSsmTpr, CPT = D / TPR;
  for (int tau = 0; tau < n; ++tau) {
    const float4* k4 = reinterpret_cast<const float4*>(sk + tau * D) + c0;
    // four independent partial sums: the dot product's dependent chain is d / 16 long
    float u0 = 0.0f, u1 = 0.0f, u2 = 0.0f, u3 = 0.0f;
#pragma unroll
    for (int c = 0; c < CPT / 4; ++c) {
      const float4 kk = k4[c * TPR];
      u0 = fmaf(S[4 * c], kk.x, u0);
      u1 = fmaf(S[4 * c + 1], kk.y, u1);
      u2 = fmaf(S[4 * c + 2], kk.z, u2);
      u3 = fmaf(S[4 * c + 3], kk.w, u3);
    }
    float u = (u0 + u1) + (u2 + u3);
#pragma unroll
    for (int o = 1; o < TPR; o <<= 1) u += __shfl_xor_sync(0xFFFFFFFFu, u, o);
    const float alpha = sab[2 * tau], beta = sab[2 * tau + 1];
    const float coef = beta * (sv[tau * D + row] - alpha * u);
#pragma unroll
    for (int c = 0; c < CPT / 4; ++c) {
      const float4 kk = k4[c * TPR];
      S[4 * c] = alpha * S[4 * c] + coef * kk.x;
      S[4 * c + 1] = alpha * S[4 * c + 1] + coef * kk.y;
      S[4 * c + 2] = alpha * S[4 * c + 2] + coef * kk.z;
      S[4 * c + 3] = alpha * S[4 * c + 3] + coef * kk.w;
    }
    if (sq != nullptr && tau >= n_out_from) {
      const float4* q4 = reinterpret_cast<const float4*>(sq + (tau - n_out_from) * D) + c0;
      float o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f;
#pragma unroll
      for (int c = 0; c < CPT / 4; ++c) {
        const float4 qq = q4[c * TPR];
        o0 = fmaf(S[4 * c], qq.x, o0);
        o1 = fmaf(S[4 * c + 1], qq.y, o1);
        o2 = fmaf(S[4 * c + 2], qq.z, o2);
        o3 = fmaf(S[4 * c + 3], qq.w, o3);
      }
      float o = (o0 + o1) + (o2 + o3);
#pragma unroll
      for (int x = 1; x < TPR; x <<= 1) o += __shfl_xor_sync(0xFFFFFFFFu, o, x);
      if ((threadIdx.x % TPR) == 0) out[(tau - n_out_from) * D + row] = o;
    }
  }
}

template <int D>
__device__ __forceinline__ void ssm_load_rows(float* S, const float* src, int row, int c0) {
  constexpr int CPT = D / kSsmTpr;
  const float4* s4 = reinterpret_cast<const float4*>(src + row * D) + c0;
#pragma unroll
  for (int c = 0; c < CPT / 4; ++c) {
    const float4 x = s4[c * kSsmTpr];
    S[4 * c] = x.x;
    S[4 * c + 1] = x.y;
    S[4 * c + 2] = x.z;
    S[4 * c + 3] = x.w;
  }
}

template <int D>
__device__ __forceinline__ void ssm_store_rows(const float* S, float* dst, int row, int c0) {
  constexpr int CPT = D / kSsmTpr;
  float4* d4 = reinterpret_cast<float4*>(dst + row * D) + c0;
#pragma unroll
  for (int c = 0; c < CPT / 4; ++c) d4[c * kSsmTpr] = make_float4(S[4 * c], S[4 * c + 1], S[4 * c + 2], S[4 * c + 3]);
}

// Buffered tokens 0..n-1 of (request b, head h) into shared memory.
template <int D>
__device__ __forceinline__ void ssm_stage_buffer(const SsmArgs& a, size_t hb, int n, float* sk, float* sv, float* sab) {
  const float4* bk = reinterpret_cast<const float4*>(a.buf_k + hb * a.window * D);
  const float4* bv = reinterpret_cast<const float4*>(a.buf_v + hb * a.window * D);
  for (int x = threadIdx.x; x < n * D / 4; x += kSsmThreads) {
    reinterpret_cast<float4*>(sk)[x] = bk[x];
    reinterpret_cast<float4*>(sv)[x] = bv[x];
  }
  const float* bab = a.buf_ab + hb * a.window * 2;
  for (int x = threadIdx.x; x < 2 * n; x += kSsmThreads) sab[x] = bab[x];
}

// Verify: outputs of the 17 block rows from the checkpoint replayed through
// the retained buffer and the block; the block's inputs are staged in the
// buffer after the pointer (the commit decides how many stay).  grid (H, B, d / 64).
template <int D>
__global__ void __launch_bounds__(kSsmThreads, 3) ssm_verify_kernel(const SsmArgs a) {
  constexpr int TPR = kSsmTpr, CPT = D / TPR;
  extern __shared__ float4 ssm_smem4[];
  float* sm = reinterpret_cast<float*>(ssm_smem4);
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const int row = blockIdx.z * kSsmRowsPerCta + t / TPR, c0 = t % TPR;
  const int n = a.ptr[b];
  if (n < 0 || n + kRows > a.window) {  // a pointer the commit never leaves: no output, nothing staged
    if (t == 0 && h == 0 && blockIdx.z == 0) atomicOr(a.status, VSD_DEV_BAD_SEQLEN);
    return;
  }
  const size_t hb = static_cast<size_t>(b) * a.heads + h;
  const int nt = n + kRows;
  float* sk = sm;           // [nt][D]
  float* sv = sk + nt * D;  // [nt][D]
  float* sq = sv + nt * D;  // [17][D]
  float* sab = sq + kRows * D;  // [nt][2]
  ssm_stage_buffer<D>(a, hb, n, sk, sv, sab);
  const size_t blk = hb * kRows;
  for (int x = t; x < kRows * D / 4; x += kSsmThreads) {
    reinterpret_cast<float4*>(sk + n * D)[x] = reinterpret_cast<const float4*>(a.k + blk * D)[x];
    reinterpret_cast<float4*>(sv + n * D)[x] = reinterpret_cast<const float4*>(a.v + blk * D)[x];
    reinterpret_cast<float4*>(sq)[x] = reinterpret_cast<const float4*>(a.q + blk * D)[x];
  }
  if (t < kRows) {
    sab[2 * (n + t)] = a.alpha[blk + t];
    sab[2 * (n + t) + 1] = a.beta[blk + t];
  }
  float S[CPT];
  ssm_load_rows<D>(S, a.ckpt + hb * D * D, row, c0);
  __syncthreads();
  ssm_replay<D>(S, sk, sv, sab, nt, sq, n, a.out + blk * D, row, c0);
  // the block's inputs after the pointer (once per head: the first row slice)
  if (blockIdx.z != 0) return;
  float4* bk = reinterpret_cast<float4*>(a.buf_k + (hb * a.window + n) * D);
  float4* bv = reinterpret_cast<float4*>(a.buf_v + (hb * a.window + n) * D);
  for (int x = t; x < kRows * D / 4; x += kSsmThreads) {
    bk[x] = reinterpret_cast<const float4*>(sk + n * D)[x];
    bv[x] = reinterpret_cast<const float4*>(sv + n * D)[x];
  }
  if (t < 2 * kRows) a.buf_ab[(hb * a.window + n) * 2 + t] = sab[2 * n + t];
}

// The number of buffered tokens after the commit of request b (accepted
// drafts a: rows 0..a stay; -1: none).  An out-of-range a rejects the block.
__device__ __forceinline__ int ssm_committed(const SsmArgs& a, int b, bool report) {
  const int acc = a.accepted[b];
  const bool ok = acc >= -1 && acc < kRows;
  if (!ok && report) atomicOr(a.status, VSD_DEV_BAD_SEQLEN);
  return a.ptr[b] + (ok ? acc + 1 : 0);
}

// Commit, first part: a request whose next block would not fit the buffer
// folds its retained tokens into the checkpoint.  grid (H, B, d / 64).
template <int D>
__global__ void __launch_bounds__(kSsmThreads, 3) ssm_flush_kernel(const SsmArgs a) {
  constexpr int TPR = kSsmTpr, CPT = D / TPR;
  extern __shared__ float4 ssm_smem4[];
  float* sm = reinterpret_cast<float*>(ssm_smem4);
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
  const int n = ssm_committed(a, b, t == 0 && h == 0 && blockIdx.z == 0);
  if (n + kRows <= a.window || n > a.window) return;  // no flush (n > window: never left by a verify)
  const int row = blockIdx.z * kSsmRowsPerCta + t / TPR, c0 = t % TPR;
  const size_t hb = static_cast<size_t>(b) * a.heads + h;
  float* sk = sm;
  float* sv = sk + n * D;
  float* sab = sv + n * D;
  ssm_stage_buffer<D>(a, hb, n, sk, sv, sab);
  float S[CPT];
  ssm_load_rows<D>(S, a.ckpt + hb * D * D, row, c0);
  __syncthreads();
  ssm_replay<D>(S, sk, sv, sab, n, nullptr, 0, nullptr, row, c0);
  ssm_store_rows<D>(S, a.ckpt + hb * D * D, row, c0);
}

// Commit, second part: the pointers (0 after a flush).  One thread per request.
__global__ void ssm_pointer_kernel(const SsmArgs a) {
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.batch) return;
  const int n = ssm_committed(a, b, false);
  a.ptr[b] = (n + kRows > a.window) ? 0 : n;
}

// The effective state of request a.req: its checkpoint replayed through the
// retained buffer.  grid (H, 1, d / 64).
template <int D>
__global__ void __launch_bounds__(kSsmThreads, 3) ssm_state_kernel(const SsmArgs a) {
  constexpr int TPR = kSsmTpr, CPT = D / TPR;
  extern __shared__ float4 ssm_smem4[];
  float* sm = reinterpret_cast<float*>(ssm_smem4);
  const int h = blockIdx.x, t = threadIdx.x;
  const int n = min(max(a.ptr[a.req], 0), a.window);
  // (grid (H, 1, d / 64): blockIdx.z is the row slice)
  const int row = blockIdx.z * kSsmRowsPerCta + t / TPR, c0 = t % TPR;
  const size_t hb = static_cast<size_t>(a.req) * a.heads + h;
  float* sk = sm;
  float* sv = sk + n * D;
  float* sab = sv + n * D;
  ssm_stage_buffer<D>(a, hb, n, sk, sv, sab);
  float S[CPT];
  ssm_load_rows<D>(S, a.ckpt + hb * D * D, row, c0);
  __syncthreads();
  ssm_replay<D>(S, sk, sv, sab, n, nullptr, 0, nullptr, row, c0);
  ssm_store_rows<D>(S, a.state_out + static_cast<size_t>(h) * D * D, row, c0);
}

}  // namespace vsd
