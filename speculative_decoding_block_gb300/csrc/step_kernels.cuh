// step_kernels.cuh -- the light kernels of the verify step: embedding gather
// with the first RMSNorm, RMSNorm, the fused argmax / prefix-accept / KV
// commit, and helpers of the component entry points.
#pragma once

#include "vsd_common.cuh"

namespace vsd {

__device__ __forceinline__ float block_sum_128(float v, float* red) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  const float s = red[0] + red[1] + red[2] + red[3];
  __syncthreads();
  return s;
}

// x / sqrt(mean(x^2) + eps) * gamma of one row held in x (global), written as f16.
__device__ __forceinline__ void rmsnorm_row(const float* x, int H, float eps, const float* gamma, __half* u,
                                            float* red) {
  float ss = 0.0f;
  for (int i = threadIdx.x; i < H; i += 128) ss += x[i] * x[i];
  ss = block_sum_128(ss, red);
  const float r = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
  for (int i = threadIdx.x; i < H; i += 128) u[i] = __float2half_rn(x[i] * r * gamma[i]);
}

struct EmbedArgs {
  const uint16_t* embed;  // [V][H] bf16
  int vocab, hidden;
  const int* seq_lens;    // [B]
  const int* pending;     // [B]
  const int* drafts;      // [B][16]
  int max_tokens;
  float eps;
  const float* gamma;
  float* x;               // [M][H] residual stream
  __half* u;              // [M][H] normalised (layer-0 input)
  int* ctx_len;           // [B] validated context length (0 if invalid)
  float* hidden0;         // optional [M][H]
  int* status;
};

// One CTA (128 threads) per row b*17 + j: token = pending (j = 0) or draft j-1.
__global__ void __launch_bounds__(128) embed_norm_kernel(const EmbedArgs a) {
  __shared__ float red[4];
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x, b = row / kRows, j = row % kRows;
  int tok = j == 0 ? a.pending[b] : a.drafts[b * kBlock + j - 1];
  if (tok < 0 || tok >= a.vocab) {
    if (threadIdx.x == 0) atomicOr(a.status, VSD_DEV_BAD_TOKEN);
    tok = 0;
  }
  if (j == 0 && threadIdx.x == 0) {
    const int L = a.seq_lens[b];
    const bool ok = L >= 0 && L + kRows <= a.max_tokens;
    if (!ok) atomicOr(a.status, VSD_DEV_BAD_SEQLEN);
    a.ctx_len[b] = ok ? L : 0;
  }
  const uint16_t* e = a.embed + static_cast<size_t>(tok) * a.hidden;
  float* x = a.x + static_cast<size_t>(row) * a.hidden;
  for (int i = threadIdx.x; i < a.hidden; i += 128) {
    const float v = __uint_as_float(static_cast<uint32_t>(e[i]) << 16);
    x[i] = v;
    if (a.hidden0) a.hidden0[static_cast<size_t>(row) * a.hidden + i] = v;
  }
  __syncthreads();
  rmsnorm_row(x, a.hidden, a.eps, a.gamma, a.u + static_cast<size_t>(row) * a.hidden, red);
}

__global__ void __launch_bounds__(128) rmsnorm_kernel(const float* x, int hidden, float eps, const float* gamma,
                                                      __half* u, float* copy_out) {
  __shared__ float red[4];
  pdl_wait();
  pdl_launch_dependents();
  const size_t row = blockIdx.x;
  if (copy_out)
    for (int i = threadIdx.x; i < hidden; i += 128) copy_out[row * hidden + i] = x[row * hidden + i];
  rmsnorm_row(x + row * hidden, hidden, eps, gamma, u + row * hidden, red);
}

struct CommitArgs {
  int vocab, layers, n_kv, hd, batch_cap, num_pages, pages_per_req, max_tokens;
  unsigned long long* keys;       // [B*17], reset to 0 after use
  const int* drafts;              // [B][16]
  int* seq_lens;                  // [B] in/out
  int* pending;                   // [B] in/out
  int* accepted;                  // [B]
  int* out_tokens;                // [B][17]
  const int* page_table;          // [max_batch][ppr]
  const __nv_bfloat16* k_new;     // [layers][Bcap][n_kv][32][hd]
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_pool;          // [layers][pages][n_kv][16][hd]
  __nv_bfloat16* v_pool;
  int* status;
};

// Greedy tokens from the argmax keys, accepted length = first draft that
// differs (16 if none), outputs, then the K/V rows 0..a of the block move from
// scratch into the request's cache pages at positions L..L+a, and finally
// seq_len += a+1 and pending = g_a.  One CTA per request.
__global__ void __launch_bounds__(256) accept_commit_kernel(const CommitArgs a) {
  __shared__ int g[kRows];
  __shared__ int s_acc, s_valid, s_len;
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x, t = threadIdx.x;
  if (t < 32) {
    int gt = -1, dt = -1;
    bool bad = false;
    if (t < kRows) {
      const unsigned long long k = a.keys[b * kRows + t];
      gt = k ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull)) : -1;
      if (gt < 0 || gt >= a.vocab) bad = true;
      g[t] = gt;
    }
    if (t < kBlock) {
      dt = a.drafts[b * kBlock + t];
      if (dt < 0 || dt >= a.vocab) bad = true;
    }
    const unsigned mism = __ballot_sync(0xFFFFFFFFu, t < kBlock && dt != gt);
    const unsigned badm = __ballot_sync(0xFFFFFFFFu, bad);
    if (t == 0) {
      const int L = a.seq_lens[b];
      const int p = a.pending[b];
      const bool ok = badm == 0 && L >= 0 && L + kRows <= a.max_tokens && p >= 0 && p < a.vocab;
      s_valid = ok ? 1 : 0;
      s_acc = mism ? (__ffs(mism) - 1) : kBlock;
      s_len = L;
    }
  }
  __syncthreads();
  const int acc = s_acc, L = s_len;
  if (!s_valid) {
    if (t < kRows) a.out_tokens[b * kRows + t] = -1;
    if (t == 0) a.accepted[b] = -1;
    __syncthreads();
    if (t < kRows) a.keys[b * kRows + t] = 0;
    return;
  }
  if (t < kRows) a.out_tokens[b * kRows + t] = t <= acc ? g[t] : -1;
  if (t == 0) a.accepted[b] = acc;
  // KV commit: rows 0..acc of every layer / K,V / head, 16-byte pieces
  const int pieces = a.hd / 8;
  const int per_row = 2 * a.n_kv * pieces;
  const int total = (acc + 1) * a.layers * per_row;
  for (int idx = t; idx < total; idx += blockDim.x) {
    const int piece = idx % pieces;
    int rest = idx / pieces;
    const int h = rest % a.n_kv;
    rest /= a.n_kv;
    const int kv = rest & 1;
    rest >>= 1;
    const int j = rest % (acc + 1);
    const int l = rest / (acc + 1);
    const int pos = L + j;
    int page = a.page_table[b * a.pages_per_req + pos / kPage];
    if (page < 0 || page >= a.num_pages) {
      atomicOr(a.status, VSD_DEV_BAD_PAGE);
      continue;
    }
    const __nv_bfloat16* src = (kv ? a.v_new : a.k_new) +
                               ((((static_cast<size_t>(l) * a.batch_cap + b) * a.n_kv + h) * 32 + j) * a.hd) + piece * 8;
    __nv_bfloat16* dst = (kv ? a.v_pool : a.k_pool) +
                         ((((static_cast<size_t>(l) * a.num_pages + page) * a.n_kv + h) * kPage + pos % kPage) * a.hd) +
                         piece * 8;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
  __syncthreads();
  if (t == 0) {
    a.seq_lens[b] = L + acc + 1;
    a.pending[b] = g[acc];
  }
  if (t < kRows) a.keys[b * kRows + t] = 0;
}

// Argmax keys of given float32 logits (component entry point): one CTA per row.
__global__ void __launch_bounds__(256) logits_argmax_kernel(const float* logits, int vocab, unsigned long long* keys) {
  __shared__ unsigned long long red[8];
  const size_t row = blockIdx.x;
  unsigned long long best = 0;
  for (int i = threadIdx.x; i < vocab; i += 256) {
    const unsigned long long k = argmax_key(logits[row * vocab + i], static_cast<uint32_t>(i));
    best = k > best ? k : best;
  }
  for (int m = 16; m >= 1; m >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, m);
    best = o > best ? o : best;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) best = red[w] > best ? red[w] : best;
    keys[row] = best;
  }
}

// Block rows [layers?][B][17][n_kv][hd] -> scratch [layer][Bcap][n_kv][32][hd].
__global__ void scatter_block_rows_kernel(const __nv_bfloat16* src, int layers, int B, int n_kv, int hd,
                                          int batch_cap, int layer0, __nv_bfloat16* dst) {
  const size_t n = static_cast<size_t>(layers) * B * kRows * n_kv * hd;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int d = i % hd;
    size_t r = i / hd;
    const int h = r % n_kv;
    r /= n_kv;
    const int j = r % kRows;
    r /= kRows;
    const int b = r % B;
    const int l = static_cast<int>(r / B) + layer0;
    dst[(((static_cast<size_t>(l) * batch_cap + b) * n_kv + h) * 32 + j) * hd + d] = src[i];
  }
}

// q [B][17][n_q][hd] -> attention tile [B][n_kv][128][hd], row = j*group + hq.
__global__ void scatter_q_kernel(const __nv_bfloat16* q, int B, int n_q, int n_kv, int hd, __nv_bfloat16* tile) {
  const int group = n_q / n_kv;
  const size_t n = static_cast<size_t>(B) * kRows * n_q * hd;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int d = i % hd;
    size_t r = i / hd;
    const int hh = r % n_q;
    r /= n_q;
    const int j = r % kRows;
    const int b = static_cast<int>(r / kRows);
    tile[((static_cast<size_t>(b) * n_kv + hh / group) * 128 + j * group + hh % group) * hd + d] = q[i];
  }
}

__global__ void clamp_ctx_kernel(const int* seq_lens, int B, int max_tokens, int* ctx_len, int* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) {
    const int L = seq_lens[b];
    const bool ok = L >= 0 && L + kRows <= max_tokens;
    if (!ok) atomicOr(status, VSD_DEV_BAD_SEQLEN);
    ctx_len[b] = ok ? L : 0;
  }
}

// Cache rows of one request <-> dense [layers][count][n_kv][hd] (write = 1: dense -> cache).
__global__ void kv_rows_kernel(__nv_bfloat16* pool, const int* page_table, int ppr, int num_pages, int layers,
                               int n_kv, int hd, int req, int start, int count, __nv_bfloat16* dense, int write,
                               int* status) {
  const size_t n = static_cast<size_t>(layers) * count * n_kv * hd;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int d = i % hd;
    size_t r = i / hd;
    const int h = r % n_kv;
    r /= n_kv;
    const int t = r % count;
    const int l = static_cast<int>(r / count);
    const int pos = start + t;
    const int page = page_table[req * ppr + pos / kPage];
    if (page < 0 || page >= num_pages) {
      atomicOr(status, VSD_DEV_BAD_PAGE);
      continue;
    }
    __nv_bfloat16* c = pool + (((static_cast<size_t>(l) * num_pages + page) * n_kv + h) * kPage + pos % kPage) * hd + d;
    if (write) *c = dense[i];
    else dense[i] = *c;
  }
}

__global__ void check_pages_kernel(const int* table, size_t n, int num_pages, int* status) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    if (table[i] < 0 || table[i] >= num_pages) atomicOr(status, VSD_DEV_BAD_PAGE);
}

}  // namespace vsd
