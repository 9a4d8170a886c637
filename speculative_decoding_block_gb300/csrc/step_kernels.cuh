// step_kernels.cuh -- the light kernels of the verify step: embedding gather,
// the fused argmax / prefix-accept / KV commit, and helpers of the component
// entry points.
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

struct EmbedArgs {
  const uint16_t* embed;  // [V][H] bf16
  int vocab, hidden;
  const int* seq_lens;    // [B]
  const int* pending;     // [B]
  const int* drafts;      // [B][16]
  int max_tokens;
  float* x;               // [M][H] residual stream
  __half* x16;            // [M][H] f16 copy (first GEMM's input), hi = f16(x)
  size_t x16_lo;          // elements from a hi value to its lo copy f16(x - hi) (0: hi only)
  float* ssq;             // [ceil(H/128)][ssq_ld] sums of squares per 128-feature slice
  int ssq_ld;
  int* ctx_len;           // [B] validated context length (0 if invalid)
  int* req_ok;            // [B] 1 if seq_len and pending token are valid
  unsigned long long* keys;  // [M] argmax keys of the step, cleared here
  float* hidden0;         // optional [M][H]
  // draft mode (anchor != nullptr): row 0 of request b is anchor[b] (the
  // target's last residual row, fp32 [B][H]) and rows 1..16 embed mask_token;
  // pending and drafts are not read
  const float* anchor;
  int mask_token;
  int* status;
  Trace trace;
};

constexpr int kMaxSlices = 128;  // hidden <= 128 * 128

// One CTA (128 threads) per row b*17 + j: token = pending (j = 0) or draft j-1.
// The row's RMSNorm is not applied here: the consuming GEMM scales its
// result per token by 1/sqrt(mean(x^2) + eps), from the sums of squares
// written here per 128-feature slice.
__global__ void __launch_bounds__(128) embed_kernel(const EmbedArgs a) {
  __shared__ float part[kMaxSlices][4];
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) trace_start(a.trace);
  const int row = blockIdx.x, b = row / kRows, j = row % kRows;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const bool draft = a.anchor != nullptr;
  const int L = a.seq_lens[b];
  const bool idle = L == kIdleSlot;  // an empty slot: computed on, never committed, not an error
  int tok = draft ? a.mask_token : (j == 0 ? a.pending[b] : a.drafts[b * kBlock + j - 1]);
  const bool tok_ok = tok >= 0 && tok < a.vocab;
  if (!tok_ok) {
    if (t == 0 && !idle) atomicOr(a.status, VSD_DEV_BAD_TOKEN);
    tok = 0;
  }
  if (t == 0) {
    a.keys[row] = 0ull;
    if (j == 0) {
      const bool ok = L >= 0 && L + kRows <= a.max_tokens;
      if (!ok && !idle) atomicOr(a.status, VSD_DEV_BAD_SEQLEN);
      a.ctx_len[b] = ok ? L : 0;
      a.req_ok[b] = (ok && tok_ok) ? 1 : 0;
    }
  }
  const uint16_t* e = a.embed + static_cast<size_t>(tok) * a.hidden;
  const float* anchor_row = (draft && j == 0) ? a.anchor + static_cast<size_t>(b) * a.hidden : nullptr;
  const size_t o = static_cast<size_t>(row) * a.hidden;
  const int slices = (a.hidden + 127) / 128;
  for (int k0 = 0; k0 < slices; k0 += 8) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {  // loads first
      const int i = (k0 + k) * 128 + t;
      v[k] = (k0 + k < slices && i < a.hidden)
                 ? (anchor_row ? anchor_row[i] : __uint_as_float(static_cast<uint32_t>(e[i]) << 16))
                 : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = (k0 + k) * 128 + t;
      if (k0 + k < slices && i < a.hidden) {
        a.x[o + i] = v[k];
        const __half hi = __float2half_rn(v[k]);
        a.x16[o + i] = hi;
        if (a.x16_lo) a.x16[o + i + a.x16_lo] = __float2half_rn(v[k] - __half2float(hi));
        if (a.hidden0) a.hidden0[o + i] = v[k];
      }
      float sq = v[k] * v[k];
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, m);
      if (lane == 0 && k0 + k < slices) part[k0 + k][warp] = sq;
    }
  }
  __syncthreads();
  if (t < slices)
    a.ssq[static_cast<size_t>(t) * a.ssq_ld + row] = part[t][0] + part[t][1] + part[t][2] + part[t][3];
  if (t == 0) trace_end(a.trace, 1);
}

// Validation of the caller's per-request state (component entry points that
// run without the embedding kernel).
__global__ void validate_requests_kernel(const int* seq_lens, const int* pending, int B, int vocab, int max_tokens,
                                         int* ctx_len, int* req_ok, int* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int L = seq_lens[b], p = pending[b];
  const bool ok = L >= 0 && L + kRows <= max_tokens;
  if (!ok) atomicOr(status, VSD_DEV_BAD_SEQLEN);
  if (p < 0 || p >= vocab) atomicOr(status, VSD_DEV_BAD_TOKEN);
  ctx_len[b] = ok ? L : 0;
  req_ok[b] = (ok && p >= 0 && p < vocab) ? 1 : 0;
}

// Test-only: one CTA waits, with the kernels' bounded-wait pattern, on a
// global flag and on a shared-memory mbarrier that nothing ever completes;
// after `limit` SM cycles each gives up, records VSD_DEV_TIMEOUT and the
// kernel returns (no copy or MMA is in flight, so it exits cleanly).
__global__ void wait_probe_kernel(const int* flag, long long limit, int* status) {
  __shared__ uint64_t never_full;
  if (threadIdx.x == 0) {
    mbar_init(&never_full, 1);
    fence_mbar_init();
  }
  __syncthreads();
  bool gave_up = false;
  if (threadIdx.x == 0 || threadIdx.x == 32) {
    const long long t0 = clock64();
    while (threadIdx.x == 0 ? ld_acquire_gpu(flag) == 0 : !mbar_test_wait(&never_full, 0)) {
      if (clock64() - t0 > limit) {
        gave_up = true;
        break;
      }
    }
  }
  if (gave_up) atomicOr(status, VSD_DEV_TIMEOUT);
}

struct CommitArgs {
  int vocab, layers, n_kv, hd, batch_cap, num_pages, pages_per_req;
  const unsigned long long* keys;  // [B*17]
  const int* decided;             // optional [B][18] (stochastic verification): a, then out tokens -- used instead of keys
  const int* drafts;              // [B][16]
  const int* ctx_len;             // [B] validated committed length
  const int* req_ok;              // [B]
  int* seq_lens;                  // [B] out (written by the layer-0 CTA only)
  int* pending;                   // [B] out
  int* accepted;                  // [B]
  int* out_tokens;                // [B][17]
  const int* page_table;          // [max_batch][ppr]
  const __nv_bfloat16* k_new;     // [layers][Bcap][n_kv][32][hd]
  const __nv_bfloat16* v_new;
  __nv_bfloat16* k_pool;          // [layers][pages][n_kv][16][hd]
  __nv_bfloat16* v_pool;
  // optional: the residual row of the last accepted position, x[b*17 + a],
  // copied to anchor[b] ([B][hidden] fp32) -- the drafter's conditioning input
  const float* x;
  float* anchor;
  int hidden;
  int* status;
  Trace trace;
};

// Greedy tokens from the argmax keys, accepted length a = first draft that
// differs (16 if none); CTA (b, l) moves the K/V rows 0..a of layer l from
// scratch into request b's cache pages at positions L..L+a; CTA (b, 0) also
// writes the outputs and then seq_len = L + a + 1, pending = g_a.  All CTAs
// read L from the step's validated copy, so the in-place update races with
// nothing.  A request is rejected (accepted = -1, outputs -1, cache and
// lengths untouched) when its length or a token was out of range, when a
// page of its rows [0, L + 17) lies outside the pool (the attention read its
// context through them), or when the step's kernel gave up on a wait (its
// outputs are then incomplete): then every request of the step is rejected.
__global__ void __launch_bounds__(256) accept_commit_kernel(const CommitArgs a) {
  __shared__ int g[kRows];
  __shared__ int page[kRows];
  __shared__ int s_acc, s_valid;
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x, l = blockIdx.y, t = threadIdx.x;
  if (t == 0 && l == 0) trace_start(a.trace);
  const int L = a.ctx_len[b];
  const bool timed_out = (*reinterpret_cast<volatile int*>(a.status) & VSD_DEV_TIMEOUT) != 0;
  int bad_page = 0;
  for (int i = t; i < (L + kRows + kPage - 1) / kPage; i += blockDim.x) {
    const int pg = a.page_table[b * a.pages_per_req + i];
    bad_page |= (pg < 0 || pg >= a.num_pages) ? 1 : 0;
  }
  bad_page = __syncthreads_or(bad_page);
  if (t < 32) {
    int gt = -1, dt = -1;
    bool bad = false;
    if (t < kRows) {
      if (a.decided) {
        const int dacc = a.decided[b * (kRows + 1)];
        gt = a.decided[b * (kRows + 1) + 1 + t];
        if (t <= dacc && (gt < 0 || gt >= a.vocab)) bad = true;
        if (t > dacc) gt = -1;
      } else {
        const unsigned long long k = a.keys[b * kRows + t];
        gt = k ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull)) : -1;
        if (gt < 0 || gt >= a.vocab) bad = true;
      }
      g[t] = gt;
    }
    if (t < kRows) page[t] = a.page_table[b * a.pages_per_req + (L + t) / kPage];
    if (t < kBlock) {
      dt = a.drafts[b * kBlock + t];
      if (dt < 0 || dt >= a.vocab) bad = true;
    }
    const unsigned mism = __ballot_sync(0xFFFFFFFFu, t < kBlock && dt != gt);
    const unsigned badm = __ballot_sync(0xFFFFFFFFu, bad);
    if (t == 0) {
      const int acc0 = a.decided ? a.decided[b * (kRows + 1)] : (mism ? (__ffs(mism) - 1) : kBlock);
      if (bad_page && l == 0) atomicOr(a.status, VSD_DEV_BAD_PAGE);
      s_valid = (badm == 0 && a.req_ok[b] && !bad_page && !timed_out) ? 1 : 0;
      s_acc = acc0;
    }
  }
  __syncthreads();
  const int acc = s_acc;
  if (!s_valid) {
    if (l == 0) {
      if (t < kRows) a.out_tokens[b * kRows + t] = -1;
      if (t == 0) a.accepted[b] = -1;
    }
    if (t == 0) trace_end(a.trace, 1);
    return;
  }
  // KV commit of layer l: rows 0..acc, K and V, every head, 16-byte pieces
  const int pieces = a.hd / 8;
  const int total = (acc + 1) * 2 * a.n_kv * pieces;
#pragma unroll 4
  for (int idx = t; idx < total; idx += blockDim.x) {
    const int piece = idx % pieces;
    int rest = idx / pieces;
    const int h = rest % a.n_kv;
    rest /= a.n_kv;
    const int kv = rest & 1;
    const int j = rest >> 1;
    const int pos = L + j;
    const __nv_bfloat16* src =
        (kv ? a.v_new : a.k_new) + ((((static_cast<size_t>(l) * a.batch_cap + b) * a.n_kv + h) * 32 + j) * a.hd) +
        piece * 8;
    __nv_bfloat16* dst = (kv ? a.v_pool : a.k_pool) +
                         ((((static_cast<size_t>(l) * a.num_pages + page[j]) * a.n_kv + h) * kPage + pos % kPage) *
                          a.hd) +
                         piece * 8;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
  if (l == 0) {
    if (t < kRows) a.out_tokens[b * kRows + t] = t <= acc ? g[t] : -1;
    if (t == 0) {
      a.accepted[b] = acc;
      a.seq_lens[b] = L + acc + 1;
      a.pending[b] = g[acc];
    }
    if (a.anchor) {
      const float* src = a.x + (static_cast<size_t>(b) * kRows + acc) * a.hidden;
      for (int i = t; i < a.hidden; i += blockDim.x) a.anchor[static_cast<size_t>(b) * a.hidden + i] = src[i];
    }
  }
  if (t == 0) trace_end(a.trace, 1);
}

// ------------------------------------------------------------------ device-resident loop
// Slots of the loop hold requests of a queue; request q's context sits in
// cache slot first_queued + q (its page-table row), written by the caller.
struct LoopArgs {
  int B, Q, out_cap, hidden, pages_per_req, first_queued;
  int* slot_req;          // [B] request in slot b, -1 empty
  int* next_req;          // [1] queue head
  const int* req_len;     // [Q] committed length at admission
  const int* req_pending; // [Q] pending token at admission
  const int* req_budget;  // [Q] tokens to generate
  const float* req_anchor;// [Q][hidden] anchor row at admission
  int* req_generated;     // [Q] out
  int* req_admit_iter;    // [Q] out: loop iteration of admission (-1 never)
  int* req_out;           // [Q][out_cap] out
  int* seq_lens;          // [B] slot state (kIdleSlot when empty)
  int* pending;           // [B]
  const int* accepted;    // [B] of the step
  const int* out_tokens;  // [B][17] of the step
  int* page_table;        // [max_batch][ppr]
  float* anchor;          // [max_batch][hidden] the cache's anchor rows
  int* iter;              // [1] loop iteration counter
  int* status;
};

// Before a step: retire requests that reached their budget, admit queued
// requests into empty slots in queue order (page-table row, length,
// pending token and anchor row of the request).  One CTA.
__global__ void __launch_bounds__(256) loop_schedule_kernel(const LoopArgs a) {
  __shared__ int admit_q[kMaxLoopSlots];
  __shared__ int head;
  pdl_wait();
  pdl_launch_dependents();
  const int t = threadIdx.x;
  if (t == 0) {
    head = *a.next_req;
    const int it = *a.iter;
    for (int b = 0; b < a.B; ++b) {
      int q = a.slot_req[b];
      if (q >= 0 && a.req_generated[q] >= a.req_budget[q]) q = -1;  // retired
      if (q < 0 && head < a.Q) {
        q = head++;
        a.req_admit_iter[q] = it;
        admit_q[b] = q;
      } else {
        admit_q[b] = -1;
      }
      a.slot_req[b] = q;
      if (q < 0) a.seq_lens[b] = kIdleSlot;
    }
    *a.next_req = head;
  }
  __syncthreads();
  for (int b = 0; b < a.B; ++b) {
    const int q = admit_q[b];
    if (q < 0) continue;
    for (int i = t; i < a.pages_per_req; i += blockDim.x)
      a.page_table[static_cast<size_t>(b) * a.pages_per_req + i] =
          a.page_table[static_cast<size_t>(a.first_queued + q) * a.pages_per_req + i];
    for (int i = t; i < a.hidden; i += blockDim.x)
      a.anchor[static_cast<size_t>(b) * a.hidden + i] = a.req_anchor[static_cast<size_t>(q) * a.hidden + i];
    if (t == 0) {
      a.seq_lens[b] = a.req_len[q];
      a.pending[b] = a.req_pending[q];
    }
  }
}

// After a step: append each busy slot's accepted tokens to its request's
// output (up to out_cap) and count them; advance the iteration counter.
__global__ void loop_collect_kernel(const LoopArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x, t = threadIdx.x;  // one warp per slot
  const int q = a.slot_req[b];
  if (q >= 0) {
    const int acc = a.accepted[b];
    const int g0 = a.req_generated[q];
    if (acc >= 0) {
      if (t <= acc && g0 + t < a.out_cap) a.req_out[static_cast<size_t>(q) * a.out_cap + g0 + t] = a.out_tokens[b * kRows + t];
      __syncwarp();
      if (t == 0) a.req_generated[q] = g0 + acc + 1;
    } else if (t == 0) {
      atomicOr(a.status, VSD_DEV_BAD_SEQLEN);  // a busy slot whose step was rejected
    }
  }
  if (b == 0 && t == 0) *a.iter += 1;
}

// ------------------------------------------------------------------ stochastic verification
struct SampleArgs {
  int vocab, hidden, n_tiles, m_alloc, ssq_slices;
  float inv_temp, inv_hidden, eps;
  // per (row, 128-row vocabulary tile): maximum m of y = logit / T * log2(e)
  // and sum of 2^(y - m)
  const float* tile_max;     // [M][n_tiles]
  const float* tile_sum;     // [M][n_tiles]
  const float* draft_logit;  // [M]
  const int* drafts;         // [B][16]
  const float* u_accept;     // [B][16]
  const float* u_sample;     // [B][17]
  const __half* head;        // the head's f16 tiles [vocab/128][hidden/64][128 x 64], MMA layout (as the GEMM reads them)
  int head_k_tiles;
  const __half* x16;         // [M][hidden] hi, lo copy m_alloc rows later: the head's input rows
  const float* ssq;          // [slices][m_alloc] sums of squares of the final residual rows
  int* decided;              // [B][18]: accepted count a, then out tokens 0..16 (-1 beyond a)
};

// One CTA (256 threads) per request.  Every weight is taken relative to its
// row's maximum, w(v) = 2^(y_v - M_j) with y = logit / T * log2(e) and M_j the
// row's largest y, so that no logit overflows or saturates the exponential:
// accept draft j while u_accept[j] < p_j(d_j) = w(d_j) / Z_j, Z_j = sum of
// w over the vocabulary (from the per-tile (max, sum) pairs); at the first
// rejection (or after 16 acceptances) sample row a by inverse CDF over
// token ids in increasing order, without the rejected draft: the vocabulary
// tile holding the target mass comes from the per-tile sums, its 128 logits
// are recomputed from the head rows.
__global__ void __launch_bounds__(256) sample_decide_kernel(const SampleArgs a) {
  __shared__ float red[256];
  __shared__ float z_row[kRows], m_row[kRows];
  __shared__ float w_tile[128];
  __shared__ int s_acc, s_tile, s_excl;
  __shared__ float s_base, s_target, s_we;
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x, t = threadIdx.x;
  const float c2 = a.inv_temp * kLog2e;
  // M_j, then Z_j: strided partials, then a fixed tree (deterministic)
  for (int j = 0; j < kRows; ++j) {
    const size_t r0 = static_cast<size_t>(b * kRows + j) * a.n_tiles;
    float mx = -INFINITY;
    for (int i = t; i < a.n_tiles; i += 256) mx = fmaxf(mx, a.tile_max[r0 + i]);
    red[t] = mx;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
      if (t < w) red[t] = fmaxf(red[t], red[t + w]);
      __syncthreads();
    }
    const float M = red[0];
    __syncthreads();
    float sum = 0.0f;
    for (int i = t; i < a.n_tiles; i += 256) sum += a.tile_sum[r0 + i] * ex2(a.tile_max[r0 + i] - M);
    red[t] = sum;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
      if (t < w) red[t] += red[t + w];
      __syncthreads();
    }
    if (t == 0) {
      z_row[j] = red[0];
      m_row[j] = M;
    }
    __syncthreads();
  }
  if (t == 0) {
    int acc = kBlock;
    for (int j = 0; j < kBlock; ++j) {
      const int d = a.drafts[b * kBlock + j];
      const float p =
          (d >= 0 && d < a.vocab) ? ex2(a.draft_logit[b * kRows + j] * c2 - m_row[j]) / z_row[j] : 0.0f;
      if (!(a.u_accept[b * kBlock + j] < p)) {
        acc = j;
        break;
      }
    }
    const int d = acc < kBlock ? a.drafts[b * kBlock + acc] : -1;
    const bool excl = d >= 0 && d < a.vocab;
    const float we = excl ? ex2(a.draft_logit[b * kRows + acc] * c2 - m_row[acc]) : 0.0f;
    s_acc = acc;
    s_excl = excl ? d : -1;
    s_we = we;
    s_target = a.u_sample[b * kRows + acc] * fmaxf(z_row[acc] - we, 0.0f);
  }
  __syncthreads();
  const int acc = s_acc, r = b * kRows + acc;
  const float M = m_row[acc];
  // the tile holding the target mass: chunk sums of consecutive tiles (the
  // draft's weight taken out of its tile), a scan of the 256 chunk sums,
  // then a scan inside the chunk
  const float* tm = a.tile_max + static_cast<size_t>(r) * a.n_tiles;
  const float* ts = a.tile_sum + static_cast<size_t>(r) * a.n_tiles;
  const int per = (a.n_tiles + 255) / 256;
  auto tile_w = [&](int i) {
    return ts[i] * ex2(tm[i] - M) - ((s_excl >= 0 && i == s_excl / 128) ? s_we : 0.0f);
  };
  {
    float sum = 0.0f;
    for (int i = t * per; i < min(a.n_tiles, (t + 1) * per); ++i) sum += tile_w(i);
    red[t] = sum;
  }
  __syncthreads();
  if (t == 0) {
    float run = 0.0f;
    int c = 255;
    for (int i = 0; i < 256; ++i) {
      if (run + red[i] >= s_target && red[i] > 0.0f) {
        c = i;
        break;
      }
      run += red[i];
    }
    int tile = min(a.n_tiles - 1, c * per + per - 1);
    for (int i = c * per; i < min(a.n_tiles, (c + 1) * per); ++i) {
      const float wi = tile_w(i);
      if (run + wi >= s_target && wi > 0.0f) {
        tile = i;
        break;
      }
      run += wi;
    }
    s_tile = tile;
    s_base = run;
  }
  __syncthreads();
  const int tile = s_tile;
  // the tile's 128 logits: two threads per head row, halves of the hidden size, 8 values per load
  float ss = 0.0f;
  for (int k = 0; k < a.ssq_slices; ++k) ss += a.ssq[static_cast<size_t>(k) * a.m_alloc + r];
  const float rs = 1.0f / sqrtf(ss * a.inv_hidden + a.eps);
  {
    const int i = t >> 1, half = t & 1;
    const int v = tile * 128 + i;
    float dot = 0.0f;
    if (v < a.vocab) {
      // 16-byte chunk q of head row v: tile (v / 128, q / 8), swizzled chunk (q % 8) of tile row v % 128
      const __half* wtiles = a.head + static_cast<size_t>(v >> 7) * a.head_k_tiles * 8192;
      const uint32_t wr = static_cast<uint32_t>(v & 127);
      const __half* xh = a.x16 + static_cast<size_t>(r) * a.hidden;
      const __half* xl = xh + static_cast<size_t>(a.m_alloc) * a.hidden;
      const int n8 = a.hidden / 8, h8 = n8 / 2;
      for (int q = half ? h8 : 0; q < (half ? n8 : h8); ++q) {
        const uint4 w4 =
            *reinterpret_cast<const uint4*>(wtiles + static_cast<size_t>(q >> 3) * 8192 + sw128_off(wr, q & 7) / 2);
        const uint4 h4 = reinterpret_cast<const uint4*>(xh)[q];
        const uint4 l4 = reinterpret_cast<const uint4*>(xl)[q];
        const __half2* w2 = reinterpret_cast<const __half2*>(&w4);
        const __half2* hh = reinterpret_cast<const __half2*>(&h4);
        const __half2* ll = reinterpret_cast<const __half2*>(&l4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 wf = __half22float2(w2[e]), hf = __half22float2(hh[e]), lf = __half22float2(ll[e]);
          dot += wf.x * (hf.x + lf.x) + wf.y * (hf.y + lf.y);
        }
      }
    }
    dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 1);
    if (half == 0) w_tile[i] = (v < a.vocab && v != s_excl) ? ex2(dot * rs * c2 - M) : 0.0f;
  }
  __syncthreads();
  if (t == 0) {
    float run = s_base;
    int tok = -1, last = -1;
    for (int i = 0; i < 128; ++i) {
      if (w_tile[i] <= 0.0f) continue;
      last = tile * 128 + i;
      run += w_tile[i];
      if (run >= s_target) {
        tok = last;
        break;
      }
    }
    if (tok < 0) tok = last;  // rounding: the mass ran out inside the tile
    int* dec = a.decided + b * (kRows + 1);
    dec[0] = acc;
    for (int j = 0; j < kRows; ++j)
      dec[1 + j] = j < acc ? a.drafts[b * kBlock + j] : (j == acc ? tok : -1);
  }
}

// Drafts from the argmax keys of a draft pass: drafts[b][j] = token of row
// b*17 + 1 + j (j = 0..15), -1 if the row has no key.
__global__ void draft_pick_kernel(const unsigned long long* keys, int B, int vocab, int* drafts, int* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= B * kBlock) return;
  const int b = i / kBlock, j = i % kBlock;
  const unsigned long long k = keys[b * kRows + 1 + j];
  int tok = k ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull)) : -1;
  if (tok < 0 || tok >= vocab) {
    atomicOr(status, VSD_DEV_BAD_TOKEN);
    tok = -1;
  }
  drafts[i] = tok;
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
