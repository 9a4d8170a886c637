// gemm.cuh -- weight-streaming GEMM for the verify rows on tcgen05 / TMEM.
//
// Computes, for one weight matrix W [N, K] in BF16, FP8 E4M3 (per-row fp32
// scale) or NVFP4 (E2M1 values, E4M3 scale per 16 k, fp32 tensor scale),
//     Y[t, n] = sum_k X[t, k] * W[n, k]
// over the M = 17 * batch token rows X (f16, row-major [M, K]).
//
// Swap-AB: the weight tile is the 128-row A operand and the tokens are the
// MMA's N dimension, so one CTA covers 128 output features x n_tok tokens.
// Weight tiles arrive by TMA (BF16 matrices, repacked once as f16 when the
// model is created: tiled tensor copy with the 128-byte swizzle straight into
// the MMA operand; FP8 / NVFP4: one 1-D bulk copy of a pre-packed tile,
// expanded exactly to f16 in shared memory -- E4M3 and E2M1 x E4M3 values
// are all exact f16 numbers).  Activation tiles arrive by TMA with the same
// swizzle.  The fp32 accumulator sits in TMEM (double-buffered so the
// epilogue of one tile overlaps the MMAs of the next).  Per-row (FP8) and
// per-tensor (NVFP4) fp32 scales are applied in the epilogue.
//
// Warp roles (320 threads): warps 0-3 expand weights into the f16 A tile,
// warps 4-7 run the epilogue (warp w reads TMEM lanes 32*(w%4)..), warp 8
// issues TMA, warp 9 allocates TMEM and issues the MMAs.
//
// When the output tiles alone cannot fill the GPU, the k dimension is split
// over a thread-block cluster of cs CTAs: rank r accumulates k tiles
// [r*kps, (r+1)*kps), stores its partial tile in shared memory, and every CTA
// then sums the cs partials of its own column groups straight from the peers'
// shared memory (distributed shared memory), in rank order -- deterministic,
// no global-memory round trip.  Clusters are persistent over output tiles.
//
// The RMSNorm in front of QKV, gate/up and lm_head is folded into the GEMM:
// the input rows arrive unnormalised (f16 copy of the fp32 residual) and the
// result of token t is scaled by r_t = 1/sqrt(sum(x_t^2)/hidden + eps), from
// sums of squares that the residual epilogue writes per 128-feature tile.
//
// Epilogues fuse the neighbouring element-wise steps of the decoder layer
// ("The Inference Stack Behind OCRia", section "Avoiding unnecessary memory
// transfers": intermediates stay on chip):
//   STORE  : y = acc * scale                       (component entry point)
//   RESID  : x += acc * scale; f16 copy of x; sums of squares of x per tile
//   QKV    : RoPE on q and k, q -> attention tile layout, k / v -> block scratch
//   SILU   : silu(gate) * up -> f16 MLP activation (gate/up rows interleaved)
//   ARGMAX : per token, max over vocab rows -> 64-bit argmax key (atomicMax)
#pragma once

#include <type_traits>

#include "vsd_common.cuh"

namespace vsd {

enum WFmt { W_BF16 = 0, W_FP8 = 1, W_NVFP4 = 2 };
enum Epi { EPI_STORE = 0, EPI_RESID = 1, EPI_QKV = 2, EPI_SILU = 3, EPI_ARGMAX = 4, EPI_SAMPLE = 5 };

constexpr int kGemmThreads = 320;
constexpr int kTileN = 128;   // weight rows per tile (MMA M)
constexpr int kActBoxes = 16;  // activation box heights 16..256 rows (MMA N)
constexpr int kTileK = 64;    // k per stage (one 128-byte swizzle row of f16)
constexpr uint32_t kFp8TileBytes = kTileN * kTileK;                  // 8192
constexpr uint32_t kFp4ValBytes = kTileN * kTileK / 2;               // 4096
constexpr uint32_t kFp4TileBytes = kFp4ValBytes + kTileN * kTileK / 16;  // 4608

__host__ __device__ constexpr uint32_t raw_region_bytes(int wf) {
  return wf == W_FP8 ? 8192u : (wf == W_NVFP4 ? 5120u : 0u);
}

struct GemmArgs {
  // weights
  const uint8_t* w_tiles;  // FP8 / NVFP4: [n_tiles][k_tiles][tile bytes]
  const float* row_scale;  // FP8 / NVFP4: fp32 per packed row (row scale, or tensor scale of its matrix)
  int n_rows;              // valid packed rows
  int n_tiles, k_tiles;
  int tok_tiles, n_tok;    // token tiles, tokens per tile (MMA N)
  int cs, kps;             // cluster size = k splits, k tiles per split
  int m_tokens;            // valid token rows
  int rd, da, db;          // depths of the weight / expanded-weight / activation rings
  // Activations are pairs of f16 rows, hi = f16(x) and lo = f16(x - hi), so
  // that the 16-bit MMA inputs carry about 22 significant bits: the
  // activation map holds the lo rows act_lo_rows rows after the hi rows
  // (0: hi only, one MMA per k step instead of two).  Epilogues that write
  // activations (x16_out, act_out, q_tile) put the lo copy out_lo elements
  // after the hi copy (0: hi only).
  int act_lo_rows;
  size_t out_lo;
  int r_alias;             // split-K buffer shares the rings' space (host sets it when a CTA has one item)
  // RMSNorm of the input rows, folded in as a per-token scale of the result:
  // r[t] = 1 / sqrt(sum_i ssq_in[i][t] / hidden + eps)  (ssq_in == nullptr: no scale)
  const float* ssq_in;
  int n_ssq, ssq_ld;
  float inv_hidden, eps;
  // STORE / RESID
  float* out_f32;
  int ld_out;
  __half* x16_out;         // RESID: f16 copy of the updated rows (next GEMM's input)
  float* ssq_out;          // RESID: [tile][ssq_ld] sum of squares of the updated rows per 128-feature tile
  float* hidden_out;       // RESID (optional): copy of the updated rows
  // layer l of a multi-layer launch writes its block K / V and its hidden
  // rows this many elements after layer 0's (0: single-layer launches)
  size_t kv_layer_stride, hidden_layer_stride;
  // QKV
  __nv_bfloat16* q_tile;   // [B][n_kv][128][hd]
  __nv_bfloat16* k_new;    // [B][n_kv][32][hd] (this layer)
  __nv_bfloat16* v_new;
  const int* ctx_len;      // [B]
  const float2* rope;      // [positions][hd/2] (cos, sin)
  int n_q, n_kv, head_dim;
  // SILU
  __half* act_out;         // [rows][ffn]
  int ffn;
  // ARGMAX
  unsigned long long* keys;  // [M]
  float* logits;             // optional [M][vocab] (ARGMAX, SAMPLE)
  // SAMPLE: per (token row, 128-row vocabulary tile) the maximum m of
  // y = logit / T * log2(e) and the sum of 2^(y - m), and the logit of each
  // row's draft token (rows j < 16 of a request)
  float inv_temp;
  const int* drafts;         // [B][16]
  float* tile_max;           // [M][n_tiles]
  float* tile_sum;           // [M][n_tiles]
  float* draft_logit;        // [M]
  int* status;
  Trace trace;
};

// Shared memory rings (sizes chosen by the host):
//   W ring (rd slots): weight tiles as loaded -- f16 tiles (16 KB, MMA-ready)
//          or raw FP8 (8 KB) / NVFP4 (4.5 KB) tiles; deep enough to hold a
//          CTA's whole weight stream, so it fills before the grid-dependency
//          wait while the previous kernel still runs;
//   A ring (da slots, FP8 / NVFP4 only): 16 KB f16 expansions of raw tiles;
//   B ring (db slots): activation tiles, n_tok x 128 bytes;
//   R: split-K exchange buffer (cs > 1: n_tok columns x (128 + 4) fp32,
//      column-major so a warp's read of one column from a peer is one
//      contiguous 128-byte segment); then the control block.
struct GemmSmem {
  uint32_t a_off, b_off, b_bytes, w_off, w_bytes, r_off, r_ld, ctrl_off;
};

__host__ __device__ inline uint32_t weight_slot_bytes(int wf) {
  return wf == W_BF16 ? 16384u : (wf == W_FP8 ? kFp8TileBytes : kFp4TileBytes);
}

__host__ __device__ inline GemmSmem gemm_smem_layout(int wf, int n_tok, int rd, int da, int db, int cs,
                                                    bool lo, bool r_alias) {
  GemmSmem s;
  s.w_bytes = weight_slot_bytes(wf);
  s.b_bytes = static_cast<uint32_t>(n_tok) * 128u * (lo ? 2u : 1u);  // hi tile, then lo tile
  uint32_t off = 0;
  if (wf == W_BF16) {  // weight slots are MMA operands: 1024-byte aligned, first
    s.w_off = 0;
    off = s.w_bytes * rd;
    s.a_off = 0;
  } else {
    s.a_off = 0;
    off = 16384u * da;
  }
  s.b_off = off;
  off += s.b_bytes * db;
  if (wf != W_BF16) {
    s.w_off = off;
    off += s.w_bytes * rd;
    off = (off + 1023u) & ~1023u;
  }
  s.r_ld = 128u + 4u;
  const uint32_t r_bytes = cs > 1 ? ((static_cast<uint32_t>(n_tok) * s.r_ld * 4u + 1023u) & ~1023u) : 0u;
  if (r_alias) {
    // one item per CTA: the rings are idle once its accumulator is complete,
    // so the split-K exchange buffer reuses their space
    s.r_off = 0;
    s.ctrl_off = off > r_bytes ? off : r_bytes;
  } else {
    s.r_off = off;
    s.ctrl_off = off + r_bytes;
  }
  return s;
}

// control block: barriers (1 KB), per-warp argmax keys [2][2][4][16] (2 KB),
// running argmax keys (8 KB), sums of squares (4 KB), per-token row scales
// (1 KB), per-token positions (1 KB, QKV)
constexpr uint32_t kCtrlT = 1024, kCtrlBest = kCtrlT + 2048, kCtrlSq = kCtrlBest + 8192, kCtrlRs = kCtrlSq + 4096,
                   kCtrlPos = kCtrlRs + 1024;
constexpr int kBestCap = 1024;  // token columns whose running argmax fits in shared memory
constexpr int kMaxRd = 32, kMaxDb = 16, kMaxDa = 4;
__host__ __device__ inline uint32_t gemm_ctrl_bytes() { return kCtrlPos + 1024u; }
__host__ __device__ inline uint32_t gemm_smem_bytes(int wf, int n_tok, int rd, int da, int db, int cs, bool lo,
                                                    bool r_alias) {
  return 1024u + gemm_smem_layout(wf, n_tok, rd, da, db, cs, lo, r_alias).ctrl_off + gemm_ctrl_bytes();
}

// Iterates over the (item, k-tile) sequence of one CTA: items (tile, token
// tile) are dealt to clusters; the CTA of rank r covers k tiles
// [r * kps, (r + 1) * kps) of every item.
struct ItemIter {
  int item, total, stride, kt, kt_begin, kt_end;
  const GemmArgs* a;
  __device__ ItemIter(const GemmArgs* args, int first, int stride_, int total_, int rank)
      : item(first), total(total_), stride(stride_), a(args) {
    kt_begin = rank * args->kps;
    kt_end = min(args->k_tiles, kt_begin + args->kps);
    kt = kt_begin;
  }
  __device__ bool done() const { return item >= total || kt_begin >= kt_end; }
  __device__ bool first_k() const { return kt == kt_begin; }
  __device__ bool last_k() const { return kt + 1 == kt_end; }
  __device__ int tile() const { return item / a->tok_tiles; }
  __device__ int tok_tile() const { return item % a->tok_tiles; }
  __device__ void next() {
    if (++kt >= kt_end) {
      item += stride;
      kt = kt_begin;
    }
  }
};

template <int WF, int NT>
__device__ __forceinline__ void expand_weights(uint8_t* __restrict__ a_tile, const uint8_t* __restrict__ raw,
                                               int t) {
  // 1024 chunks of 8 f16 (16 bytes); thread t of NT handles chunks t + NT i.
  // All raw words are loaded first so that the loads overlap each other.
  constexpr int N = 1024 / NT;
  if constexpr (WF == W_FP8) {
    uint2 v[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int q = t + NT * i;
      v[i] = *reinterpret_cast<const uint2*>(raw + (q >> 3) * 64 + (q & 7) * 8);
    }
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int q = t + NT * i;
      uint4 o;
      o.x = e4m3x2_to_f16x2(static_cast<uint16_t>(v[i].x & 0xFFFF));
      o.y = e4m3x2_to_f16x2(static_cast<uint16_t>(v[i].x >> 16));
      o.z = e4m3x2_to_f16x2(static_cast<uint16_t>(v[i].y & 0xFFFF));
      o.w = e4m3x2_to_f16x2(static_cast<uint16_t>(v[i].y >> 16));
      *reinterpret_cast<uint4*>(a_tile + sw128_off(q >> 3, q & 7)) = o;
    }
  } else {
    uint32_t v[N], sb[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int q = t + NT * i;
      const int r = q >> 3, c = q & 7;
      v[i] = *reinterpret_cast<const uint32_t*>(raw + r * 32 + c * 4);
      sb[i] = raw[kFp4ValBytes + r * 4 + (c >> 1)];
    }
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int q = t + NT * i;
      const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint16_t>(sb[i] | (sb[i] << 8)));
      uint32_t h[4];
      e2m1x8_to_f16x8(v[i], h);
      const __half2 sc = *reinterpret_cast<const __half2*>(&s2);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        __half2 x = *reinterpret_cast<__half2*>(&h[j]);
        x = __hmul2(x, sc);  // exact: both factors have <= 4 significant bits
        h[j] = *reinterpret_cast<uint32_t*>(&x);
      }
      *reinterpret_cast<uint4*>(a_tile + sw128_off(q >> 3, q & 7)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
  }
}

__device__ __forceinline__ float shfl_xor_any(float v, int m) { return __shfl_xor_sync(0xFFFFFFFFu, v, m); }
__device__ __forceinline__ unsigned long long shfl_xor_any(unsigned long long v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

// Reduce-scatter of 16 per-lane values over the 32 lanes of a warp: after
// four halving exchanges (lane bits 4..1) and one final pair exchange, lane L
// holds the combination over all 32 lanes of element
// T(L) = 8*b4 + 4*b3 + 2*b2 + b1 (lanes L and L^1 hold the same element).
// 16 shuffles instead of 16 x 5 for sixteen butterfly reductions.
template <typename T, typename Op>
__device__ __forceinline__ T warp_reduce_scatter16(const T (&x)[16], int lane, Op op) {
  T y[8], z[4], w[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const T keep = b4 ? x[k + 8] : x[k], send = b4 ? x[k] : x[k + 8];
    y[k] = op(keep, shfl_xor_any(send, 16));
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const T keep = b3 ? y[k + 4] : y[k], send = b3 ? y[k] : y[k + 4];
    z[k] = op(keep, shfl_xor_any(send, 8));
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const T keep = b2 ? z[k + 2] : z[k], send = b2 ? z[k] : z[k + 2];
    w[k] = op(keep, shfl_xor_any(send, 4));
  }
  const T keep = b1 ? w[1] : w[0], send = b1 ? w[0] : w[1];
  const T u = op(keep, shfl_xor_any(send, 2));
  return op(u, shfl_xor_any(u, 1));
}
__device__ __forceinline__ int scatter16_element(int lane) {
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

// Epilogue of one 16-column group: v[i] is the fp32 result of packed row
// `row` (0..127 inside the tile) for token column c0 + i; `scale` is the
// weight row's scale, rs the per-column token scales (1 when the input is not
// normalised), pos the per-column cache positions (QKV).  Every variant
// computes all sixteen values first and stores with predicates, so the
// sixteen columns overlap instead of running one branch at a time.
template <int EPI, int WF>
__device__ __forceinline__ void epilogue_cols(const GemmArgs& a, int tile, int tt, int row, int c0, float* v,
                                              float scale, const float* rs, const int* pos,
                                              unsigned long long* wbest, float* sq_red, int warp_e, int lane,
                                              int layer = 0) {
  const int prow = tile * kTileN + row;  // packed row
  const bool row_ok = prow < a.n_rows;
  const int tok0 = tt * a.n_tok + c0;
  float x[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = v[i] * scale * rs[c0 + i];

  if constexpr (EPI == EPI_STORE) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = tok0 + i;
      if (row_ok && tok < a.m_tokens) a.out_f32[static_cast<size_t>(tok) * a.ld_out + prow] = x[i];
    }
  } else if constexpr (EPI == EPI_RESID) {
    float old[16];  // every load issued before the first store
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = tok0 + i;
      // (read at L2: in a multi-phase launch other SMs wrote these rows)
      old[i] = (row_ok && tok < a.m_tokens) ? __ldcg(a.out_f32 + static_cast<size_t>(tok) * a.ld_out + prow) : 0.0f;
    }
    float sq[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = tok0 + i;
      const bool ok = row_ok && tok < a.m_tokens;
      const float r = old[i] + x[i];  // residual GEMM inputs are not normalised: rs == 1
      sq[i] = ok ? r * r : 0.0f;
      if (ok) {
        const size_t o = static_cast<size_t>(tok) * a.ld_out + prow;
        a.out_f32[o] = r;
        const __half hi = __float2half_rn(r);
        a.x16_out[o] = hi;
        if (a.out_lo) a.x16_out[o + a.out_lo] = __float2half_rn(r - __half2float(hi));
        if (a.hidden_out) a.hidden_out[o + layer * a.hidden_layer_stride] = r;
      }
    }
    const float tot = warp_reduce_scatter16(sq, lane, [](float p, float q) { return p + q; });
    if ((lane & 1) == 0) sq_red[warp_e * 256 + c0 + scatter16_element(lane)] = tot;
  } else if constexpr (EPI == EPI_QKV) {
    const int hd = a.head_dim, half = hd >> 1;
    const int head = prow / hd, r = prow - head * hd;
    const int d = (r & 1) ? (r >> 1) + half : (r >> 1);
    const int fi = r >> 1;  // rotation frequency index
    const int group = a.n_q / a.n_kv;
    const bool rotate = head < a.n_q + a.n_kv;
    const bool is_q = head < a.n_q;
    float y[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 c = rotate ? a.rope[static_cast<size_t>(pos[c0 + i]) * half + fi] : make_float2(1.0f, 0.0f);
      const float xp = __shfl_xor_sync(0xFFFFFFFFu, x[i], 1);
      y[i] = (r & 1) ? (x[i] * c.x + xp * c.y) : (x[i] * c.x - xp * c.y);
    }
    // destination: q tile [B][n_kv][128][hd] (row j * group + hq) or block K / V [B][n_kv][32][hd]
    __nv_bfloat16* dst;
    int kvh, rstride, roff;
    if (is_q) {
      kvh = head / group;
      dst = a.q_tile;
      rstride = 128;
      roff = head - kvh * group;  // + j * group
    } else {
      kvh = rotate ? head - a.n_q : head - a.n_q - a.n_kv;
      dst = (rotate ? a.k_new : a.v_new) + layer * a.kv_layer_stride;
      rstride = 32;
      roff = 0;
    }
    const int jmul = is_q ? group : 1;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = tok0 + i;
      if (row_ok && tok < a.m_tokens) {
        const int b = tok / kRows, j = tok - b * kRows;
        const size_t o = ((static_cast<size_t>(b) * a.n_kv + kvh) * rstride + j * jmul + roff) * hd + d;
        const float val = rotate ? y[i] : x[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(val);
        dst[o] = hi;  // K / V: the cache format; q: the hi half of the attention's q tile
        if (is_q && a.out_lo) dst[o + a.out_lo] = __float2bfloat16_rn(val - __bfloat162float(hi));
      }
    }
  } else if constexpr (EPI == EPI_SILU) {
    // rows 2f / 2f+1 of the tile are gate / up of feature f: the pair of
    // lanes splits the sixteen columns (even lane 0..7, odd lane 8..15)
    const int feat = tile * 64 + (row >> 1);
    const bool odd = row & 1;
    float g[8], u[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float send = odd ? x[k] : x[k + 8];  // partner's half
      const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, 1);
      const float mine = odd ? x[k + 8] : x[k];
      g[k] = odd ? recv : mine;   // gate lives on the even lane
      u[k] = odd ? mine : recv;   // up on the odd lane
    }
    const int cbase = odd ? 8 : 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int tok = tok0 + cbase + k;
      const float sg = __fdividef(g[k], 1.0f + __expf(-g[k]));
      if (feat < a.ffn && tok < a.m_tokens) {
        const size_t o = static_cast<size_t>(tok) * a.ffn + feat;
        const float y = sg * u[k];
        const __half hi = __float2half_rn(y);
        a.act_out[o] = hi;
        if (a.out_lo) a.act_out[o + a.out_lo] = __float2half_rn(y - __half2float(hi));
      }
    }
  } else if constexpr (EPI == EPI_SAMPLE) {
    // tempered logits y = logit / T in log2 units; per column, the maximum
    // over the warp's 32 vocabulary rows and the sum of 2^(y - max), merged
    // pairwise (reduce-scatter); the caller folds the four warps
    const float c2 = a.inv_temp * kLog2e;
    unsigned long long e[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = tok0 + i;
      const bool ok = row_ok && tok < a.m_tokens;
      if (a.logits && ok) a.logits[static_cast<size_t>(tok) * a.n_rows + prow] = x[i];
      if (ok && prow == pos[c0 + i]) a.draft_logit[tok] = x[i];
      e[i] = ok ? ms_pack(x[i] * c2, 1.0f) : ms_pack(-INFINITY, 0.0f);
    }
    const unsigned long long tot = warp_reduce_scatter16(e, lane, [](unsigned long long p, unsigned long long q) {
      return ms_merge(p, q);
    });
    if ((lane & 1) == 0) wbest[warp_e * 16 + scatter16_element(lane)] = tot;
  } else if constexpr (EPI == EPI_ARGMAX) {
    unsigned long long key[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = tok0 + i;
      if (a.logits && row_ok && tok < a.m_tokens) a.logits[static_cast<size_t>(tok) * a.n_rows + prow] = x[i];
      key[i] = row_ok ? argmax_key(x[i], static_cast<uint32_t>(prow)) : 0ull;
    }
    const unsigned long long best =
        warp_reduce_scatter16(key, lane, [](unsigned long long p, unsigned long long q) { return p > q ? p : q; });
    if ((lane & 1) == 0) wbest[warp_e * 16 + scatter16_element(lane)] = best;
  }
}

template <int WF, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_act, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const bool act_lo = a.act_lo_rows > 0;
  const GemmSmem L = gemm_smem_layout(WF, a.n_tok, a.rd, a.da, a.db, a.cs, act_lo, a.r_alias != 0);
  const int RD = a.rd, DA = a.da, DB = a.db;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.ctrl_off);
  uint64_t* wfull = bars;                // weight tile landed
  uint64_t* wempty = wfull + kMaxRd;     // weight slot free again
  uint64_t* bfull = wempty + kMaxRd;     // activation tile landed
  uint64_t* bempty = bfull + kMaxDb;     // activation slot free again
  uint64_t* conv = bempty + kMaxDb;      // expanded tile ready (FP8 / NVFP4)
  uint64_t* cempty = conv + kMaxDa;      // expanded slot free again
  uint64_t* tfull = cempty + kMaxDa;     // [2] accumulator complete
  uint64_t* tempty = tfull + 2;          // [2] accumulator read out
  uint64_t* rfull = tempty + 2;          // peers' partials are in their R buffers
  uint64_t* rfree = rfull + 1;           // peers finished reading this CTA's R buffer
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(rfree + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_p + 1);
  // ARGMAX: per-warp column maxima of a 16-column group, two parities [2][4 warps][16]
  unsigned long long* wbest = reinterpret_cast<unsigned long long*>(smem + L.ctrl_off + kCtrlT);
  unsigned long long* best = reinterpret_cast<unsigned long long*>(smem + L.ctrl_off + kCtrlBest);
  float* sq_red = reinterpret_cast<float*>(smem + L.ctrl_off + kCtrlSq);
  float* rs = reinterpret_cast<float*>(smem + L.ctrl_off + kCtrlRs);
  int* pos_s = reinterpret_cast<int*>(smem + L.ctrl_off + kCtrlPos);
  float* R = reinterpret_cast<float*>(smem + L.r_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cs = a.cs;
  const int rank = cs > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int cluster = cs > 1 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int n_clusters = cs > 1 ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
  const int total = a.n_tiles * a.tok_tiles;
  // One item per CTA (the usual case for the FP8 / NVFP4 layer GEMMs): the
  // epilogue warps have nothing to do during the k loop, so warps 0-7 share
  // the weight expansion, and warps 0-3 also compute the per-token scales.
  const bool wide = WF != W_BF16 && total <= n_clusters;
  const bool has_item = cluster < total;
  const int conv_n = wide ? 256 : 128;
  // warps 0-3 join the epilogue when they have no expansion to run meanwhile
  const bool ep8 = WF == W_BF16 || wide;
  // With lo rows and n_tok <= 128, the hi and lo rows form one B operand of
  // 2 n_tok rows: one MMA per k step yields W x_hi in accumulator columns
  // [0, n_tok) and W x_lo in [n_tok, 2 n_tok), summed by the epilogue (MMA
  // instructions cost about the same for any N, so this halves them).  For
  // wider tiles the lo product is a second MMA into the same columns.  Two
  // accumulator buffers.
  const bool stacked = act_lo && 2 * a.n_tok <= 256;
  const int acc_w = stacked ? 2 * a.n_tok : a.n_tok;
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(2 * acc_w)) tmem_cols <<= 1;
  if (threadIdx.x == 0) trace_start(a.trace);

  if (threadIdx.x == 0) {
    for (int i = 0; i < RD; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], WF == W_BF16 ? 1 : conv_n);
    }
    for (int i = 0; i < DB; ++i) {
      mbar_init(&bfull[i], 1);
      mbar_init(&bempty[i], 1);
    }
    for (int i = 0; i < DA; ++i) {
      mbar_init(&conv[i], conv_n);
      mbar_init(&cempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], ep8 ? 256 : 128);
    }
    mbar_init(rfull, cs);
    mbar_init(rfree, cs);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_base_p, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (cs > 1) cluster_sync();  // every CTA of the cluster has its barriers initialised
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_p;
  pdl_launch_dependents();
  if (threadIdx.x == 0) trace_point(a.trace, 1);

  // per-token scale of the normalised input rows (and, for QKV, the cache
  // position of each token, whose RoPE row is pulled into L2 early); reads
  // what the previous kernels wrote, so only after the grid dependency wait
  auto token_scales = [&](int item, int t0, int nt) {
    const int tt = item % a.tok_tiles;
    for (int c = t0; c < a.n_tok; c += nt) {
      float r = 1.0f;
      const int tok = tt * a.n_tok + c;
      if (a.ssq_in && tok < a.m_tokens) {
        float ss = 0.0f;
#pragma unroll 8
        for (int k = 0; k < a.n_ssq; ++k) ss += a.ssq_in[static_cast<size_t>(k) * a.ssq_ld + tok];
        r = 1.0f / sqrtf(ss * a.inv_hidden + a.eps);
      }
      rs[c] = r;
      if constexpr (EPI == EPI_QKV) {
        int p = 0;
        if (tok < a.m_tokens) {
          p = a.ctx_len[tok / kRows] + tok % kRows;
          const char* row_p = reinterpret_cast<const char*>(a.rope + static_cast<size_t>(p) * (a.head_dim >> 1));
          for (int off = 0; off < (a.head_dim >> 1) * 8; off += 128) prefetch_l2(row_p + off);
        }
        pos_s[c] = p;
      }
      if constexpr (EPI == EPI_SAMPLE) {  // the column's draft token (-1: the bonus row, padding)
        const int j = tok % kRows;
        pos_s[c] = (tok < a.m_tokens && j < kBlock) ? a.drafts[(tok / kRows) * kBlock + j] : -1;
      }
    }
  };
  // weight expansion of the CTA's k tiles: NT = 256 chunk slots, by 256
  // threads (wide mode) or by 128 threads taking slots t and t + 128 (one
  // instantiation keeps the kernel's code small); in the wide mode warps 0-3
  // compute the token scales once the first expanded tiles are ready, and
  // publish them on named barrier 3
  auto expand_all = [&](auto nt_const, int t) {
    constexpr int NT = decltype(nt_const)::value;
    bool scales_done = !(wide && has_item && warp < 4);
    ItemIter it(&a, cluster, n_clusters, total, rank);
    int r = 0, c = 0;           // weight and expansion slots of tile i
    uint32_t rp = 0, cp = 0;    // their phase parities
    for (int i = 0; !it.done(); it.next(), ++i) {
      if (!scales_done && i == DA) {
        pdl_wait();
        token_scales(cluster, t, 128);
        named_bar_arrive(3, 256);
        scales_done = true;
      }
      if (!mbar_wait(&wfull[r], rp, abort_flag, a.status)) break;
      if (i >= DA && !mbar_wait(&cempty[c], cp ^ 1u, abort_flag, a.status)) break;
      if (t == 0 && i == 0) trace_point(a.trace, 3);
      expand_weights<WF, NT>(smem + L.a_off + c * 16384, smem + L.w_off + r * L.w_bytes, t);
      if (!wide)  // 128 threads: each also takes the chunks of thread t + 128
        expand_weights<WF, NT>(smem + L.a_off + c * 16384, smem + L.w_off + r * L.w_bytes, t + 128);
      fence_proxy_async();
      mbar_arrive(&conv[c]);
      mbar_arrive(&wempty[r]);
      if (++r == RD) {
        r = 0;
        rp ^= 1u;
      }
      if (++c == DA) {
        c = 0;
        cp ^= 1u;
      }
    }
    if (!scales_done) {
      pdl_wait();
      token_scales(cluster, t, 128);
      named_bar_arrive(3, 256);
    }
  };

  if (warp == 8) {
    // ---------------------------------------------------------- TMA producer (weights + activations)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      auto issue_w = [&](int r, const ItemIter& it) {
        uint8_t* dst = smem + L.w_off + r * L.w_bytes;
        mbar_expect_tx(&wfull[r], L.w_bytes);
        // every format is pre-packed in tiles (16-bit ones already in the MMA's swizzled layout)
        const uint8_t* src = a.w_tiles + (static_cast<size_t>(it.tile()) * a.k_tiles + it.kt) * L.w_bytes;
        bulk_load(dst, src, L.w_bytes, &wfull[r], pol_w);
      };
      auto issue_b = [&](int b, const ItemIter& it) {
        uint8_t* dst = smem + L.b_off + b * L.b_bytes;
        mbar_expect_tx(&bfull[b], L.b_bytes);
        // one box of n_tok rows (the host encodes the map with that box height); lo rows follow the hi tile
        const int r0 = it.tok_tile() * a.n_tok;
        tma_load_2d_hint(dst, &tm_act, &bfull[b], it.kt * kTileK, r0, pol_a);
        if (act_lo) tma_load_2d_hint(dst + a.n_tok * 128, &tm_act, &bfull[b], it.kt * kTileK, a.act_lo_rows + r0, pol_a);
      };
      // weights do not depend on the previous kernel: fill the weight ring before the grid dependency wait
      ItemIter itw(&a, cluster, n_clusters, total, rank), itb(&a, cluster, n_clusters, total, rank);
      // (wi, bi: tiles issued; ws, bs: next slot; wp, bp: parity of the release
      // of that slot's previous tile)
      int wi = 0, bi = 0, bs = 0;
      uint32_t wp = 0, bp = 0;
      for (; wi < RD && !itw.done(); ++wi, itw.next()) issue_w(wi, itw);
      int ws = wi == RD ? 0 : wi;
      pdl_wait();
      trace_point(a.trace, 2);
      // then serve both rings as their slots free up, never blocking on one while the other could proceed
      long long t_last = cycles();
      bool ok = true;
      while (!itw.done() || !itb.done()) {
        bool progress = false;
        if (!itb.done() && (bi < DB || mbar_test_wait(&bempty[bs], bp))) {
          issue_b(bs, itb);
          ++bi;
          if (++bs == DB) {  // slot 0 again: wait for the previous round's release
            bs = 0;
            bp = bi == DB ? 0u : bp ^ 1u;
          }
          itb.next();
          progress = true;
        }
        if (!itw.done() && (wi < RD || mbar_test_wait(&wempty[ws], wp))) {
          issue_w(ws, itw);
          ++wi;
          if (++ws == RD) {
            ws = 0;
            wp ^= 1u;
          }
          itw.next();
          progress = true;
        }
        if (progress) {
          t_last = cycles();
          continue;
        }
        // nothing to issue: poll again (a 64 ns back-off here measured
        // slower, as did one in the epilogue's wait for the accumulator)
        if (*abort_flag || cycles() - t_last > kWaitLimitCycles) {
          if (!*abort_flag) atomicOr(a.status, VSD_DEV_TIMEOUT);
          *abort_flag = 1;
          ok = false;
          break;
        }
      }
      if (!ok) {
        // drain: let the copies already in flight land before the CTA exits
        volatile int never = 0;
        for (int i = max(0, wi - RD); i < wi; ++i) mbar_wait(&wfull[i % RD], (i / RD) & 1, &never, nullptr);
        for (int i = max(0, bi - DB); i < bi; ++i) mbar_wait(&bfull[i % DB], (i / DB) & 1, &never, nullptr);
      }
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, acc_w, false, false, false);
      ItemIter it(&a, cluster, n_clusters, total, rank);
      // 16-bit weights are MMA-ready on arrival; FP8 / NVFP4 after expansion.
      // Ring slots and phases advance by counting (no division per k tile);
      // descriptors are the slot's base descriptor plus the address offset
      // (bits 0-13 hold address / 16).
      const int NA = WF == W_BF16 ? RD : DA;
      uint64_t* afull = WF == W_BF16 ? wfull : conv;
      uint64_t* aempty = WF == W_BF16 ? wempty : cempty;
      const uint64_t a_desc0 = sw128_desc(smem_u32(smem + (WF == W_BF16 ? L.w_off : L.a_off)), 16, 1024);
      const uint64_t b_desc0 = sw128_desc(smem_u32(smem + L.b_off), 16, 1024);
      const uint32_t b_step = L.b_bytes >> 4, lo_step = static_cast<uint32_t>(a.n_tok) * 8u;
      int s = 0, b = 0, acc = 0;
      uint32_t sp = 0, bp = 0;
      bool ok = true, first_tile = true;
      while (ok && !it.done()) {
        const int ab = acc & 1;
        if (acc >= 2 && !mbar_wait(&tempty[ab], ((acc >> 1) - 1) & 1, abort_flag, a.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(ab * acc_w);
        uint32_t accum = 0;
        bool last = false;
        do {
          if (!mbar_wait(&afull[s], sp, abort_flag, a.status) || !mbar_wait(&bfull[b], bp, abort_flag, a.status)) {
            ok = false;
            break;
          }
          if (first_tile) {
            trace_point(a.trace, 4);
            first_tile = false;
          }
          tc_fence_after();
          const uint64_t ad = a_desc0 + static_cast<uint64_t>(s) * 1024u;
          const uint64_t bd = b_desc0 + static_cast<uint64_t>(b) * b_step;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // stacked: B = hi rows then lo rows, one operand of acc_w rows
            umma_f16(d, ad + 2 * kk, bd + 2 * kk, idesc, accum | kk);
            if (act_lo && !stacked) umma_f16(d, ad + 2 * kk, bd + lo_step + 2 * kk, idesc, 1u);
          }
          accum = 1;
          umma_commit(&aempty[s]);
          umma_commit(&bempty[b]);
          last = it.last_k();
          it.next();
          if (++s == NA) {
            s = 0;
            sp ^= 1u;
          }
          if (++b == DB) {
            b = 0;
            bp ^= 1u;
          }
        } while (!last);
        if (!ok) break;
        umma_commit(&tfull[ab]);
        if (acc == 0) trace_point(a.trace, 5);
        ++acc;
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    // Warps 4-7 always; warps 0-3 too once they are free (16-bit weights: no
    // expansion; wide mode: expansion finished with the k loop).  Each set of
    // four warps covers the 128 TMEM lanes, and the two sets take alternate
    // 16-column groups, so two warps per scheduler hide each other's latency.
    const int half = warp < 4 ? 1 : 0;
    if constexpr (WF != W_BF16) {
      if (wide || half)  // one instantiation: 256 threads, or 128 threads taking two chunk sets each
        expand_all(std::integral_constant<int, 256>{}, static_cast<int>(threadIdx.x));
    }
    if (!half || ep8) {
      const int we = warp & 3;  // TMEM lane quarter
      const int row = we * 32 + lane;
      const int et = threadIdx.x & 127;     // thread of this set
      const int et2 = half * 128 + et;      // thread of the epilogue
      const int n_sets = ep8 ? 2 : 1;
      const int ep_n = 128 * n_sets;        // epilogue threads
      const int groups = a.n_tok / 16;
      const bool alive = rank * a.kps < a.k_tiles;
      // ARGMAX: running best key per token column of this CTA, flushed once at the end
      const bool keep_best = a.tok_tiles * a.n_tok <= kBestCap;
      if constexpr (EPI == EPI_ARGMAX)
        for (int c = et2; c < kBestCap; c += ep_n) best[c] = 0ull;
      // weight row scales are constant: the first item's is read before the grid dependency wait
      auto row_scale_of = [&](int item) -> float {
        if constexpr (WF == W_BF16) {
          return 1.0f;
        } else {
          const int prow = (item / a.tok_tiles) * kTileN + row;
          return prow < a.n_rows ? a.row_scale[prow] : 0.0f;
        }
      };
      float scale_next = (alive && cluster < total) ? row_scale_of(cluster) : 0.0f;
      pdl_wait();  // the token scales and positions read what the previous kernels wrote
      named_bar_sync(1, ep_n);
      int acc = 0;
      for (int item = cluster; alive && item < total; item += n_clusters, ++acc) {
        const int ab = acc & 1;
        const int tile = item / a.tok_tiles, tt = item % a.tok_tiles;
        const float scale = scale_next;
        if (item + n_clusters < total) scale_next = row_scale_of(item + n_clusters);
        // per-token scales: computed here while the MMAs run, or (wide mode)
        // by warps 0-3 during the expansion, published on barrier 3
        if (wide) {
          if (!half) named_bar_sync(3, 256);
        } else {
          token_scales(item, et2, ep_n);
        }
        named_bar_sync(1, ep_n);
        if (et2 == 0 && acc == 0) trace_point(a.trace, 8);
        if (cs > 1 && acc > 0 && !mbar_wait_cluster(rfree, (acc - 1) & 1, abort_flag, a.status)) break;
        if (!mbar_wait(&tfull[ab], (acc >> 1) & 1, abort_flag, a.status)) break;
        if (et2 == 0 && acc == 0) trace_point(a.trace, 6);
        if constexpr (EPI == EPI_RESID) {
          // the residual rows this thread updates: into L1 now, read after the reduction
          const int prow = tile * kTileN + row;
          if (prow < a.n_rows)
            for (int g = rank + cs * half; g < groups; g += cs * n_sets)
              for (int i = 0; i < 16; ++i) {
                const int tok = tt * a.n_tok + g * 16 + i;
                if (tok < a.m_tokens) prefetch_l1(a.out_f32 + static_cast<size_t>(tok) * a.ld_out + prow);
              }
        }
        tc_fence_after();
        const uint32_t taddr =
            tmem_base + (static_cast<uint32_t>(we * 32) << 16) + static_cast<uint32_t>(ab * acc_w);
        // 16 columns of the result: the hi product plus, if present, the lo product
        auto load_cols = [&](int c0, float* v) {
          tmem_ld16(taddr + c0, v);
          if (stacked) {
            float w[16];
            tmem_ld16(taddr + a.n_tok + c0, w);
            tmem_ld_wait();
  #pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += w[i];
          } else {
            tmem_ld_wait();
          }
        };
        float v[16];
        if (cs > 1) {
          // partial sums of this CTA's k range -> R (column-major), then tell every CTA of the cluster
          for (int c0 = half * 16; c0 < a.n_tok; c0 += 16 * n_sets) {
            load_cols(c0, v);
  #pragma unroll
            for (int i = 0; i < 16; ++i) R[(c0 + i) * L.r_ld + row] = v[i];
          }
          tc_fence_before();
          mbar_arrive(&tempty[ab]);
          named_bar_sync(1, ep_n);
          if (et2 < cs) {  // one thread per peer: the cluster-scope fence and remote arrive cost ~0.2-0.7 us each
            fence_acq_rel_cluster();
            mbar_arrive_remote(mapa_shared(smem_u32(rfull), et2));
          }
          if (!mbar_wait_cluster(rfull, acc & 1, abort_flag, a.status)) break;
          if (et2 == 0 && acc == 0) trace_point(a.trace, 7);
        }
        // column groups of this set: every n_sets-th of this CTA's (all groups
        // when cs == 1, every cs-th for a split-K rank)
        int gi = 0;
        for (int g = rank + cs * half; g < groups; g += cs * n_sets, ++gi) {
          const int c0 = g * 16;
          if (cs == 1) {
            load_cols(c0, v);
          } else {
            const uint32_t local = smem_u32(R + c0 * L.r_ld + row);
  #pragma unroll 1
            for (int h4 = 0; h4 < 16; h4 += 4) {  // 4 columns at a time, every peer's loads in flight
              float x[8][4];
  #pragma unroll
              for (int p = 0; p < 8; ++p)
                if (p < cs) {
                  const uint32_t ra = mapa_shared(local, p) + h4 * L.r_ld * 4;
  #pragma unroll
                  for (int i = 0; i < 4; ++i) x[p][i] = ld_dsmem_f32(ra + i * L.r_ld * 4);
                }
  #pragma unroll
              for (int i = 0; i < 4; ++i) v[h4 + i] = 0.0f;
  #pragma unroll
              for (int p = 0; p < 8; ++p)  // fixed order: deterministic sum
                if (p < cs) {
  #pragma unroll
                  for (int i = 0; i < 4; ++i) v[h4 + i] += x[p][i];
                }
            }
          }
          if (et2 == 0 && acc == 0 && g == rank) trace_point(a.trace, 12);
          // ARGMAX: per-warp maxima, [set][parity][4 warps][16]
          unsigned long long* wb = wbest + half * 128 + (gi & 1) * 64;
          epilogue_cols<EPI, WF>(a, tile, tt, row, c0, v, scale, rs, pos_s, wb, sq_red, we, lane);
          if (et2 == 0 && acc == 0 && g == rank) trace_point(a.trace, 14);
          if constexpr (EPI == EPI_ARGMAX) {
            named_bar_sync(4 + half, 128);  // this set's four warps only
            if (et < 16) {  // fold the four warps' maxima of column c0 + et (the other parity is written next)
              unsigned long long k = wb[et];
  #pragma unroll
              for (int w = 1; w < 4; ++w) k = wb[w * 16 + et] > k ? wb[w * 16 + et] : k;
              const int col = tt * a.n_tok + c0 + et;
              if (keep_best) {
                if (k > best[col]) best[col] = k;
              } else if (col < a.m_tokens && k) {
                atomicMax(a.keys + col, k);
              }
            }
            if (et2 == 0 && acc == 0 && g == rank) trace_point(a.trace, 15);
          }
          if constexpr (EPI == EPI_SAMPLE) {
            named_bar_sync(4 + half, 128);  // this set's four warps only
            if (et < 16) {  // the tile's (max, sum) for column c0 + et, warps in fixed order (deterministic)
              const unsigned long long r = ms_merge(ms_merge(ms_merge(wb[et], wb[16 + et]), wb[32 + et]), wb[48 + et]);
              const int col = tt * a.n_tok + c0 + et;
              if (col < a.m_tokens) {
                a.tile_max[static_cast<size_t>(col) * a.n_tiles + tile] = ms_max(r);
                a.tile_sum[static_cast<size_t>(col) * a.n_tiles + tile] = ms_sum(r);
              }
            }
          }
        }
        if (cs == 1) {
          tc_fence_before();
          mbar_arrive(&tempty[ab]);
        }
        named_bar_sync(1, ep_n);
        if (et2 == 0 && acc == 0) trace_point(a.trace, 9);
        if (cs > 1 && et2 < cs) {
          fence_acq_rel_cluster();
          mbar_arrive_remote(mapa_shared(smem_u32(rfree), et2));
        }
        if constexpr (EPI == EPI_RESID) {
          for (int c = et2; c < a.n_tok; c += ep_n) {
            const int tok = tt * a.n_tok + c;
            if ((c / 16) % cs == rank && tok < a.m_tokens)
              a.ssq_out[static_cast<size_t>(tile) * a.ssq_ld + tok] =
                  sq_red[c] + sq_red[256 + c] + sq_red[512 + c] + sq_red[768 + c];
          }
        }
        named_bar_sync(1, ep_n);
        if (et2 == 0 && acc == 0) trace_point(a.trace, 10);
      }
      // the peers read this CTA's R buffer until they arrive on rfree: wait for
      // that before the CTA may exit (its shared memory must stay valid)
      if (cs > 1 && acc > 0) mbar_wait_cluster(rfree, (acc - 1) & 1, abort_flag, a.status);
      if constexpr (EPI == EPI_ARGMAX) {
        if (keep_best)
          for (int c = et2; c < a.tok_tiles * a.n_tok; c += ep_n)
            if (c < a.m_tokens && best[c]) atomicMax(a.keys + c, best[c]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_end(a.trace, 11);
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace vsd
