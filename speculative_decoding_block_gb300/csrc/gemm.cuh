// gemm.cuh -- weight-streaming GEMM for the verify rows on tcgen05 / TMEM.
//
// Computes, for one weight matrix W [N, K] in BF16, FP8 E4M3 (per-row fp32
// scale) or NVFP4 (E2M1 values, E4M3 scale per 16 k, fp32 tensor scale),
//     Y[t, n] = sum_k X[t, k] * W[n, k]
// over the M = 17 * batch token rows X (f16, row-major [M, K]).
//
// Swap-AB: the weight tile is the 128-row A operand and the tokens are the
// MMA's N dimension, so one CTA covers 128 output features x n_tok tokens.
// Weight tiles arrive by TMA (BF16: tiled tensor copy with the 128-byte
// swizzle, converted to f16 in place; FP8 / NVFP4: one 1-D bulk copy of a
// pre-packed tile, expanded exactly to f16 -- E4M3 and E2M1 x E4M3 values are
// all exact f16 numbers).  Activation tiles arrive by TMA with the same
// swizzle.  The fp32 accumulator sits in TMEM (double-buffered so the
// epilogue of one tile overlaps the MMAs of the next).  Per-row and
// per-tensor scales are applied in the epilogue.
//
// Warp roles (320 threads): warps 0-3 expand weights into the f16 A tile,
// warps 4-7 run the epilogue (warp w reads TMEM lanes 32*(w%4)..), warp 8
// issues TMA, warp 9 allocates TMEM and issues the MMAs.  CTAs are
// persistent over work items (tile, token tile, k split); split-K partial
// sums go to a workspace and the last CTA of a tile adds them in split order
// (deterministic) before running the epilogue.
//
// Epilogues fuse the neighbouring element-wise steps of the decoder layer
// ("The Inference Stack Behind OCRia", section "Avoiding unnecessary memory
// transfers": intermediates stay on chip):
//   STORE  : y = acc * scale                       (component entry point)
//   RESID  : x_resid += acc * scale                (O and down projections)
//   QKV    : RoPE on q and k, q -> attention tile layout, k / v -> block scratch
//   SILU   : silu(gate) * up -> f16 MLP activation (gate/up rows interleaved)
//   ARGMAX : per token, max over vocab rows -> 64-bit argmax key (atomicMax)
#pragma once

#include "vsd_common.cuh"

namespace vsd {

enum WFmt { W_BF16 = 0, W_FP8 = 1, W_NVFP4 = 2 };
enum Epi { EPI_STORE = 0, EPI_RESID = 1, EPI_QKV = 2, EPI_SILU = 3, EPI_ARGMAX = 4 };

constexpr int kGemmThreads = 320;
constexpr int kTileN = 128;   // weight rows per tile (MMA M)
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
  int splits, kt_per_split;
  int m_tokens;            // valid token rows
  int stages;
  // STORE / RESID
  float* out_f32;
  int ld_out;
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
  float* logits;             // optional [M][vocab]
  // split-K
  float* partials;
  int* counters;
  int* status;
};

struct GemmSmem {
  // offsets inside the dynamic shared memory (after 1024-byte alignment)
  uint32_t stage_bytes, b_off, ctrl_off;
};

__host__ __device__ inline GemmSmem gemm_smem_layout(int wf, int n_tok, int stages) {
  GemmSmem s;
  s.b_off = 16384u + raw_region_bytes(wf);
  s.stage_bytes = s.b_off + static_cast<uint32_t>(n_tok) * 128u;
  s.ctrl_off = s.stage_bytes * static_cast<uint32_t>(stages);
  return s;
}
// control block: 4*stages+4 barriers, tmem base, abort flag, last flag, argmax reduction
__host__ __device__ inline uint32_t gemm_ctrl_bytes() { return 1024u + 8192u; }
__host__ __device__ inline uint32_t gemm_smem_bytes(int wf, int n_tok, int stages) {
  return 1024u + gemm_smem_layout(wf, n_tok, stages).ctrl_off + gemm_ctrl_bytes();
}

// Iterates over the (item, k-tile) sequence of one CTA.
struct ItemIter {
  int item, total, stride, kt, kt_end;
  const GemmArgs* a;
  __device__ void set_item() {
    const int split = item % a->splits;
    kt = split * a->kt_per_split;
    kt_end = min(a->k_tiles, kt + a->kt_per_split);
  }
  __device__ ItemIter(const GemmArgs* args, int first, int stride_, int total_)
      : item(first), total(total_), stride(stride_), kt(0), kt_end(0), a(args) {
    if (item < total) set_item();
  }
  __device__ bool done() const { return item >= total; }
  __device__ bool first_k() const { return kt == (item % a->splits) * a->kt_per_split; }
  __device__ bool last_k() const { return kt + 1 == kt_end; }
  __device__ int tile() const { return item / (a->splits * a->tok_tiles); }
  __device__ int tok_tile() const { return (item / a->splits) % a->tok_tiles; }
  __device__ void next() {
    if (++kt >= kt_end) {
      item += stride;
      if (item < total) set_item();
    }
  }
};

template <int WF>
__device__ __forceinline__ void expand_weights(uint8_t* a_tile, const uint8_t* raw, int t) {
  // 1024 chunks of 8 f16 (16 bytes); thread t handles chunks t + 128 i.
#pragma unroll 4
  for (int i = 0; i < 8; ++i) {
    const int q = t + 128 * i;
    const int r = q >> 3, c = q & 7;
    uint4 o;
    if constexpr (WF == W_BF16) {
      uint4* p = reinterpret_cast<uint4*>(a_tile + q * 16);  // in place, position unchanged
      const uint4 v = *p;
      o.x = bf16x2_to_f16x2(v.x);
      o.y = bf16x2_to_f16x2(v.y);
      o.z = bf16x2_to_f16x2(v.z);
      o.w = bf16x2_to_f16x2(v.w);
      *p = o;
    } else if constexpr (WF == W_FP8) {
      const uint2 v = *reinterpret_cast<const uint2*>(raw + r * 64 + c * 8);
      o.x = e4m3x2_to_f16x2(static_cast<uint16_t>(v.x & 0xFFFF));
      o.y = e4m3x2_to_f16x2(static_cast<uint16_t>(v.x >> 16));
      o.z = e4m3x2_to_f16x2(static_cast<uint16_t>(v.y & 0xFFFF));
      o.w = e4m3x2_to_f16x2(static_cast<uint16_t>(v.y >> 16));
      *reinterpret_cast<uint4*>(a_tile + sw128_off(r, c)) = o;
    } else {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(raw + r * 32 + c * 4);
      const uint32_t sb = raw[kFp4ValBytes + r * 4 + (c >> 1)];
      const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint16_t>(sb | (sb << 8)));
      uint32_t h[4];
      e2m1x8_to_f16x8(v, h);
      const __half2 sc = *reinterpret_cast<const __half2*>(&s2);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        __half2 x = *reinterpret_cast<__half2*>(&h[j]);
        x = __hmul2(x, sc);  // exact: both factors have <= 4 significant bits
        h[j] = *reinterpret_cast<uint32_t*>(&x);
      }
      o = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(a_tile + sw128_off(r, c)) = o;
    }
  }
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

// Epilogue of one 16-column group: v[i] is the fp32 result of packed row
// `row` (0..127 inside the tile) for token column c0 + i.
template <int EPI, int WF>
__device__ __forceinline__ void epilogue_cols(const GemmArgs& a, int tile, int tt, int row, int c0,
                                              float* v, unsigned long long* red, int warp_e, int lane) {
  const int prow = tile * kTileN + row;  // packed row
  const bool row_ok = prow < a.n_rows;
  float scale = 1.0f;
  if constexpr (WF != W_BF16) scale = row_ok ? a.row_scale[prow] : 0.0f;
  const int tok0 = tt * a.n_tok + c0;

  if constexpr (EPI == EPI_STORE || EPI == EPI_RESID) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = tok0 + i;
      if (row_ok && tok < a.m_tokens) {
        float* p = a.out_f32 + static_cast<size_t>(tok) * a.ld_out + prow;
        if constexpr (EPI == EPI_RESID) *p += v[i] * scale;
        else *p = v[i] * scale;
      }
    }
  } else if constexpr (EPI == EPI_QKV) {
    const int hd = a.head_dim, half = hd >> 1;
    const int head = prow / hd, r = prow % hd;
    const int d = (r & 1) ? (r >> 1) + half : (r >> 1);
    const int fi = r >> 1;  // rotation frequency index
    const int group = a.n_q / a.n_kv;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float x = v[i] * scale;
      const float xp = __shfl_xor_sync(0xFFFFFFFFu, x, 1);
      const int tok = tok0 + i;
      if (!row_ok || tok >= a.m_tokens) continue;
      const int b = tok / kRows, j = tok % kRows;
      if (head < a.n_q + a.n_kv) {  // q or k: rotate
        const float2 cs = a.rope[static_cast<size_t>(a.ctx_len[b] + j) * half + fi];
        const float y = (r & 1) ? (x * cs.x + xp * cs.y) : (x * cs.x - xp * cs.y);
        if (head < a.n_q) {
          const int kvh = head / group, hq = head % group;
          a.q_tile[((static_cast<size_t>(b) * a.n_kv + kvh) * 128 + j * group + hq) * hd + d] =
              __float2bfloat16_rn(y);
        } else {
          const int kvh = head - a.n_q;
          a.k_new[((static_cast<size_t>(b) * a.n_kv + kvh) * 32 + j) * hd + d] = __float2bfloat16_rn(y);
        }
      } else {
        const int kvh = head - a.n_q - a.n_kv;
        a.v_new[((static_cast<size_t>(b) * a.n_kv + kvh) * 32 + j) * hd + d] = __float2bfloat16_rn(x);
      }
    }
  } else if constexpr (EPI == EPI_SILU) {
    const int feat = tile * 64 + (row >> 1);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float x = v[i] * scale;
      const float up = __shfl_xor_sync(0xFFFFFFFFu, x, 1);
      const int tok = tok0 + i;
      if ((row & 1) == 0 && feat < a.ffn && tok < a.m_tokens) {
        const float g = x / (1.0f + expf(-x));
        a.act_out[static_cast<size_t>(tok) * a.ffn + feat] = __float2half_rn(g * up);
      }
    }
  } else if constexpr (EPI == EPI_ARGMAX) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int tok = tok0 + i;
      const float x = v[i] * scale;
      if (a.logits && row_ok && tok < a.m_tokens) a.logits[static_cast<size_t>(tok) * a.n_rows + prow] = x;
      unsigned long long key = row_ok ? argmax_key(x, static_cast<uint32_t>(prow)) : 0ull;
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        const unsigned long long o = shfl_xor_u64(key, m);
        key = o > key ? o : key;
      }
      if (lane == 0) red[warp_e * 256 + c0 + i] = key;
    }
  }
}

template <int WF, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_w,
                const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const GemmSmem L = gemm_smem_layout(WF, a.n_tok, a.stages);
  const int S = a.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.ctrl_off);
  uint64_t* wfull = bars;
  uint64_t* afull = bars + S;
  uint64_t* conv = bars + 2 * S;
  uint64_t* empty = bars + 3 * S;
  uint64_t* tfull = bars + 4 * S;
  uint64_t* tempty = bars + 4 * S + 2;
  uint32_t* tmem_base_p = reinterpret_cast<uint32_t*>(bars + 4 * S + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_p + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_base_p + 2);
  unsigned long long* red = reinterpret_cast<unsigned long long*>(smem + L.ctrl_off + 1024);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = a.n_tiles * a.tok_tiles * a.splits;
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(2 * a.n_tok)) tmem_cols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&afull[s], 1);
      mbar_init(&conv[s], 128);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_base_p, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_p;
  pdl_launch_dependents();

  if (warp == 8) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      const uint32_t wbytes = WF == W_BF16 ? 16384u : (WF == W_FP8 ? kFp8TileBytes : kFp4TileBytes);
      auto issue_w = [&](int cnt, const ItemIter& it) {
        const int s = cnt % S;
        uint8_t* st = smem + s * L.stage_bytes;
        mbar_expect_tx(&wfull[s], wbytes);
        if constexpr (WF == W_BF16) {
          tma_load_2d_hint(st, &tm_w, &wfull[s], it.kt * kTileK, it.tile() * kTileN, pol_w);
        } else {
          const uint8_t* src = a.w_tiles + (static_cast<size_t>(it.tile()) * a.k_tiles + it.kt) * wbytes;
          bulk_load(st + 16384, src, wbytes, &wfull[s], pol_w);
        }
      };
      // weights do not depend on the previous kernel: start them before the grid dependency wait
      int pre = 0;
      {
        ItemIter it(&a, blockIdx.x, gridDim.x, total);
        for (; pre < S && !it.done(); ++pre, it.next()) issue_w(pre, it);
      }
      pdl_wait();
      ItemIter it(&a, blockIdx.x, gridDim.x, total);
      int cnt = 0;
      bool ok = true;
      for (; !it.done(); it.next(), ++cnt) {
        const int s = cnt % S;
        if (cnt >= S && !mbar_wait(&empty[s], ((cnt / S) - 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        if (cnt >= pre) issue_w(cnt, it);
        uint8_t* bt = smem + s * L.stage_bytes + L.b_off;
        mbar_expect_tx(&afull[s], static_cast<uint32_t>(a.n_tok) * 128u);
        const int r0 = it.tok_tile() * a.n_tok;
        for (int i = 0; i < a.n_tok / 16; ++i)
          tma_load_2d_hint(bt + i * 2048, &tm_act, &afull[s], it.kt * kTileK, r0 + 16 * i, pol_a);
      }
      if (!ok) {
        // drain: let the copies already in flight land before the CTA exits
        const int issued = max(cnt, pre);
        for (int c = max(0, issued - S); c < issued; ++c) {
          volatile int never = 0;
          mbar_wait(&wfull[c % S], (c / S) & 1, &never, nullptr);
          if (c < cnt) mbar_wait(&afull[c % S], (c / S) & 1, &never, nullptr);
        }
      }
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------- weight expansion
    const int t = threadIdx.x;
    ItemIter it(&a, blockIdx.x, gridDim.x, total);
    for (int cnt = 0; !it.done(); it.next(), ++cnt) {
      const int s = cnt % S;
      if (!mbar_wait(&wfull[s], (cnt / S) & 1, abort_flag, a.status)) break;
      uint8_t* st = smem + s * L.stage_bytes;
      expand_weights<WF>(st, st + 16384, t);
      fence_proxy_async();
      mbar_arrive(&conv[s]);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, a.n_tok, false, false, false);
      ItemIter it(&a, blockIdx.x, gridDim.x, total);
      int cnt = 0, acc = 0;
      bool ok = true;
      while (ok && !it.done()) {
        const int ab = acc & 1;
        if (acc >= 2 && !mbar_wait(&tempty[ab], ((acc >> 1) - 1) & 1, abort_flag, a.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(ab * a.n_tok);
        bool last = false;
        do {
          const int s = cnt % S;
          const uint32_t par = (cnt / S) & 1;
          if (!mbar_wait(&conv[s], par, abort_flag, a.status) ||
              !mbar_wait(&afull[s], par, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * L.stage_bytes);
          const uint32_t sb = smem_u32(smem + s * L.stage_bytes + L.b_off);
          const bool first = it.first_k();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            umma_f16(d, sw128_desc(sa + kk * 32, 16, 1024), sw128_desc(sb + kk * 32, 16, 1024), idesc,
                     (first && kk == 0) ? 0u : 1u);
          }
          umma_commit(&empty[s]);
          last = it.last_k();
          it.next();
          ++cnt;
        } while (!last);
        if (!ok) break;
        umma_commit(&tfull[ab]);
        ++acc;
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue (warps 4..7)
    const int we = warp - 4;  // == warp % 4: TMEM lane quarter
    const int row = we * 32 + lane;
    const int et = threadIdx.x - 128;
    int acc = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++acc) {
      const int ab = acc & 1;
      if (!mbar_wait(&tfull[ab], (acc >> 1) & 1, abort_flag, a.status)) break;
      tc_fence_after();
      const int tile = item / (a.splits * a.tok_tiles);
      const int tt = (item / a.splits) % a.tok_tiles;
      const int split = item % a.splits;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(we * 32) << 16) + static_cast<uint32_t>(ab * a.n_tok);
      float v[16];
      if (a.splits == 1) {
        for (int c0 = 0; c0 < a.n_tok; c0 += 16) {
          tmem_ld16(taddr + c0, v);
          tmem_ld_wait();
          epilogue_cols<EPI, WF>(a, tile, tt, row, c0, v, red, we, lane);
        }
        tc_fence_before();
        mbar_arrive(&tempty[ab]);
      } else {
        const int tid = tile * a.tok_tiles + tt;
        float* base = a.partials + static_cast<size_t>(tid) * a.splits * 128 * a.n_tok;
        float* mine = base + static_cast<size_t>(split) * 128 * a.n_tok;
        for (int c0 = 0; c0 < a.n_tok; c0 += 16) {
          tmem_ld16(taddr + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) __stcg(mine + (c0 + i) * 128 + row, v[i]);
        }
        tc_fence_before();
        mbar_arrive(&tempty[ab]);
        __threadfence();
        named_bar_sync(1, 128);
        if (et == 0) *last_flag = (atomicAdd(&a.counters[tid], 1) == a.splits - 1) ? 1 : 0;
        named_bar_sync(1, 128);
        if (*last_flag) {
          __threadfence();
          for (int c0 = 0; c0 < a.n_tok; c0 += 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.0f;
            for (int sp = 0; sp < a.splits; ++sp) {
              const float* p = base + static_cast<size_t>(sp) * 128 * a.n_tok + c0 * 128 + row;
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] += __ldcg(p + i * 128);
            }
            epilogue_cols<EPI, WF>(a, tile, tt, row, c0, v, red, we, lane);
          }
          if (et == 0) a.counters[tid] = 0;
        } else {
          continue;  // this CTA's split is done; the last CTA runs the epilogue
        }
      }
      if constexpr (EPI == EPI_ARGMAX) {
        named_bar_sync(1, 128);
        for (int c = et; c < a.n_tok; c += 128) {
          unsigned long long k = red[c];
          for (int w = 1; w < 4; ++w) k = red[w * 256 + c] > k ? red[w * 256 + c] : k;
          const int tok = tt * a.n_tok + c;
          if (tok < a.m_tokens) atomicMax(a.keys + tok, k);
        }
        named_bar_sync(1, 128);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

}  // namespace vsd
