// replay_ssm.cuh -- ReplaySSM-style verification and rollback of a recurrent
// (gated delta rule) layer under block speculative decoding.
//
// "The Inference Stack Behind OCRia", section "Make speculative verification
// cheaper": a GDN layer's fixed-size state is kept as a checkpoint plus a
// small buffer of recent tokens; outputs are computed from the checkpoint and
// the buffered tokens, the checkpoint is rewritten only at periodic flushes,
// and rejected drafts are rolled back by moving the buffer pointer.  The
// pages give no update rule; the gated delta rule of Gated DeltaNet is used:
//     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
//     o_t = S_t q_t,
// per request and head, S of d x d (d_k = d_v = d).
//
// Form used here.  With u_t = beta_t (v_t - alpha_t S_{t-1} k_t) (the
// token's corrected value) the update reads S_t = alpha_t S_{t-1} + u_t k_t^T,
// so with L_t = sum of log alpha over the tokens since the checkpoint S_0,
//     S_t = e^{L_t} S_0 + sum_{s<=t} e^{L_t - L_s} u_s k_s^T.
// Hence, for a new token t after the retained ones,
//     u_t = beta_t (v_t - e^{L_t} S_0 k_t - sum_{s<t} e^{L_t - L_s} (k_s.k_t) u_s),
//     o_t = e^{L_t} S_0 q_t + sum_{s<=t} e^{L_t - L_s} (k_s.q_t) u_s.
// The buffer keeps, per retained token, k_s, u_s and L_s (u_s depends only on
// the checkpoint and the tokens before s, so rejected rows never touch it).
// The checkpoint and the retained keys are stored as the tensor cores read
// them: f16 hi / lo images with a power-of-2 scale per row (about 22
// significant bits), so that the verify copies them into shared memory
// with bulk copies, the next item's while the current one computes.
// A verify block then costs two products with the checkpoint per block row
// (S_0 k_t, S_0 q_t) plus dot products with the buffered keys -- dense
// contractions, run on the tensor cores -- and a 17-step triangular solve
// per state row, instead of a replay of the whole buffer through the d x d
// state; a flush folds the buffer into the checkpoint with the closed form
// above.
#pragma once

#include "vsd_common.cuh"

namespace vsd {

constexpr int kSsmThreads = 256;
constexpr int kSsmMaxWindow = 128;         // d = 64; d = 128 allows up to 64 (shared memory)
constexpr int kSsmCoefLd = 20;             // 17 coefficients per key row, padded for float4 reads
constexpr float kSsmMinLogGate = -200.0f;  // log alpha floor: e^-200 underflows to 0 in every product
constexpr int kSsmN = 48;                  // MMA N: the block vectors, padded
constexpr int kSsmTmemCols = 128;          // P at columns 0-47, G at 64-111
constexpr uint32_t kSsmAtomA = 16384;      // one 64-wide K atom of a 128-row tile in shared memory
constexpr uint32_t kSsmAtomB = kSsmN * 128;

__host__ __device__ inline int ssm_max_window(int d) { return d == 128 ? 64 : kSsmMaxWindow; }
__host__ __device__ inline int ssm_exp_stride(int window) { return (window + 3) & ~3; }  // 16-byte rows

struct SsmArgs {
  int heads, d, window, batch;
  // a verify block [B][H][17][d] (q, k, v) and [B][H][17] (alpha, beta)
  const float *q, *k, *v, *alpha, *beta;
  float* out;             // [B][H][17][d]
  uint8_t* ckpt;          // [max_batch][H] checkpoint images, 4 d^2 bytes each
  int* ckpt_exp;          // [max_batch][H][d] their row exponents
  uint8_t* buf_k;         // [max_batch][H] retained-key images, 4 window d bytes each
  int* buf_kexp;          // [max_batch][H][exp_stride(window)] their row exponents
  float* buf_u;           // [max_batch][H][window][d] corrected values
  double* buf_L;          // [max_batch][H][window] log gate sums since the checkpoint (double: the
                          // coefficients use differences of nearby sums, which stay exact)
  int* ptr;               // [max_batch] retained buffered tokens
  const int* accepted;    // [B] commit: accepted drafts a (-1: rejected)
  const float* state_in;  // [H][d][d] a request's new state (set)
  float* state_out;       // [H][d][d] a request's effective state (get)
  int req;                // that request
  int* status;
};

// ---------------------------------------------------------------- images
// An image of R rows x d columns: the f16 hi values, then the f16 lo
// values, each as d / 64 atoms of R rows x 128 bytes with the 128-byte
// swizzle: element (r, k) in atom k / 64, row r, 16-byte chunk (k % 64) / 8
// (swizzled by r % 8), half-word k % 8.  Row r stands for x = (hi + lo) 2^-e_r.
struct SsmImage {
  uint32_t atom, lo;  // bytes per atom, offset of the lo half
};
__host__ __device__ inline SsmImage ssm_image(int rows, int d) {
  SsmImage g;
  g.atom = static_cast<uint32_t>(rows) * 128u;
  g.lo = static_cast<uint32_t>(d / 64) * g.atom;
  return g;
}
__device__ __forceinline__ uint32_t ssm_img_off(const SsmImage& g, int r, int k0) {
  return static_cast<uint32_t>(k0 >> 6) * g.atom + sw128_off(static_cast<uint32_t>(r), (k0 & 63) >> 3) +
         static_cast<uint32_t>((k0 >> 2) & 1) * 8u;
}
__device__ __forceinline__ float ssm_pow2(int e) { return __int_as_float((127 + e) << 23); }

// Values k0..k0+3 of row r (k0 % 4 == 0), times 2^-e.
__device__ __forceinline__ float4 ssm_img_get4(const uint8_t* img, const SsmImage& g, int r, int k0, int e) {
  const uint32_t off = ssm_img_off(g, r, k0);
  const uint2 h = *reinterpret_cast<const uint2*>(img + off);
  const uint2 l = *reinterpret_cast<const uint2*>(img + g.lo + off);
  const __half2 h01 = *reinterpret_cast<const __half2*>(&h.x), h23 = *reinterpret_cast<const __half2*>(&h.y);
  const __half2 l01 = *reinterpret_cast<const __half2*>(&l.x), l23 = *reinterpret_cast<const __half2*>(&l.y);
  const float s = ssm_pow2(-e);
  return make_float4((__low2float(h01) + __low2float(l01)) * s, (__high2float(h01) + __high2float(l01)) * s,
                     (__low2float(h23) + __low2float(l23)) * s, (__high2float(h23) + __high2float(l23)) * s);
}
// Stores y (already scaled by 2^e) at k0..k0+3 of row r as hi / lo.
__device__ __forceinline__ void ssm_img_put4(uint8_t* img, const SsmImage& g, int r, int k0, float4 y) {
  const uint32_t off = ssm_img_off(g, r, k0);
  const uint32_t h01 = f32x2_to_f16x2(y.x, y.y), h23 = f32x2_to_f16x2(y.z, y.w);
  const __half2 a01 = *reinterpret_cast<const __half2*>(&h01), a23 = *reinterpret_cast<const __half2*>(&h23);
  const uint32_t l01 = f32x2_to_f16x2(y.x - __low2float(a01), y.y - __high2float(a01));
  const uint32_t l23 = f32x2_to_f16x2(y.z - __low2float(a23), y.w - __high2float(a23));
  *reinterpret_cast<uint2*>(img + off) = make_uint2(h01, h23);
  *reinterpret_cast<uint2*>(img + g.lo + off) = make_uint2(l01, l23);
}

// Exponent e with max * 2^e in [2^14, 2^15) (127 for m = 0: no bound),
// clamped so that 2^e and 2^-e are normal floats.
__device__ __forceinline__ int ssm_scale_exp(float m) {
  if (!(m > 0.0f)) return 127;
  int ex;
  frexpf(m, &ex);  // m = f 2^ex, f in [0.5, 1)
  return max(-120, min(120, 15 - ex));
}

// Rows are converted a whole row per warp instruction (d = 128; two rows
// for d = 64), lane l holding the row's values 4l..4l+3, so that every
// global load is one contiguous run of whole lines.  Slot i of a thread is
// row r0 + (8 i + warp) RPI + lane / LPR.
template <int D>
struct SsmTile {
  static constexpr int LPR = D / 4;     // lanes per row
  static constexpr int RPI = 32 / LPR;  // rows per warp instruction
  static constexpr int RPP = 8 * RPI;   // rows per pass of the 8 warps
};
template <int D>
__device__ __forceinline__ int ssm_tile_row(int i) {
  return (8 * i + static_cast<int>(threadIdx.x >> 5)) * SsmTile<D>::RPI +
         static_cast<int>(threadIdx.x & 31) / SsmTile<D>::LPR;
}
// Loads slots 0..N-1 (row r from src(r); zero for r >= rows or a null src).
template <int D, int N, typename Src>
__device__ __forceinline__ void ssm_tile_load(float4* x, int r0, int rows, Src src) {
  const int l4 = static_cast<int>(threadIdx.x & 31) % SsmTile<D>::LPR;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const int r = r0 + ssm_tile_row<D>(i);
    const float* s = r < rows ? src(r) : nullptr;
    x[i] = s ? reinterpret_cast<const float4*>(s)[l4] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}
// Stores slots 0..N-1 with r < rows as row images (each row scaled by its
// own 2^e, a min-reduction over the row's lanes; e into expo[r]), into
// `img` and, when img2 is set, into img2 / expo2 too.
template <int D, int N>
__device__ __forceinline__ void ssm_tile_store(const float4* x, int r0, int rows, uint8_t* img, const SsmImage& g,
                                               int* expo, uint8_t* img2 = nullptr, SsmImage g2 = SsmImage{},
                                               int* expo2 = nullptr) {
  constexpr int LPR = SsmTile<D>::LPR;
  const int lane = static_cast<int>(threadIdx.x & 31), l4 = lane % LPR;
  const unsigned mask = LPR == 32 ? 0xFFFFFFFFu : (0xFFFFu << (lane & 16));
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const int r = r0 + ssm_tile_row<D>(i);
    if (r >= rows) continue;  // the row's lanes agree
    const float4 v = x[i];
    const float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    int e = __reduce_min_sync(mask, ssm_scale_exp(m));
    if (e == 127) e = 0;  // a zero row
    const float sc = ssm_pow2(e);
    const float4 y = make_float4(v.x * sc, v.y * sc, v.z * sc, v.w * sc);
    ssm_img_put4(img, g, r, 4 * l4, y);
    if (l4 == 0) expo[r] = e;
    if (img2 != nullptr) {
      ssm_img_put4(img2, g2, r, 4 * l4, y);
      if (l4 == 0) expo2[r] = e;
    }
  }
}

// ---------------------------------------------------------------- verify
// The verify's two dense products run on the tensor cores (tcgen05.mma
// kind::f16, fp32 accumulation in TMEM):
//   P = S_0 X^T     (d state rows x 48 columns),
//   G = K X^T       (the retained and block keys, up to 128 rows x 48),
// with X the block's vectors in columns 0-15 k_0..k_15, 16-31 q_0..q_15,
// 32 k_16, 33 q_16 (34-47 zero); the operands are row images (above).
struct SsmVerifyLayout {
  uint32_t a, k, b, u, v, coefA, coefB, L, eL, Lrel, beta, expS, expK, expKb, expB, bar, total;
};
__host__ __device__ inline SsmVerifyLayout ssm_verify_layout(int d, int window) {
  SsmVerifyLayout l{};
  const uint32_t na = static_cast<uint32_t>(d / 64);
  uint32_t o = 0;
  l.a = o;  o += 2u * na * kSsmAtomA;  // checkpoint tile: hi atoms, then lo atoms (128 rows each)
  l.k = o;  o += 2u * na * kSsmAtomA;  // key tile
  l.b = o;  o += 2u * na * kSsmAtomB;  // block-vector tile
  l.u = o;  o += 4u * window * d;      // corrected values: retained, then the block's
  l.v = o;  o += 4u * kRows * d;
  l.coefA = o;  o += 4u * window * kSsmCoefLd;
  l.coefB = o;  o += 4u * window * kSsmCoefLd;
  l.L = o;  o += 8u * window;          // (every region before is a multiple of 16 bytes)
  l.eL = o;  o += 4u * kRows;
  l.Lrel = o;  o += 4u * kRows;
  l.beta = o;  o += 4u * kRows;
  o = (o + 15u) & ~15u;
  l.expS = o;  o += 2u * 4u * 128u;    // two items' checkpoint row exponents (bulk-copied)
  l.expK = o;  o += 2u * 4u * 128u;    // two items' retained-key row exponents (bulk-copied)
  l.expKb = o;  o += 4u * 32u;         // the block keys' exponents (apart: a copy may round up over them)
  l.expB = o;  o += 4u * kSsmN;
  o = (o + 15u) & ~15u;
  l.bar = o;  o += 48u;               // four mbarriers, the TMEM base, the abort flag
  l.total = o + 1024u;                // + alignment of the dynamic shared memory base
  return l;
}
__host__ __device__ inline uint32_t ssm_fold_smem_bytes(int d, int window) {
  return static_cast<uint32_t>(2 * window * d + window) * 4u;
}

// One product tile issue: (A hi, B hi), (A hi, B lo), (A lo, B hi)
// over the K atoms, into TMEM columns d_col..d_col + 47; commit on bar.
template <int D>
__device__ __forceinline__ void ssm_issue(uint32_t d_tmem, const uint8_t* a_tile, const uint8_t* b_tile,
                                          uint64_t* bar) {
  constexpr uint32_t NA = D / 64;
  const uint32_t idesc = idesc_f16(128, kSsmN, false, false, false);
  const uint64_t ah = sw128_desc(smem_u32(a_tile), 16, 1024), al = sw128_desc(smem_u32(a_tile + NA * kSsmAtomA), 16, 1024);
  const uint64_t bh = sw128_desc(smem_u32(b_tile), 16, 1024), bl = sw128_desc(smem_u32(b_tile + NA * kSsmAtomB), 16, 1024);
  const uint64_t ad[3] = {ah, ah, al}, bd[3] = {bh, bl, bh};
#pragma unroll
  for (int pr = 0; pr < 3; ++pr)
#pragma unroll
    for (uint32_t at = 0; at < NA; ++at)
#pragma unroll
      for (uint32_t kk = 0; kk < 4; ++kk)  // 16-element K steps inside the 128-byte atom
        umma_f16(d_tmem, ad[pr] + at * (kSsmAtomA >> 4) + 2 * kk, bd[pr] + at * (kSsmAtomB >> 4) + 2 * kk, idesc,
                 (pr | at | kk) != 0 ? 1u : 0u);
  umma_commit(bar);
}

// This warp's 17 values of one TMEM product row: lane quarter q's row, k
// columns (kind 0: 0-15 and 32) or q columns (kind 1: 16-31 and 33), each
// divided by 2^(row exponent + column exponent).
__device__ __forceinline__ void ssm_tmem_row(uint32_t taddr, int kind, int row_exp, const int* expB, float* out) {
  float v0[16], v1[16];
  tmem_ld16(taddr + 16u * kind, v0);
  tmem_ld16(taddr + 32u, v1);
  tmem_ld_wait();
  const float rs = ssm_pow2(-row_exp);
#pragma unroll
  for (int j = 0; j < 16; ++j) out[j] = v0[j] * rs * ssm_pow2(-expB[16 * kind + j]);
  out[16] = (kind ? v1[1] : v1[0]) * rs * ssm_pow2(-expB[32 + kind]);
}

// Verify: outputs of the 17 block rows, and the block's keys, corrected
// values and log gates staged in the buffer after the pointer (the commit
// decides how many stay).  Persistent: grid min(H B, SMs), 256 threads, one
// (request, head) item at a time.  Per item:
//   1. the block vectors into the B tile, the block's keys into the key
//      tile after the retained rows (and into the buffer's key image); the
//      retained corrected values, v and the log sums by cp.async; the block's
//      log sums;
//   2. wait for the item's checkpoint and retained-key images (bulk copies
//      issued during the previous item); P = S_0 X^T and G = K X^T on the
//      tensor cores; as soon as each product has read its tile, the next
//      item's images are copied in;
//   3. from TMEM: warps 0-3 take the k columns of their lane quarter's rows,
//      warps 4-7 the q columns (P), then the coefficients
//      e^{L_t - L_s} (k_s.k_t) and e^{L_t - L_s} (k_s.q_t) from G;
//   4. per state row: warps 0-3 solve the block's corrected values in token
//      order, warps 4-7 then form the outputs; both first sum the retained
//      tokens' terms.
template <int D>
__global__ void __launch_bounds__(kSsmThreads, 1) ssm_verify_kernel(const SsmArgs a) {
  constexpr uint32_t NA = D / 64;
  constexpr int NXB = kSsmN / SsmTile<D>::RPP;                  // block-vector rows per thread
  constexpr int NBK = (kRows + SsmTile<D>::RPP - 1) / SsmTile<D>::RPP;  // block-key rows per thread
  extern __shared__ uint8_t ssm_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ssm_smem_raw) + 1023) & ~uintptr_t(1023));
  const SsmVerifyLayout l = ssm_verify_layout(D, a.window);
  uint8_t* tA = base + l.a;
  uint8_t* tK = base + l.k;
  uint8_t* tB = base + l.b;
  float* su = reinterpret_cast<float*>(base + l.u);
  float* sv = reinterpret_cast<float*>(base + l.v);
  float* sA = reinterpret_cast<float*>(base + l.coefA);
  float* sB = reinterpret_cast<float*>(base + l.coefB);
  double* sL = reinterpret_cast<double*>(base + l.L);
  float* seL = reinterpret_cast<float*>(base + l.eL);
  float* sLrel = reinterpret_cast<float*>(base + l.Lrel);  // [17] L_t - L_ref of the block rows
  float* sbeta = reinterpret_cast<float*>(base + l.beta);
  int* expS = reinterpret_cast<int*>(base + l.expS);  // [2][128]
  int* expK = reinterpret_cast<int*>(base + l.expK);  // [2][128]
  int* expKb = reinterpret_cast<int*>(base + l.expKb);  // [17], row nb + j
  int* expB = reinterpret_cast<int*>(base + l.expB);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + l.bar);  // checkpoint in, keys in, P done, G done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + l.bar + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + l.bar + 36);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int quarter = warp & 3, kind = warp >> 2;
  const int row = 32 * quarter + lane;  // TMEM lane of this thread
  const SsmImage gS = ssm_image(D, D), gKb = ssm_image(a.window, D), gT = ssm_image(128, D);
  const SsmImage gB = ssm_image(kSsmN, D);
  if (t == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kSsmTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
  pdl_wait();
  const int items = a.heads * a.batch;
  const int kstride = ssm_exp_stride(a.window);
  const uint64_t pol = policy_evict_first();
  // bulk copies (one thread): an item's checkpoint image and exponents into
  // the checkpoint tile / expS[slot], its first nb key rows into the key tile
  // copy groups and product pairs issued / seen complete (thread 0's view),
  // for the drain after a timed-out wait
  uint32_t n_ck = 0, n_keys = 0, n_mma = 0, d_ck = 0, d_keys = 0, d_mma = 0;
  auto issue_ckpt = [&](int it_, int slot) {
    ++n_ck;
    const size_t hbi = static_cast<size_t>(it_ / a.heads) * a.heads + it_ % a.heads;
    const uint8_t* img = a.ckpt + hbi * D * D * 4;
    mbar_expect_tx(&bars[0], 2u * NA * gS.atom + D * 4u);
#pragma unroll
    for (uint32_t h2 = 0; h2 < 2; ++h2)
#pragma unroll
      for (uint32_t at = 0; at < NA; ++at)
        bulk_load(tA + (h2 * NA + at) * kSsmAtomA, img + (h2 * NA + at) * gS.atom, gS.atom, &bars[0], pol);
    bulk_load(expS + slot * 128, a.ckpt_exp + hbi * D, D * 4u, &bars[0], pol);
  };
  auto issue_keys = [&](int it_, int nbi, int slot) {
    ++n_keys;
    nbi = min(max(nbi, 0), a.window - kRows);
    const size_t hbi = static_cast<size_t>(it_ / a.heads) * a.heads + it_ % a.heads;
    const uint8_t* img = a.buf_k + hbi * a.window * D * 4;
    const uint32_t rows_b = static_cast<uint32_t>(nbi) * 128u, eb = static_cast<uint32_t>(ssm_exp_stride(nbi)) * 4u;
    if (nbi == 0) {
      mbar_arrive(&bars[1]);
      return;
    }
    mbar_expect_tx(&bars[1], 2u * NA * rows_b + eb);
#pragma unroll
    for (uint32_t h2 = 0; h2 < 2; ++h2)
#pragma unroll
      for (uint32_t at = 0; at < NA; ++at)
        bulk_load(tK + (h2 * NA + at) * kSsmAtomA, img + (h2 * NA + at) * gKb.atom, rows_b, &bars[1], pol);
    bulk_load(expK + slot * 128, a.buf_kexp + hbi * kstride, eb, &bars[1], pol);
  };
  int nb_next = blockIdx.x < items ? a.ptr[blockIdx.x / a.heads] : 0;
  if (t == 0 && static_cast<int>(blockIdx.x) < items) {
    issue_ckpt(blockIdx.x, 0);
    issue_keys(blockIdx.x, nb_next, 0);
  }
  uint32_t it = 0, mma_ph = 0;  // items walked, products completed
  for (int item = blockIdx.x; item < items; item += gridDim.x, ++it) {
    const int slot = static_cast<int>(it & 1u);
    const int b = item / a.heads, h = item % a.heads;
    const int nb = nb_next;
    const size_t hb = static_cast<size_t>(b) * a.heads + h;
    const size_t blk = hb * kRows, brow = hb * a.window;
    const int nx = item + gridDim.x;
    if (nx < items) {
      nb_next = a.ptr[nx / a.heads];  // used by the next item: its latency hides behind this one
      if (t == kSsmThreads - 32) {    // the next item's block inputs and retained buffer into L2
        const size_t hbn = static_cast<size_t>(nx / a.heads) * a.heads + nx % a.heads;
        bulk_prefetch_l2(a.k + hbn * kRows * D, kRows * D * 4u);
        bulk_prefetch_l2(a.q + hbn * kRows * D, kRows * D * 4u);
        bulk_prefetch_l2(a.v + hbn * kRows * D, kRows * D * 4u);
        prefetch_l2(a.alpha + hbn * kRows);
        prefetch_l2(a.beta + hbn * kRows);
        const int nbn = min(max(nb_next, 0), a.window);
        if (nbn > 0) {
          prefetch_l2(a.buf_L + hbn * a.window + nbn - 1);
          bulk_prefetch_l2(a.buf_u + hbn * a.window * D, nbn * D * 4u);
        }
      }
    }
    const bool bad = nb < 0 || nb + kRows > a.window;  // a pointer the commit never leaves
    const int nt = nb + kRows;
    // ---- 1. the block's operands and the staging copies
    if (!bad) {
      constexpr int R4 = D / 4;
      for (int x = t; x < kRows * R4; x += kSsmThreads) cp_async16(sv + 4 * x, a.v + blk * D + 4 * x);
      for (int x = t; x < nb * R4; x += kSsmThreads) cp_async16(su + 4 * x, a.buf_u + brow * D + 4 * x);
      for (int x = t; x < nb; x += kSsmThreads) cp_async8(sL + x, a.buf_L + brow + x);
      float4 xb[NXB];
      ssm_tile_load<D, NXB>(xb, 0, kSsmN, [&](int r) -> const float* {
        // B rows: 0-15 k_0..k_15, 16-31 q_0..q_15, 32 k_16, 33 q_16, then zero
        if (r < 16 || r == 32) return a.k + (blk + (r < 16 ? r : 16)) * D;
        if (r < 34) return a.q + (blk + (r < 32 ? r - 16 : 16)) * D;
        return nullptr;
      });
      float4 xk[NBK];
      ssm_tile_load<D, NBK>(xk, nb, nt, [&](int r) { return a.k + (blk + r - nb) * D; });
      if (warp == 0) {  // the block's log gate sums, continuing the last retained token's
        const double base_L = nb > 0 ? a.buf_L[brow + nb - 1] : 0.0;
        float la = 0.0f, beta = 0.0f;
        if (lane < kRows) {
          la = fmaxf(logf(a.alpha[blk + lane]), kSsmMinLogGate);
          beta = a.beta[blk + lane];
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {  // the block's own sums stay small: float suffices
          const float y = __shfl_up_sync(0xFFFFFFFFu, la, o);
          if (lane >= o) la += y;
        }
        if (lane < kRows) {
          sL[nb + lane] = base_L + static_cast<double>(la);
          seL[lane] = expf(static_cast<float>(base_L + static_cast<double>(la)));
          sLrel[lane] = la;  // relative to L_ref = the last retained token's sum
          sbeta[lane] = beta;
        }
      }
      ssm_tile_store<D, NXB>(xb, 0, kSsmN, tB, gB, expB);
      // the block's keys after the retained rows: key tile and the buffer's image
      ssm_tile_store<D, NBK>(xk, nb, nt, tK, gT, expKb - nb, a.buf_k + hb * a.window * D * 4, gKb,
                             a.buf_kexp + hb * kstride);
    }
    // ---- 2. the item's images
    if (mbar_wait(&bars[0], it & 1u, abort_flag, a.status)) ++d_ck;
    if (mbar_wait(&bars[1], it & 1u, abort_flag, a.status)) ++d_keys;
    cp_async_wait_all();
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) break;
    if (bad) {
      if (t == 0) {
        atomicOr(a.status, VSD_DEV_BAD_SEQLEN);
        if (nx < items) {
          issue_ckpt(nx, slot ^ 1);
          issue_keys(nx, nb_next, slot ^ 1);
        }
      }
      continue;  // uniform over the CTA
    }
    if (t == 0) {
      tc_fence_after();
      ssm_issue<D>(tmem, tA, tB, &bars[2]);
      ssm_issue<D>(tmem + 64u, tK, tB, &bars[3]);
      ++n_mma;
    }
    // ---- 3. P rows, then the coefficients from G
    const bool p_done = mbar_wait(&bars[2], mma_ph & 1u, abort_flag, a.status);
    tc_fence_after();
    if (t == 0 && nx < items) issue_ckpt(nx, slot ^ 1);  // the checkpoint tile is free
    float P[kRows];
    if (row < D) ssm_tmem_row(taddr, kind, expS[slot * 128 + row], expB, P);
    if (mbar_wait(&bars[3], mma_ph & 1u, abort_flag, a.status) && p_done) ++d_mma;
    ++mma_ph;
    tc_fence_after();
    if (t == 0 && nx < items) issue_keys(nx, nb_next, slot ^ 1);  // the key tile is free
    if (32 * quarter < nt) {  // warp-uniform (the TMEM load is warp-wide); rows >= nt write nothing
      // coefficients of key row s = row against the block's tokens (kind 0: k_t, 1: q_t)
      float g[kRows];
      ssm_tmem_row(taddr + 64u, kind, row < nb ? expK[slot * 128 + row] : expKb[min(row - nb, kRows - 1)], expB, g);
      if (row < nt) {
        // L_s - L_ref once in double, then float differences: the terms that
        // matter (nearby tokens) have small exponents, far ones underflow
        const float Ls = static_cast<float>(sL[row] - (nb > 0 ? sL[nb - 1] : 0.0));
        float* dst = (kind ? sB : sA) + row * kSsmCoefLd;
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          // a: strictly earlier tokens (s < nb + t); b: up to the token itself
          const bool used = row < nb + j + kind;
          dst[j] = used ? expf(sLrel[j] - Ls) * g[j] : 0.0f;
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) break;
    // ---- 4. per state row
    float X[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) X[j] = 0.0f;
    const float* C = kind ? sB : sA;
    if (row < D) {
      // the retained tokens' terms, two tokens' loads ahead of their FMAs
      auto add_rows = [&](int s0, int cnt) {
        float u[2];
        float4 cc[2][5];
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (q < cnt) {
            u[q] = su[(s0 + q) * D + row];
#pragma unroll
            for (int j = 0; j < 5; ++j) cc[q][j] = reinterpret_cast<const float4*>(C + (s0 + q) * kSsmCoefLd)[j];
          }
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (q < cnt) {
#pragma unroll
            for (int j = 0; j < 5; ++j) {
              X[4 * j] = fmaf(cc[q][j].x, u[q], X[4 * j]);
              if (4 * j + 1 < kRows) X[4 * j + 1] = fmaf(cc[q][j].y, u[q], X[4 * j + 1]);
              if (4 * j + 2 < kRows) X[4 * j + 2] = fmaf(cc[q][j].z, u[q], X[4 * j + 2]);
              if (4 * j + 3 < kRows) X[4 * j + 3] = fmaf(cc[q][j].w, u[q], X[4 * j + 3]);
            }
          }
      };
      int s0 = 0;
      for (; s0 + 2 <= nb; s0 += 2) add_rows(s0, 2);
      if (s0 < nb) add_rows(s0, nb - s0);
      if (kind == 0) {
        // the block's corrected values in token order; each one's terms go
        // into the later tokens' sums at once (the dependent chain per
        // token is then one product, not a dot product)
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
          const float ui = sbeta[i] * (sv[i * D + row] - fmaf(seL[i], P[i], X[i]));
          su[(nb + i) * D + row] = ui;
          a.buf_u[(brow + nb + i) * D + row] = ui;
          const float* ci = C + (nb + i) * kSsmCoefLd;
#pragma unroll
          for (int j = i + 1; j < kRows; ++j) X[j] = fmaf(ci[j], ui, X[j]);
        }
      }
    }
    __syncthreads();
    if (row < D && kind == 1) {  // outputs
#pragma unroll
      for (int j = 0; j < kRows; ++j) {
        float acc = fmaf(seL[j], P[j], X[j]);
#pragma unroll
        for (int i = 0; i <= j; ++i) acc = fmaf(C[(nb + i) * kSsmCoefLd + j], su[(nb + i) * D + row], acc);
        a.out[(blk + j) * D + row] = acc;
      }
    }
    if (t < kRows) a.buf_L[brow + nb + t] = sL[nb + t];  // the block's log sums after the pointer
    __syncthreads();  // the shared buffers are reused by the next item
  }
  if (*abort_flag && t == 0) {
    // a wait ran out (VSD_DEV_TIMEOUT is set): let this CTA's copies and
    // products in flight land (each wait bounded) before the shared memory
    // and TMEM are released
    volatile int never = 0;
    for (uint32_t p = d_ck; p < n_ck; ++p) mbar_wait(&bars[0], p & 1u, &never, nullptr);
    for (uint32_t p = d_keys; p < n_keys; ++p) mbar_wait(&bars[1], p & 1u, &never, nullptr);
    for (uint32_t p = d_mma; p < n_mma; ++p) {
      mbar_wait(&bars[2], p & 1u, &never, nullptr);
      mbar_wait(&bars[3], p & 1u, &never, nullptr);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kSsmTmemCols);
  }
}

// ---------------------------------------------------------------- fold
// S = e^{L_{n-1}} S_0 + sum_{s<n} e^{L_{n-1} - L_s} u_s k_s^T for (request,
// head) hb with n retained tokens; S_0 is the checkpoint image, or the fp32
// rows src (set).  The result goes to dst (fp32 rows, get) or, when dst is
// null, back into the checkpoint image (each thread rewrites what it read).
// 256 threads; a 4-lane group holds two rows, lane p float4 chunks p, p + 4,
// ... of both (the group's lanes read consecutive 16-byte pieces of a shared
// key: one wavefront, no bank conflict).
template <int D>
__device__ __forceinline__ void ssm_fold(const SsmArgs& a, size_t hb, int n, const float* src, float* dst, float* sm) {
  constexpr int CPT = D / 4;
  const int t = threadIdx.x, g = t / 4, p = t % 4;
  const size_t brow = hb * a.window;
  const SsmImage gK = ssm_image(a.window, D), gS = ssm_image(D, D);
  const uint8_t* kimg = a.buf_k + brow * D * 4;
  const int* kexp = a.buf_kexp + hb * ssm_exp_stride(a.window);
  uint8_t* cimg = a.ckpt + hb * D * D * 4;
  int* cexp = a.ckpt_exp + hb * D;
  float* sk = sm;          // [n][D]
  float* su = sk + n * D;  // [n][D]
  float* sc = su + n * D;  // [n] e^{L_{n-1} - L_s}
  for (int x = t; x < n * D / 4; x += kSsmThreads) {
    const int r = x / (D / 4), k0 = 4 * (x % (D / 4));
    reinterpret_cast<float4*>(sk)[x] = ssm_img_get4(kimg, gK, r, k0, kexp[r]);
    reinterpret_cast<float4*>(su)[x] = reinterpret_cast<const float4*>(a.buf_u + brow * D)[x];
  }
  const double Ln = n > 0 ? a.buf_L[brow + n - 1] : 0.0;
  for (int x = t; x < n; x += kSsmThreads) sc[x] = expf(static_cast<float>(Ln - a.buf_L[brow + x]));
  const bool has_rows = 2 * g < D;  // warp-uniform (d = 64 leaves warps 4-7 idle)
  float S[2 * CPT];
  if (has_rows) {
    const float e = expf(static_cast<float>(Ln));
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = 2 * g + rr;
#pragma unroll
      for (int c = 0; c < CPT / 4; ++c) {
        const int k0 = 4 * (p + 4 * c);
        const float4 v = src ? *reinterpret_cast<const float4*>(src + static_cast<size_t>(r) * D + k0)
                             : ssm_img_get4(cimg, gS, r, k0, cexp[r]);
        S[rr * CPT + 4 * c] = v.x * e;
        S[rr * CPT + 4 * c + 1] = v.y * e;
        S[rr * CPT + 4 * c + 2] = v.z * e;
        S[rr * CPT + 4 * c + 3] = v.w * e;
      }
    }
  }
  __syncthreads();
  if (!has_rows) return;
  for (int s = 0; s < n; ++s) {
    const float2 uu = *reinterpret_cast<const float2*>(su + s * D + 2 * g);
    const float c0 = sc[s] * uu.x, c1 = sc[s] * uu.y;
    const float4* kk4 = reinterpret_cast<const float4*>(sk + s * D) + p;
#pragma unroll
    for (int c = 0; c < CPT / 4; ++c) {
      const float4 kk = kk4[c * 4];
      S[4 * c] = fmaf(c0, kk.x, S[4 * c]);
      S[4 * c + 1] = fmaf(c0, kk.y, S[4 * c + 1]);
      S[4 * c + 2] = fmaf(c0, kk.z, S[4 * c + 2]);
      S[4 * c + 3] = fmaf(c0, kk.w, S[4 * c + 3]);
      S[CPT + 4 * c] = fmaf(c1, kk.x, S[CPT + 4 * c]);
      S[CPT + 4 * c + 1] = fmaf(c1, kk.y, S[CPT + 4 * c + 1]);
      S[CPT + 4 * c + 2] = fmaf(c1, kk.z, S[CPT + 4 * c + 2]);
      S[CPT + 4 * c + 3] = fmaf(c1, kk.w, S[CPT + 4 * c + 3]);
    }
  }
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = 2 * g + rr;
    if (dst != nullptr) {
      float4* d4 = reinterpret_cast<float4*>(dst + static_cast<size_t>(r) * D) + p;
#pragma unroll
      for (int c = 0; c < CPT / 4; ++c)
        d4[c * 4] = make_float4(S[rr * CPT + 4 * c], S[rr * CPT + 4 * c + 1], S[rr * CPT + 4 * c + 2],
                                S[rr * CPT + 4 * c + 3]);
    } else {
      float m = 0.0f;
#pragma unroll
      for (int j = 0; j < CPT; ++j) m = fmaxf(m, fabsf(S[rr * CPT + j]));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      int e = ssm_scale_exp(m);
      if (e == 127) e = 0;
      const float sc2 = ssm_pow2(e);
#pragma unroll
      for (int c = 0; c < CPT / 4; ++c)
        ssm_img_put4(cimg, gS, r, 4 * (p + 4 * c),
                     make_float4(S[rr * CPT + 4 * c] * sc2, S[rr * CPT + 4 * c + 1] * sc2,
                                 S[rr * CPT + 4 * c + 2] * sc2, S[rr * CPT + 4 * c + 3] * sc2));
      if (p == 0) cexp[r] = e;
    }
  }
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
// folds its retained tokens into the checkpoint.  grid (H, B).
template <int D>
__global__ void __launch_bounds__(kSsmThreads, 2) ssm_flush_kernel(const SsmArgs a) {
  extern __shared__ float4 ssm_smem4[];
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y;
  const int n = ssm_committed(a, b, threadIdx.x == 0 && h == 0);
  if (n + kRows <= a.window || n > a.window) return;  // no flush (n > window: never left by a verify)
  ssm_fold<D>(a, static_cast<size_t>(b) * a.heads + h, n, nullptr, nullptr, reinterpret_cast<float*>(ssm_smem4));
}

// Commit, second part: the pointers (0 after a flush).  One thread per request.
__global__ void ssm_pointer_kernel(const SsmArgs a) {
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.batch) return;
  const int n = ssm_committed(a, b, false);
  a.ptr[b] = (n + kRows > a.window) ? 0 : n;
}

// The effective state of request a.req (the closed form of its checkpoint
// and retained buffer) into a.state_out.  grid (H).
template <int D>
__global__ void __launch_bounds__(kSsmThreads, 2) ssm_state_kernel(const SsmArgs a) {
  extern __shared__ float4 ssm_smem4[];
  const int h = blockIdx.x;
  const int n = min(max(a.ptr[a.req], 0), a.window);
  ssm_fold<D>(a, static_cast<size_t>(a.req) * a.heads + h, n, nullptr,
              a.state_out + static_cast<size_t>(h) * D * D, reinterpret_cast<float*>(ssm_smem4));
}

// Request a.req's checkpoint := a.state_in (fp32 rows), as an image; the
// caller empties its buffer.  grid (H).
template <int D>
__global__ void __launch_bounds__(kSsmThreads, 2) ssm_set_kernel(const SsmArgs a) {
  extern __shared__ float4 ssm_smem4[];
  const int h = blockIdx.x;
  ssm_fold<D>(a, static_cast<size_t>(a.req) * a.heads + h, 0, a.state_in + static_cast<size_t>(h) * D * D,
              nullptr, reinterpret_cast<float*>(ssm_smem4));
}

}  // namespace vsd
