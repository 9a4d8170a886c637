// quant_kernels.cuh -- round-to-nearest weight quantisers (BF16 master ->
// FP8 E4M3 per-row / NVFP4) and the repacking of canonical weights into the
// GEMM's tile layout.
//
// Scale arithmetic is float32 with one IEEE rounding per operation
// (__fdiv_rn / __fmul_rn, no contraction), and the codes come from the
// hardware's round-to-nearest-even saturating conversions, so the bytes are
// a deterministic function of the master weights:
//   FP8  : s = amax_row / 448;  q = e4m3(w / s)
//   NVFP4: S = amax / 2688;  s_blk = e4m3(amax_blk / (6 S));  q = e2m1(w / (e4m3(s_blk) S))
// (weight recipe: "The Inference Stack Behind OCRia", section "Reducing the
// data moved: workload-aware quantization"; plain rounding replaces the
// pages' activation-aware calibration).
#pragma once

#include "vsd_common.cuh"

namespace vsd {

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t v) { return __uint_as_float(static_cast<uint32_t>(v) << 16); }

__device__ __forceinline__ float block_max_256(float v, float* red) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < 8; ++i) r = fmaxf(r, red[i]);
  __syncthreads();
  return r;
}

// One CTA (256 threads) per row; K even.
__global__ void __launch_bounds__(256) quant_fp8_rowwise_kernel(const uint16_t* w, int K, uint8_t* q, float* scale) {
  __shared__ float red[8];
  const size_t row = blockIdx.x;
  const uint16_t* wr = w + row * K;
  float amax = 0.0f;
  for (int i = threadIdx.x; i < K; i += 256) amax = fmaxf(amax, fabsf(bf16_bits_to_f32(wr[i])));
  amax = block_max_256(amax, red);
  const float s = __fdiv_rn(amax, 448.0f);
  if (threadIdx.x == 0) scale[row] = s;
  uint16_t* qr = reinterpret_cast<uint16_t*>(q + row * K);
  for (int i = threadIdx.x; i < K / 2; i += 256) {
    uint16_t code = 0;
    if (s != 0.0f) {
      const float a = __fdiv_rn(bf16_bits_to_f32(wr[2 * i]), s);
      const float b = __fdiv_rn(bf16_bits_to_f32(wr[2 * i + 1]), s);
      code = f32x2_to_e4m3x2(a, b);
    }
    qr[i] = code;
  }
}

// Pass 1: amax of the whole tensor as float bits (non-negative floats order like ints).
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* w, size_t n, unsigned int* amax_bits) {
  __shared__ float red[8];
  float m = 0.0f;
  for (size_t i = blockIdx.x * 256ull + threadIdx.x; i < n; i += static_cast<size_t>(gridDim.x) * 256ull)
    m = fmaxf(m, fabsf(bf16_bits_to_f32(w[i])));
  m = block_max_256(m, red);
  if (threadIdx.x == 0) atomicMax(amax_bits, __float_as_uint(m));
}

// Pass 2: one thread per 16-element block.  amax_t holds the tensor amax.
__global__ void __launch_bounds__(256) quant_nvfp4_kernel(const uint16_t* w, size_t n_blocks, const float* amax_t,
                                                          uint8_t* q, uint8_t* sblk) {
  const size_t i = blockIdx.x * 256ull + threadIdx.x;
  if (i >= n_blocks) return;
  const float S = __fdiv_rn(*amax_t, 2688.0f);
  const uint16_t* wb = w + i * 16;
  float v[16], am = 0.0f;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    v[e] = bf16_bits_to_f32(wb[e]);
    am = fmaxf(am, fabsf(v[e]));
  }
  uint32_t sb = 0;
  float scale = 0.0f;
  if (S != 0.0f) {
    const float den = __fmul_rn(6.0f, S);
    sb = f32x2_to_e4m3x2(__fdiv_rn(am, den), 0.0f) & 0xFFu;
    scale = __fmul_rn(e4m3_to_f32(sb), S);
  }
  sblk[i] = static_cast<uint8_t>(sb);
  uint16_t out[4] = {0, 0, 0, 0};
  if (scale != 0.0f) {
#pragma unroll
    for (int e = 0; e < 16; e += 4)
      out[e / 4] = f32x4_to_e2m1x4(__fdiv_rn(v[e], scale), __fdiv_rn(v[e + 1], scale), __fdiv_rn(v[e + 2], scale),
                                   __fdiv_rn(v[e + 3], scale));
  }
  uint2 pk;
  pk.x = static_cast<uint32_t>(out[0]) | (static_cast<uint32_t>(out[1]) << 16);
  pk.y = static_cast<uint32_t>(out[2]) | (static_cast<uint32_t>(out[3]) << 16);
  *reinterpret_cast<uint2*>(q + i * 8) = pk;
}

// Pass 3: amax -> tensor scale, in place.
__global__ void nvfp4_tensor_scale_kernel(float* s) { *s = __fdiv_rn(*s, 2688.0f); }

// ------------------------------------------------------------------ packing
// perm[p] = source row of packed row p, or -1 for a zero row.

// FP8: tiles [n_tiles][k_tiles][128][64] bytes; row scales follow the permutation.
__global__ void pack_fp8_kernel(const uint8_t* q, const float* scale, const int* perm, int n_packed, int K,
                                int k_tiles, uint8_t* tiles, float* row_scale) {
  const int tile = blockIdx.y, kt = blockIdx.x;
  uint8_t* dst = tiles + (static_cast<size_t>(tile) * k_tiles + kt) * 8192;
  for (int i = threadIdx.x; i < 8192; i += blockDim.x) {
    const int r = i >> 6, c = i & 63;
    const int p = tile * 128 + r, k = kt * 64 + c;
    const int src = p < n_packed ? perm[p] : -1;
    dst[i] = (src >= 0 && k < K) ? q[static_cast<size_t>(src) * K + k] : 0;
  }
  if (kt == 0)
    for (int r = threadIdx.x; r < 128; r += blockDim.x) {
      const int p = tile * 128 + r;
      if (p < n_packed) row_scale[p] = perm[p] >= 0 ? scale[perm[p]] : 0.0f;
    }
}

// NVFP4: tiles [n_tiles][k_tiles][128 x 32 value bytes | 128 x 4 scale bytes].
__global__ void pack_fp4_kernel(const uint8_t* q, const uint8_t* sblk, const int* perm, int n_packed, int K,
                                int k_tiles, uint8_t* tiles) {
  const int tile = blockIdx.y, kt = blockIdx.x;
  uint8_t* dst = tiles + (static_cast<size_t>(tile) * k_tiles + kt) * 4608;
  for (int i = threadIdx.x; i < 4608; i += blockDim.x) {
    uint8_t v = 0;
    if (i < 4096) {
      const int r = i >> 5, c = i & 31;
      const int p = tile * 128 + r, kb = kt * 32 + c;  // byte column
      const int src = p < n_packed ? perm[p] : -1;
      if (src >= 0 && kb < K / 2) v = q[static_cast<size_t>(src) * (K / 2) + kb];
    } else {
      const int j = i - 4096, r = j >> 2, c = j & 3;
      const int p = tile * 128 + r, kb = kt * 4 + c;
      const int src = p < n_packed ? perm[p] : -1;
      if (src >= 0 && kb < K / 16) v = sblk[static_cast<size_t>(src) * (K / 16) + kb];
    }
    dst[i] = v;
  }
}

// Per-row fp32 scale of every packed row (zero for padding rows).
__global__ void pack_row_scale_kernel(const float* src_scale, const int* perm, int n_packed, float* row_scale) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p < n_packed) row_scale[p] = perm[p] >= 0 ? src_scale[perm[p]] : 0.0f;
}

// BF16 -> f16 tiles [n_tiles][k_tiles][128 rows x 64 k] laid out exactly as
// the MMA reads them from shared memory (128-byte swizzle: 16-byte chunk c of
// tile row r at r * 128 + ((c ^ (r & 7)) << 4)), so one 1-D bulk copy moves a
// tile; k beyond K and padding rows are zero.  The GEMM consumes 16-bit
// weights as f16: exact for magnitudes in [2^-14, 65504], nearest f16 below.
__global__ void pack_bf16_tiles_kernel(const uint16_t* w, const int* perm, int n_packed, int K, int k_tiles,
                                       uint16_t* tiles) {
  const int tile = blockIdx.y, kt = blockIdx.x;
  uint16_t* dst = tiles + (static_cast<size_t>(tile) * k_tiles + kt) * 8192;
  for (int i = threadIdx.x; i < 8192; i += blockDim.x) {
    const int r = i >> 6, col = i & 63;
    const int p = tile * 128 + r, k = kt * 64 + col;
    const int src = p < n_packed ? perm[p] : -1;
    const float v =
        (src >= 0 && k < K) ? __uint_as_float(static_cast<uint32_t>(w[static_cast<size_t>(src) * K + k]) << 16) : 0.0f;
    dst[sw128_off(r, col >> 3) / 2 + (col & 7)] = __half_as_ushort(__float2half_rn(v));
  }
}

}  // namespace vsd
