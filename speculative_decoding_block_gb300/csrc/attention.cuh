// attention.cuh -- GQA verify attention of the 17 block rows over the cache.
//
// For request b and KV head h, the 17 block rows x (n_q / n_kv) query heads
// sharing that KV head form one 128-row tile (row = j * group + hq).  Every
// row sees the request's committed keys [0, L_b) and the block's own keys
// 0..j (causal inside the block; OCRia post, speculative-decoding section;
// HunyuanOCR-1.5 summary, section one, inference step 3).  The context is
// split into 128-key chunks (eight 16-token pages, fetched by TMA through
// the page table -- paged KV as in "LLM inference acceleration", section
// two); the block's own 17 keys form one more 32-key chunk read from the
// step's scratch.  A CTA takes `chunks_per_split` consecutive chunks:
//   S = Q K^T     tcgen05.mma, bf16 in, fp32 in TMEM (two S buffers)
//   softmax       one thread per row straight from TMEM, running max / sum
//   O_c = P V     P written as bf16 to shared memory, V read MN-major
// and the per-chunk O_c is folded into registers with the running rescale.
// Split partials (unnormalised O, max, sum) go to a workspace; the last CTA
// of (b, h) merges them in split order and writes the f16 output row.
#pragma once

#include "vsd_common.cuh"

namespace vsd {

constexpr int kAttnThreads = 192;  // warps 0-3 softmax, 4 TMA, 5 MMA

struct AttnArgs {
  int batch_cap;     // rows of the q tile / scratch buffers = max_batch
  int n_q, n_kv, hd, group, rows_valid;
  int chunks_per_split, max_splits;
  int layer, num_pages, pages_per_req;
  const int* ctx_len;      // [B]
  const int* page_table;   // [max_batch][pages_per_req]
  float scale_log2;        // log2(e) / sqrt(hd)
  float* part_o;           // [B][n_kv][max_splits][128][hd]
  float* part_ml;          // [B][n_kv][max_splits][128][2]
  int* counters;           // [B][n_kv]
  __half* out;             // [B*17][n_q*hd]
  int* status;
};

__host__ __device__ inline uint32_t attn_stages(int hd) { return hd == 64 ? 3u : 2u; }
__host__ __device__ inline uint32_t attn_smem_bytes(int hd) {
  const uint32_t q = 128u * hd * 2u, kv = 2u * 128u * hd * 2u;
  return 1024u + q + attn_stages(hd) * kv + 32768u + 1024u;
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kn,
                const __grid_constant__ CUtensorMap tm_vn, const AttnArgs a) {
  constexpr int NS = HD == 64 ? 3 : 2;
  constexpr int NA = HD / 64;  // 64-wide swizzle atoms along head_dim
  constexpr uint32_t QB = 128u * HD * 2u, KVB = 128u * HD * 2u;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* kv_s = smem + QB;                 // stage st: K at st*2*KVB, V at +KVB
  uint8_t* p_s = kv_s + NS * 2 * KVB;        // 2 atoms of [128 rows x 64 keys]
  uint64_t* bars = reinterpret_cast<uint64_t*>(p_s + 32768);
  uint64_t* kvfull = bars;
  uint64_t* kvempty = bars + NS;
  uint64_t* qfull = bars + 2 * NS;
  uint64_t* sfull = qfull + 1;   // [2]
  uint64_t* sfree = sfull + 2;   // [2]
  uint64_t* pfull = sfree + 2;
  uint64_t* ofull = pfull + 1;
  uint64_t* ofree = ofull + 1;
  uint32_t* tmem_p = reinterpret_cast<uint32_t*>(ofree + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_p + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_p + 2);

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_wait();  // ctx_len, q tile and block K/V are produced by earlier kernels of the step
  pdl_launch_dependents();
  const int L = a.ctx_len[b];
  const int n_ctx = (L + 127) >> 7;
  const int n_chunks = n_ctx + 1;
  const int n_splits = (n_chunks + a.chunks_per_split - 1) / a.chunks_per_split;
  if (split >= n_splits) return;
  const int c_begin = split * a.chunks_per_split;
  const int n = min(n_chunks, c_begin + a.chunks_per_split) - c_begin;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kvfull[s], 1);
      mbar_init(&kvempty[s], 1);
    }
    mbar_init(qfull, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], 128);
    }
    mbar_init(pfull, 128);
    mbar_init(ofull, 1);
    mbar_init(ofree, 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_p, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_p;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      mbar_expect_tx(qfull, QB);
      for (int at = 0; at < NA; ++at)
        tma_load_2d(q_s + at * 16384, &tm_q, qfull, at * 64, (b * a.n_kv + h) * 128);
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < n; ++i, ++issued) {
        const int st = i % NS;
        if (i >= NS && !mbar_wait(&kvempty[st], ((i / NS) - 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        uint8_t* ks = kv_s + st * 2 * KVB;
        uint8_t* vs = ks + KVB;
        const int c = c_begin + i;
        if (c < n_ctx) {
          mbar_expect_tx(&kvfull[st], 2u * 128u * HD * 2u);
          for (int p = 0; p < 8; ++p) {
            const int pi = min(c * 8 + p, a.pages_per_req - 1);
            int page = a.page_table[b * a.pages_per_req + pi];
            if (page < 0 || page >= a.num_pages) {
              atomicOr(a.status, VSD_DEV_BAD_PAGE);
              page = 0;
            }
            const int row0 = ((a.layer * a.num_pages + page) * a.n_kv + h) * kPage;
            for (int at = 0; at < NA; ++at) {
              tma_load_2d_hint(ks + at * 16384 + p * 2048, &tm_kc, &kvfull[st], at * 64, row0, pol);
              tma_load_2d_hint(vs + at * 16384 + p * 2048, &tm_vc, &kvfull[st], at * 64, row0, pol);
            }
          }
        } else {
          mbar_expect_tx(&kvfull[st], 2u * 32u * HD * 2u);
          const int row0 = ((a.layer * a.batch_cap + b) * a.n_kv + h) * 32;
          for (int at = 0; at < NA; ++at) {
            tma_load_2d(ks + at * 16384, &tm_kn, &kvfull[st], at * 64, row0);
            tma_load_2d(vs + at * 16384, &tm_vn, &kvfull[st], at * 64, row0);
          }
        }
      }
      if (!ok) {
        volatile int never = 0;
        mbar_wait(qfull, 0, &never, nullptr);
        for (int i = max(0, issued - NS); i < issued; ++i) mbar_wait(&kvfull[i % NS], (i / NS) & 1, &never, nullptr);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t id_s128 = idesc_f16(128, 128, true, true, false);
      const uint32_t id_s32 = idesc_f16(128, 32, true, true, false);
      const uint32_t id_pv = idesc_f16(128, HD, true, true, true);
      const uint32_t qa = smem_u32(q_s), pa = smem_u32(p_s);
      bool ok = mbar_wait(qfull, 0, abort_flag, a.status);
      auto issue_s = [&](int i) -> bool {
        const int st = i % NS;
        if (!mbar_wait(&kvfull[st], (i / NS) & 1, abort_flag, a.status)) return false;
        if (i >= 2 && !mbar_wait(&sfree[i & 1], ((i >> 1) - 1) & 1, abort_flag, a.status)) return false;
        tc_fence_after();
        const uint32_t ka = smem_u32(kv_s + st * 2 * KVB);
        const bool blk = (c_begin + i) >= n_ctx;
        const uint32_t d = tmem + (i & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_f16(d, sw128_desc(qa + off, 16, 1024), sw128_desc(ka + off, 16, 1024), blk ? id_s32 : id_s128,
                   kk > 0 ? 1u : 0u);
        }
        umma_commit(&sfull[i & 1]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int i = 0; ok && i < n; ++i) {
        if (i + 1 < n && !issue_s(i + 1)) break;
        if (!mbar_wait(pfull, i & 1, abort_flag, a.status)) break;
        if (i >= 1 && !mbar_wait(ofree, (i - 1) & 1, abort_flag, a.status)) break;
        tc_fence_after();
        const int st = i % NS;
        const uint32_t va = smem_u32(kv_s + st * 2 * KVB + KVB);
        const bool blk = (c_begin + i) >= n_ctx;
        const int ksteps = blk ? 2 : 8;
        for (int kk = 0; kk < ksteps; ++kk) {
          const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_f16(tmem + 256, sw128_desc(pa + aoff, 16, 1024), sw128_desc(va + kk * 2048, 16384, 1024), id_pv,
                   kk > 0 ? 1u : 0u);
        }
        umma_commit(ofull);
        umma_commit(&kvempty[st]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax rows (warps 0-3)
    const int r = threadIdx.x;  // row == TMEM lane
    const bool row_ok = r < a.rows_valid;
    const int jr = row_ok ? r / a.group : 0;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float o[HD];
#pragma unroll
    for (int d = 0; d < HD; ++d) o[d] = 0.0f;
    float m = -INFINITY, l = 0.0f;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      if (!mbar_wait(&sfull[i & 1], (i >> 1) & 1, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int c = c_begin + i;
      const bool blk = c >= n_ctx;
      const int ncol = blk ? 32 : 128;
      const uint32_t sa = tmem + lane_base + (i & 1) * 128;
      float v[16];
      // pass 1: row max of the chunk
      float cm = -INFINITY;
      for (int c0 = 0; c0 < ncol; c0 += 16) {
        tmem_ld16(sa + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const int key = c0 + t;
          const bool vis = blk ? (key <= jr) : (c * 128 + key < L);
          if (vis && row_ok) cm = fmaxf(cm, v[t] * a.scale_log2);
        }
      }
      const float m_new = fmaxf(m, cm);
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
      const float alpha = exp2f(m - m_use);  // 0 on the first visible chunk (m = -inf)
      // pass 2: probabilities -> bf16 P in shared memory
      float psum = 0.0f;
      for (int c0 = 0; c0 < ncol; c0 += 16) {
        tmem_ld16(sa + c0, v);
        tmem_ld_wait();
        uint32_t w[8];
#pragma unroll
        for (int t = 0; t < 16; t += 2) {
          const int key = c0 + t;
          const bool v0 = row_ok && (blk ? (key <= jr) : (c * 128 + key < L));
          const bool v1 = row_ok && (blk ? (key + 1 <= jr) : (c * 128 + key + 1 < L));
          const float p0 = v0 ? exp2f(v[t] * a.scale_log2 - m_use) : 0.0f;
          const float p1 = v1 ? exp2f(v[t + 1] * a.scale_log2 - m_use) : 0.0f;
          w[t >> 1] = f32x2_to_bf16x2(p0, p1);
          // the sum uses the bf16-rounded probabilities that the PV product uses
          psum += __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(w[t >> 1] & 0xFFFF))) +
                  __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(w[t >> 1] >> 16)));
        }
        const int atom = c0 >> 6, ch = (c0 & 63) >> 3;
        uint8_t* prow = p_s + atom * 16384;
        *reinterpret_cast<uint4*>(prow + sw128_off(r, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(prow + sw128_off(r, ch + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      tc_fence_before();
      mbar_arrive(&sfree[i & 1]);
      fence_proxy_async();
      mbar_arrive(pfull);
      l = l * alpha + psum;
      m = m_new;
      if (!mbar_wait(ofull, i & 1, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int d0 = 0; d0 < HD; d0 += 16) {
        tmem_ld16(tmem + lane_base + 256 + d0, v);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 16; ++t) o[d0 + t] = o[d0 + t] * alpha + v[t];
      }
      tc_fence_before();
      mbar_arrive(ofree);
    }
    if (ok) {
      const size_t pair = static_cast<size_t>(b) * a.n_kv + h;
      const int hq = row_ok ? r % a.group : 0;
      __half* dst = a.out + (static_cast<size_t>(b) * kRows + jr) * (a.n_q * HD) + (h * a.group + hq) * HD;
      if (n_splits == 1) {
        if (row_ok) {
          const float inv = 1.0f / l;
#pragma unroll
          for (int d = 0; d < HD; d += 8) {
            uint4 u;
            u.x = f32x2_to_f16x2(o[d] * inv, o[d + 1] * inv);
            u.y = f32x2_to_f16x2(o[d + 2] * inv, o[d + 3] * inv);
            u.z = f32x2_to_f16x2(o[d + 4] * inv, o[d + 5] * inv);
            u.w = f32x2_to_f16x2(o[d + 6] * inv, o[d + 7] * inv);
            *reinterpret_cast<uint4*>(dst + d) = u;
          }
        }
      } else {
        float* po = a.part_o + ((pair * a.max_splits + split) * 128 + r) * HD;
        float* pml = a.part_ml + ((pair * a.max_splits + split) * 128 + r) * 2;
#pragma unroll
        for (int d = 0; d < HD; d += 4) __stcg(reinterpret_cast<float4*>(po + d), make_float4(o[d], o[d + 1], o[d + 2], o[d + 3]));
        __stcg(reinterpret_cast<float2*>(pml), make_float2(m, l));
        __threadfence();
        named_bar_sync(1, 128);
        if (r == 0) *last_flag = (atomicAdd(&a.counters[pair], 1) == n_splits - 1) ? 1 : 0;
        named_bar_sync(1, 128);
        if (*last_flag) {
          __threadfence();
          float mm = -INFINITY;
          for (int s = 0; s < n_splits; ++s)
            mm = fmaxf(mm, __ldcg(a.part_ml + ((pair * a.max_splits + s) * 128 + r) * 2));
          if (mm == -INFINITY) mm = 0.0f;
          float acc[HD];
#pragma unroll
          for (int d = 0; d < HD; ++d) acc[d] = 0.0f;
          float ls = 0.0f;
          for (int s = 0; s < n_splits; ++s) {
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml + ((pair * a.max_splits + s) * 128 + r) * 2));
            const float w = exp2f(ml.x - mm);
            ls += ml.y * w;
            const float* ps = a.part_o + ((pair * a.max_splits + s) * 128 + r) * HD;
#pragma unroll
            for (int d = 0; d < HD; d += 4) {
              const float4 x = __ldcg(reinterpret_cast<const float4*>(ps + d));
              acc[d] += x.x * w;
              acc[d + 1] += x.y * w;
              acc[d + 2] += x.z * w;
              acc[d + 3] += x.w * w;
            }
          }
          if (row_ok) {
            const float inv = 1.0f / ls;
#pragma unroll
            for (int d = 0; d < HD; d += 8) {
              uint4 u;
              u.x = f32x2_to_f16x2(acc[d] * inv, acc[d + 1] * inv);
              u.y = f32x2_to_f16x2(acc[d + 2] * inv, acc[d + 3] * inv);
              u.z = f32x2_to_f16x2(acc[d + 4] * inv, acc[d + 5] * inv);
              u.w = f32x2_to_f16x2(acc[d + 6] * inv, acc[d + 7] * inv);
              *reinterpret_cast<uint4*>(dst + d) = u;
            }
          }
          if (r == 0) a.counters[pair] = 0;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace vsd
