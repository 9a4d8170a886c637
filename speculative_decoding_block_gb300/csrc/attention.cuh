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
// step's scratch.  Work items are (request, KV head, split of
// `chunks_per_split` consecutive chunks); persistent CTAs (one per SM) walk
// the item list, which every CTA derives from the caller's sequence lengths.
// Per chunk:
//   S = Q K^T     tcgen05.mma, bf16 in, fp32 in TMEM (two S buffers)
//   softmax       two threads per row (each half of the chunk's columns)
//                 straight from TMEM, running max shared through smem
//   O_c = P V     P written as bf16 to shared memory, V read MN-major
// and the per-chunk O_c is folded into registers with the running rescale.
// Context pages do not depend on the preceding kernels of the step, so the
// page-table entries of the first chunks are read before the grid-dependency
// wait (their copies follow the q tile after it).  Split partials
// (unnormalised O, max, sum) go to a workspace; once all of a (request, head)
// pair's partials are in, each of its splits merges a slice of the pair's
// rows in split order and writes those f16 output rows.
#pragma once

#include "vsd_common.cuh"

namespace vsd {

constexpr int kAttnThreads = 320;  // warps 0-7 softmax, 8 TMA, 9 MMA
constexpr int kMaxReqs = 1024;     // requests whose item offsets fit in shared memory

struct AttnArgs {
  int batch;         // requests in this step
  int batch_cap;     // rows of the q tile / scratch buffers = max_batch
  int n_q, n_kv, hd, group, rows_valid;
  int chunks_per_split, max_splits;  // smallest split the host allows; capacity of the partials
  int layer, num_pages, pages_per_req, max_tokens;
  const int* seq_lens;     // [B] caller's committed lengths (validated here)
  const int* page_table;   // [max_batch][pages_per_req]
  float scale_log2;        // log2(e) / sqrt(hd)
  float* part_o;           // [B][n_kv][max_splits][2 halves][128][hd / 2] unnormalised partial O
  float* part_ml;          // [B][n_kv][max_splits][128][2]
  int* counters;           // [2][batch_cap][n_kv]: splits arrived / done merging, per pair (zero between launches)
  __half* out;             // [B*17][n_q*hd] f16 (hi)
  size_t out_lo;           // elements from a hi output value to its lo copy, f16(o - hi) (0: hi only)
  int q_lo_rows;           // rows of the q-tile map from a hi tile to its lo tile (0: no lo tile)
  int* status;
  Trace trace;
};

// K and V of a chunk travel in separate rings of this depth (a K slot frees
// when its S product is done, a V slot when its PV product is done)
__host__ __device__ inline uint32_t attn_stages(int hd) { return hd == 64 ? 3u : 1u; }
// q tile (hi, lo), K/V stages, P tile (hi, lo), then barriers (256 B), row
// statistics (4 KB) and item offsets
constexpr int kMaxItemPages = 1024;  // page-table entries of one item staged in shared memory (128 chunks)
__host__ __device__ inline uint32_t attn_smem_bytes(int hd) {
  const uint32_t q = 128u * hd * 2u, kv = 2u * 128u * hd * 2u;
  return 1024u + 2u * q + attn_stages(hd) * kv + 2u * 32768u + 256u + 4096u + 4u * (kMaxReqs + 1) +
         4u * kMaxItemPages;
}

__device__ __forceinline__ int valid_len(const AttnArgs& a, int b) {
  const int L = a.seq_lens[b];
  return (L >= 0 && L + kRows <= a.max_tokens) ? L : 0;
}

// Eight values v[i] * scale as f16 hi words and f16 lo words (v*scale - hi), packed in pairs.
__device__ __forceinline__ void f16_pairs8(const float* v, float scale, uint32_t* hw, uint32_t* lw) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float y0 = v[2 * e] * scale, y1 = v[2 * e + 1] * scale;
    hw[e] = f32x2_to_f16x2(y0, y1);
    const __half2 h2 = *reinterpret_cast<const __half2*>(&hw[e]);
    lw[e] = f32x2_to_f16x2(y0 - __low2float(h2), y1 - __high2float(h2));
  }
}

// Packed pairs of f32 operations (two IEEE results per instruction).
__device__ __forceinline__ void fma2_bc(float a0, float a1, float b, float c, float& d0, float& d1) {
  asm("{\n .reg .b64 x, y, z, r;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %4};\n mov.b64 z, {%5, %5};\n"
      " fma.rn.f32x2 r, x, y, z;\n mov.b64 {%0, %1}, r;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void sub2(float a0, float a1, float b0, float b1, float& d0, float& d1) {
  asm("{\n .reg .b64 x, y, r;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n sub.rn.f32x2 r, x, y;\n"
      " mov.b64 {%0, %1}, r;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{\n .reg .b64 x, y, r;\n mov.b64 x, {%0, %1};\n mov.b64 y, {%2, %3};\n add.rn.f32x2 r, x, y;\n"
      " mov.b64 {%0, %1}, r;\n}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// The maximum a row's softmax weights are taken against moves only when a
// chunk exceeds it by more than this (log2 units): weights stay <= 2^8.
constexpr float kRescaleLog2 = 8.0f;

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kc,
                const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_kn,
                const __grid_constant__ CUtensorMap tm_vn, const AttnArgs a) {
  constexpr int NS = HD == 64 ? 3 : 1;
  constexpr int NA = HD / 64;   // 64-wide swizzle atoms along head_dim
  constexpr int HH = HD / 2;    // output columns per softmax thread
  constexpr uint32_t QB = 128u * HD * 2u, KVB = 128u * HD * 2u;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // Q and P enter the MMAs as BF16 pairs hi = bf16(x), lo = bf16(x - hi)
  // (two MMAs each), so that scores and weights carry about 16 significant bits
  uint8_t* q_s = smem;                       // hi tile, lo tile at + QB
  uint8_t* kv_s = smem + 2 * QB;             // K slot st at st*KVB, V slot st at (NS + st)*KVB
  uint8_t* p_s = kv_s + NS * 2 * KVB;        // hi: 2 atoms of [128 rows x 64 keys]; lo at + 32768
  uint64_t* bars = reinterpret_cast<uint64_t*>(p_s + 2 * 32768);
  uint64_t* kfull = bars;
  uint64_t* kempty = bars + NS;
  uint64_t* vfull = bars + 2 * NS;
  uint64_t* vempty = bars + 3 * NS;
  uint64_t* qfull = bars + 4 * NS;
  uint64_t* qempty = qfull + 1;  // the item's S products are done with the q tile
  uint64_t* sfull = qempty + 1;  // [2]
  uint64_t* sfree = sfull + 2;   // [2]
  uint64_t* pfull = sfree + 2;
  uint64_t* ofull = pfull + 1;
  uint64_t* ofree = ofull + 1;
  uint64_t* pfree = ofree + 1;   // a chunk's PV product is done: its P tile may be rewritten
  uint32_t* tmem_p = reinterpret_cast<uint32_t*>(pfree + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_p + 1);
  volatile int* n_items = reinterpret_cast<volatile int*>(tmem_p + 3);
  float* xstat = reinterpret_cast<float*>(p_s + 2 * 32768 + 256);  // [2 parity][2 halves][128] maxima; then [2][2][128] sums
  int* item_off = reinterpret_cast<int*>(p_s + 2 * 32768 + 256 + 4096);  // [B + 1] first item of each request
  int* item_pages = item_off + (kMaxReqs + 1);  // [kMaxItemPages] the producer's current item's pages

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* cps_s = reinterpret_cast<volatile int*>(tmem_p + 4);
  volatile int* sum_s = reinterpret_cast<volatile int*>(tmem_p + 5);
  auto chunks_of = [&](int b) { return (valid_len(a, b) + 127) / 128 + 1; };
  // the caller's lengths are read first, so that the loads overlap the set-up
  int mine = 0;
  for (int b = threadIdx.x; b < a.batch; b += blockDim.x) mine += chunks_of(b);

  if (threadIdx.x == 0) {
    trace_start(a.trace);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    mbar_init(qfull, 1);
    mbar_init(qempty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], 256);
    }
    mbar_init(pfull, 256);
    mbar_init(ofull, 1);
    mbar_init(ofree, 256);
    mbar_init(pfree, 1);
    *abort_flag = 0;
    *sum_s = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_p, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Split size: the smallest number of chunks per split (at least the
  // host's) whose items fit in one round of the grid, so that each CTA
  // walks about one item.  seq_lens is the caller's input and does not
  // change during the step, so every CTA derives the same split.
  {
    if (mine) atomicAdd(const_cast<int*>(sum_s), mine);
    __syncthreads();
    const int total_chunks = *sum_s * a.n_kv;
    int c = max(a.chunks_per_split, (total_chunks + gridDim.x - 1) / gridDim.x);
    for (;; ++c) {  // ends: at c = the longest request's chunk count every request is one split
      __syncthreads();
      if (threadIdx.x == 0) *sum_s = 0;
      __syncthreads();
      int items = 0;
      for (int b = threadIdx.x; b < a.batch; b += blockDim.x) items += (chunks_of(b) + c - 1) / c;
      if (items) atomicAdd(const_cast<int*>(sum_s), items);
      __syncthreads();
      if (*sum_s * a.n_kv <= static_cast<int>(gridDim.x) || *sum_s == a.batch) break;
    }
    if (warp == 0) {
      // item list: request-major, then KV head, then split; each request's
      // first item by an exclusive prefix sum, 32 requests at a time
      int base = 0;
      for (int b0 = 0; b0 < a.batch; b0 += 32) {
        const int b = b0 + lane;
        const int cnt = b < a.batch ? a.n_kv * ((chunks_of(b) + c - 1) / c) : 0;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        if (b < a.batch) item_off[b] = base + incl - cnt;
        base += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (lane == 0) {
        item_off[a.batch] = base;
        *n_items = base;
        *cps_s = c;
      }
    }
    __syncthreads();
  }
  const uint32_t tmem = *tmem_p;
  const int total = *n_items;
  const int cps = *cps_s;
  auto splits_of = [&](int b) { return (chunks_of(b) + cps - 1) / cps; };
  pdl_launch_dependents();
  if (threadIdx.x == 0) trace_point(a.trace, 1);

  struct Item {
    int b, h, split, n_splits, L, n_ctx, c_begin, n;
  };
  auto decode = [&](int it) {
    Item x;
    int lo = 0, hi = a.batch - 1;  // last request whose first item is <= it
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (item_off[mid] <= it) lo = mid;
      else hi = mid - 1;
    }
    x.b = lo;
    x.n_splits = splits_of(x.b);
    const int rem = it - item_off[x.b];
    x.h = rem / x.n_splits;
    x.split = rem % x.n_splits;
    x.L = valid_len(a, x.b);
    x.n_ctx = (x.L + 127) >> 7;
    x.c_begin = x.split * cps;
    x.n = min(x.n_ctx + 1, x.c_begin + cps) - x.c_begin;
    return x;
  };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer (whole warp)
    // Lanes 0..7 each fetch one 16-row page of a context chunk (page-table
    // read and K/V copies in parallel); lane 0 arms the barriers and fetches
    // the q tile and the block's own rows.
    {
      const uint64_t pol = policy_evict_first();
      // The page-table entries of an item's context chunks, read into shared
      // memory in one pass (eight loads in flight per lane) before its first
      // copy: no chunk's copies then wait for a page-table round trip.
      // false when the item has more pages than the staging holds (the
      // chunks then read their entries one by one).
      auto stage_pages = [&](const Item& x) -> bool {
        const int npg = max(0, min(x.n_ctx, x.c_begin + x.n) - x.c_begin) * 8;
        if (npg > kMaxItemPages) return false;
        for (int j0 = 0; j0 < npg; j0 += 256) {
          int v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = j0 + u * 32 + lane;
            v[u] = j < npg ? a.page_table[x.b * a.pages_per_req + min(x.c_begin * 8 + j, a.pages_per_req - 1)] : 0;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (j0 + u * 32 + lane < npg) item_pages[j0 + u * 32 + lane] = v[u];
        }
        __syncwarp();
        return true;
      };
      // chunk i of item x, global chunk number g: K then V, each once its slot is free
      // (staged: the item's pages are in item_pages)
      auto issue = [&](const Item& x, int i, int g, bool staged) -> bool {
        const int st = g % NS;
        uint8_t* ks = kv_s + st * KVB;
        uint8_t* vs = kv_s + (NS + st) * KVB;
        const int c = x.c_begin + i;
        const bool ctx = c < x.n_ctx;
        int row0 = 0;
        if (ctx && lane < 8) {  // lane p: page p of the chunk
          const int pi = min(c * 8 + lane, a.pages_per_req - 1);
          int page = staged ? item_pages[i * 8 + lane] : a.page_table[x.b * a.pages_per_req + pi];
          if (page < 0 || page >= a.num_pages) {
            atomicOr(a.status, VSD_DEV_BAD_PAGE);
            page = 0;
          }
          row0 = ((a.layer * a.num_pages + page) * a.n_kv + x.h) * kPage;
        } else if (!ctx) {
          row0 = ((a.layer * a.batch_cap + x.b) * a.n_kv + x.h) * 32;
        }
        const uint32_t bytes = (ctx ? 128u : 32u) * HD * 2u;
        for (int part = 0; part < 2; ++part) {  // 0: K, 1: V
          uint64_t* full = part ? &vfull[st] : &kfull[st];
          uint64_t* empty = part ? &vempty[st] : &kempty[st];
          uint8_t* dst = part ? vs : ks;
          if (g >= NS && !mbar_wait(empty, ((g / NS) - 1) & 1, abort_flag, a.status)) return false;
          if (lane == 0) mbar_expect_tx(full, bytes);
          __syncwarp();
          if (ctx && lane < 8) {
#pragma unroll
            for (int at = 0; at < NA; ++at)
              tma_load_2d_hint(dst + at * 16384 + lane * 2048, part ? &tm_vc : &tm_kc, full, at * 64, row0, pol);
          } else if (!ctx && lane == 0) {
            for (int at = 0; at < NA; ++at) tma_load_2d(dst + at * 16384, part ? &tm_vn : &tm_kn, full, at * 64, row0);
          }
          __syncwarp();
        }
        return true;
      };
      // The first item's page-table entries are read before the dependency
      // wait (the table is the caller's).  Its copies are issued after the
      // wait, behind the q tile: the cooperative grid starts only once the
      // previous kernel has left, so copies issued earlier would only queue
      // ahead of q.
      bool staged = false;
      if (static_cast<int>(blockIdx.x) < total) staged = stage_pages(decode(blockIdx.x));
      pdl_wait();  // q tiles and the block's K/V come from the QKV kernel
      if (lane == 0) trace_point(a.trace, 2);
      int g = 0, ic = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < total; it += gridDim.x, ++ic) {
        const Item x = decode(it);
        if (ic > 0 && !mbar_wait(qempty, (ic - 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const int q_row = (x.b * a.n_kv + x.h) * 128;
          mbar_expect_tx(qfull, a.q_lo_rows ? 2 * QB : QB);
          for (int at = 0; at < NA; ++at) {
            tma_load_2d(q_s + at * 16384, &tm_q, qfull, at * 64, q_row);
            if (a.q_lo_rows) tma_load_2d(q_s + QB + at * 16384, &tm_q, qfull, at * 64, a.q_lo_rows + q_row);
          }
        }
        if (ic > 0) staged = stage_pages(x);
        for (int i = 0; i < x.n; ++i, ++g) {
          if (!issue(x, i, g, staged)) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) {
        volatile int never = 0;
        mbar_wait(qfull, ic & 1, &never, nullptr);
        for (int i = max(0, g - NS); i < g; ++i) {
          mbar_wait(&kfull[i % NS], (i / NS) & 1, &never, nullptr);
          mbar_wait(&vfull[i % NS], (i / NS) & 1, &never, nullptr);
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t id_s128 = idesc_f16(128, 128, true, true, false);
      const uint32_t id_s32 = idesc_f16(128, 32, true, true, false);
      const uint32_t id_pv = idesc_f16(128, HD, true, true, true);
      const uint32_t qa = smem_u32(q_s), pa = smem_u32(p_s);
      int g0 = 0, ic = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < total; it += gridDim.x, ++ic) {
        const Item x = decode(it);
        if (!mbar_wait(qfull, ic & 1, abort_flag, a.status)) break;
        auto issue_s = [&](int i) -> bool {
          const int g = g0 + i, st = g % NS;
          if (!mbar_wait(&kfull[st], (g / NS) & 1, abort_flag, a.status)) return false;
          if (g >= 2 && !mbar_wait(&sfree[g & 1], ((g >> 1) - 1) & 1, abort_flag, a.status)) return false;
          tc_fence_after();
          const uint32_t ka = smem_u32(kv_s + st * KVB);
          const bool blk = (x.c_begin + i) >= x.n_ctx;
          const uint32_t d = tmem + (g & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint64_t kd = sw128_desc(ka + off, 16, 1024);
            umma_f16(d, sw128_desc(qa + off, 16, 1024), kd, blk ? id_s32 : id_s128, kk > 0 ? 1u : 0u);
            if (a.q_lo_rows) umma_f16(d, sw128_desc(qa + QB + off, 16, 1024), kd, blk ? id_s32 : id_s128, 1u);
          }
          umma_commit(&sfull[g & 1]);
          umma_commit(&kempty[st]);
          if (i + 1 == x.n) umma_commit(qempty);  // last use of this item's q tile
          return true;
        };
        ok = issue_s(0);
        if (ic == 0) trace_point(a.trace, 3);
        for (int i = 0; ok && i < x.n; ++i) {
          const int g = g0 + i;
          if (i + 1 < x.n && !issue_s(i + 1)) {
            ok = false;
            break;
          }
          // P of chunk i is in shared memory (and any rescale of O is done);
          // the item's first product overwrites O once the previous item's O is read
          if (!mbar_wait(pfull, g & 1, abort_flag, a.status) ||
              (i == 0 && ic > 0 && !mbar_wait(ofree, (ic - 1) & 1, abort_flag, a.status))) {
            ok = false;
            break;
          }
          const int st = g % NS;
          if (!mbar_wait(&vfull[st], (g / NS) & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t va = smem_u32(kv_s + (NS + st) * KVB);
          const bool blk = (x.c_begin + i) >= x.n_ctx;
          const int ksteps = blk ? 2 : 8;
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint64_t vd = sw128_desc(va + kk * 2048, 16384, 1024);
            umma_f16(tmem + 256, sw128_desc(pa + aoff, 16, 1024), vd, id_pv, (i > 0 || kk > 0) ? 1u : 0u);
            umma_f16(tmem + 256, sw128_desc(pa + 32768 + aoff, 16, 1024), vd, id_pv, 1u);
          }
          umma_commit(pfree);
          if (i + 1 == x.n) umma_commit(ofull);  // the item's O is complete
          umma_commit(&vempty[st]);
        }
        g0 += x.n;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int q4 = warp & 3, hf = warp >> 2;  // TMEM lane quarter, column half
    const int r = q4 * 32 + lane;             // row == TMEM lane
    const bool row_ok = r < a.rows_valid;
    const int jr = row_ok ? r / a.group : 0;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const int bar_id = 2 + q4;  // the 64 threads that share these rows
    int g0 = 0, ic = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < total; it += gridDim.x, ++ic) {
      const Item x = decode(it);
      float o[HH];
      // m: the maximum this row's P values are taken against (log2 units)
      float m = -INFINITY, l = 0.0f;
      const uint32_t o_tmem = tmem + lane_base + 256 + hf * HH;  // this thread's O columns
      for (int i = 0; i < x.n; ++i) {
        const int g = g0 + i;
        if (!mbar_wait(&sfull[g & 1], (g >> 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        if (threadIdx.x == 0 && ic == 0) trace_point(a.trace, i == 0 ? 4 : 5);
        tc_fence_after();
        const int c = x.c_begin + i;
        const bool blk = c >= x.n_ctx;
        const bool need_mask = blk || (c * 128 + 128 > x.L) || !row_ok;
        const int ncol = blk ? 16 : 64;        // this thread's columns of the chunk
        const int col0 = hf * ncol;
        const uint32_t sa = tmem + lane_base + (g & 1) * 128 + col0;
        float s[64];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q * 16 < ncol) tmem_ld16(sa + q * 16, s + q * 16);
        tmem_ld_wait();
        // visible keys of this row form a prefix [0, lim) of the thread's columns:
        // block keys 0..j (causal), context keys below L, nothing for padding rows
        // (the scale is applied once to the maximum and fused into the
        // exponent's argument below: it is positive, so it commutes with max)
        const float sl = a.scale_log2;
        float cm = -INFINITY;
        if (!need_mask) {  // a full context chunk: 64 columns, all visible
#pragma unroll
          for (int t = 0; t < 64; ++t) cm = fmaxf(cm, s[t]);
        } else {
          const int lim = !row_ok ? 0 : min(ncol, blk ? jr + 1 - col0 : x.L - c * 128 - col0);
#pragma unroll
          for (int t = 0; t < 64; ++t) {
            s[t] = t < lim ? s[t] : -INFINITY;
            cm = fmaxf(cm, s[t]);
          }
        }
        cm *= sl;
        float* xs = xstat + (g & 1) * 256;
        xs[hf * 128 + r] = cm;
        named_bar_sync(bar_id, 64);
        cm = fmaxf(xs[r], xs[128 + r]);
        // O accumulates over the item's chunks in TMEM.  The maximum moves up
        // only when a chunk's maximum exceeds it by more than kRescaleLog2, so
        // P <= 2^8 (exact in the BF16 pairs and f32 sums); then the rows of O
        // accumulated so far are scaled by 2^(m_old - m_new) before this
        // chunk's product is added.
        float alpha = 1.0f;
        bool rescale = false;
        if (m == -INFINITY) {
          m = cm;  // the first chunk with a visible key (O rows are still 0)
        } else if (cm > m + kRescaleLog2) {
          alpha = ex2(m - cm);
          m = cm;
          rescale = true;
        }
        const float m_use = (m == -INFINITY) ? 0.0f : m;
        // the previous chunk's PV product must be done before its P tile is
        // rewritten, and before O is read for a rescale
        if (g >= 1 && !mbar_wait(pfree, (g - 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xFFFFFFFFu, rescale)) {
          float v[16];
#pragma unroll
          for (int d0 = 0; d0 < HH; d0 += 16) {
            tmem_ld16(o_tmem + d0, v);
            tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < 16; ++t) v[t] *= alpha;
            tmem_st16_wait(o_tmem + d0, v);
          }
        }
        // probabilities -> BF16 pairs P_hi, P_lo, one 16-byte chunk (8 keys) at a
        // time: keys [col0, col0 + ncol) of row r live in atom col0 / 64.  The
        // exponent arguments, the lo parts and the row sums run as packed
        // pairs (the softmax's instruction stream sets the chunk time).
        float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
        for (int t = 0; t < 64; t += 8) {
          if (t < ncol) {
            uint32_t w[4], wl[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              float x0, x1, l0, l1;
              fma2_bc(s[t + e], s[t + e + 1], sl, -m_use, x0, x1);
              const float p0 = ex2(x0), p1 = ex2(x1);
              w[e >> 1] = f32x2_to_bf16x2(p0, p1);
              const float h0 = __uint_as_float(w[e >> 1] << 16), h1 = __uint_as_float(w[e >> 1] & 0xFFFF0000u);
              sub2(p0, p1, h0, h1, l0, l1);
              wl[e >> 1] = f32x2_to_bf16x2(l0, l1);
              add2(ps0, ps1, p0, p1);
            }
            const int key = col0 + t;
            const uint32_t o = (key >> 6) * 16384 + sw128_off(r, (key & 63) >> 3);
            *reinterpret_cast<uint4*>(p_s + o) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(p_s + 32768 + o) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
          }
        }
        tc_fence_before();
        mbar_arrive(&sfree[g & 1]);
        fence_proxy_async();
        mbar_arrive(pfull);
        l = l * alpha + (ps0 + ps1);
      }
      g0 += x.n;
      if (!ok) break;
      // the item's O once its last product is done
      if (!mbar_wait(ofull, ic & 1, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int d0 = 0; d0 < HH; d0 += 16) {
        tmem_ld16(o_tmem + d0, o + d0);
        tmem_ld_wait();
      }
      tc_fence_before();
      mbar_arrive(ofree);
      if (threadIdx.x == 0 && ic == 0) trace_point(a.trace, 6);
      // row sum over both halves
      float* xl = xstat + 512 + (ic & 1) * 256;
      xl[hf * 128 + r] = l;
      named_bar_sync(bar_id, 64);
      const float lt = xl[r] + xl[128 + r];
      const size_t pair = static_cast<size_t>(x.b) * a.n_kv + x.h;
      const int hq = row_ok ? r % a.group : 0;
      __half* dst =
          a.out + (static_cast<size_t>(x.b) * kRows + jr) * (a.n_q * HD) + (x.h * a.group + hq) * HD + hf * HH;
      if (x.n_splits == 1) {
        if (row_ok) {
          const float inv = 1.0f / lt;
#pragma unroll
          for (int d = 0; d < HH; d += 8) {
            uint32_t hw[4], lw[4];
            f16_pairs8(o + d, inv, hw, lw);
            *reinterpret_cast<uint4*>(dst + d) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            if (a.out_lo) *reinterpret_cast<uint4*>(dst + a.out_lo + d) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        continue;
      }
      // split partial: unnormalised O as [2 halves][128 rows][HD/2] fp32 per
      // (pair, split), staged through shared memory (the P tile is free once
      // the last PV product is done) so that the global writes are coalesced
      constexpr int Q4 = HH / 4;                 // float4 per half row
      constexpr int NF4 = 128 * Q4;              // float4 per half tile
      float4* stage = reinterpret_cast<float4*>(p_s);
      auto slot = [&](int row, int d4) { return row * Q4 + (d4 ^ (row & 7)); };  // bank-spread
      const size_t split_idx = pair * a.max_splits + x.split;
      float4* po = reinterpret_cast<float4*>(a.part_o + split_idx * 128 * HD);
      for (int hh = 0; hh < 2; ++hh) {
        if (hf == hh) {
#pragma unroll
          for (int d4 = 0; d4 < Q4; ++d4)
            stage[slot(r, d4)] = make_float4(o[4 * d4], o[4 * d4 + 1], o[4 * d4 + 2], o[4 * d4 + 3]);
        }
        named_bar_sync(1, 256);
#pragma unroll
        for (int j = threadIdx.x; j < NF4; j += 256) __stcg(po + hh * NF4 + j, stage[slot(j / Q4, j % Q4)]);
        named_bar_sync(1, 256);
      }
      if (hf == 0) __stcg(reinterpret_cast<float2*>(a.part_ml) + split_idx * 128 + r, make_float2(m, lt));
      // Every split of the pair then merges a slice of the pair's rows, once
      // all of the pair's partials are written.  The splits of a pair run at
      // the same time: with more than one split per request every CTA has at
      // most one item (the split size is chosen so), and the grid (at most
      // one CTA per SM) is resident as a whole once the previous kernel's
      // CTAs have left.  The wait is bounded all the same.
      __threadfence();
      named_bar_sync(1, 256);
      int* arrived = a.counters + pair;
      int* departed = a.counters + static_cast<size_t>(a.batch_cap) * a.n_kv + pair;
      if (threadIdx.x == 0) {
        atomicAdd(arrived, 1);
        const long long t0 = cycles();
        while (ld_acquire_gpu(arrived) < x.n_splits) {
          if (cycles() - t0 > kWaitLimitCycles) {
            atomicOr(a.status, VSD_DEV_TIMEOUT);
            break;
          }
        }
      }
      named_bar_sync(1, 256);
      // rows [r0, r1) of the valid rows; per row and float4 of the output:
      // running maximum over the splits and the rescaled sums of l and O,
      // eight splits' loads in flight (split order fixed: deterministic)
      {
        const int r0 = x.split * a.rows_valid / x.n_splits, r1 = (x.split + 1) * a.rows_valid / x.n_splits;
        constexpr int Q = HD / 4;  // float4 per row
        const size_t first = pair * a.max_splits;
        const float2* pml = reinterpret_cast<const float2*>(a.part_ml) + first * 128;
        const float4* pbase = reinterpret_cast<const float4*>(a.part_o + first * 128 * HD);
        for (int idx = threadIdx.x; idx < (r1 - r0) * Q; idx += 256) {
          const int row = r0 + idx / Q, d4 = idx % Q;
          const int hh = d4 / Q4, w4 = d4 % Q4;
          const float4* po_row = pbase + hh * NF4 + row * Q4 + w4;
          float mm = -INFINITY, ls = 0.0f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int s0 = 0; s0 < x.n_splits; s0 += 8) {
            float2 ml[8];
            float4 ov[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const bool in = s0 + j < x.n_splits;
              ml[j] = in ? __ldcg(pml + (s0 + j) * 128 + row) : make_float2(-INFINITY, 0.0f);
              ov[j] = in ? __ldcg(po_row + static_cast<size_t>(s0 + j) * 2 * NF4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float bm = mm;
#pragma unroll
            for (int j = 0; j < 8; ++j) bm = fmaxf(bm, ml[j].x);
            const float bu = bm == -INFINITY ? 0.0f : bm;
            const float sc = ex2(mm - bu);  // 0 while mm = -inf
            ls *= sc;
            acc.x *= sc;
            acc.y *= sc;
            acc.z *= sc;
            acc.w *= sc;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float w = ex2(ml[j].x - bu);
              ls += ml[j].y * w;
              acc.x += ov[j].x * w;
              acc.y += ov[j].y * w;
              acc.z += ov[j].z * w;
              acc.w += ov[j].w * w;
            }
            mm = bm;
          }
          const float inv = ls > 0.0f ? 1.0f / ls : 0.0f;
          const int d = hh * HH + w4 * 4;
          __half* o_dst = a.out + (static_cast<size_t>(x.b) * kRows + row / a.group) * (a.n_q * HD) +
                          (x.h * a.group + row % a.group) * HD + d;
          const float y[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
          uint32_t hw[2], lw[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            hw[e] = f32x2_to_f16x2(y[2 * e], y[2 * e + 1]);
            const __half2 h2 = *reinterpret_cast<const __half2*>(&hw[e]);
            lw[e] = f32x2_to_f16x2(y[2 * e] - __low2float(h2), y[2 * e + 1] - __high2float(h2));
          }
          *reinterpret_cast<uint2*>(o_dst) = make_uint2(hw[0], hw[1]);
          if (a.out_lo) *reinterpret_cast<uint2*>(o_dst + a.out_lo) = make_uint2(lw[0], lw[1]);
        }
      }
      // the last split to finish resets the pair's counters for the next launch
      // (every split has passed its wait by then)
      named_bar_sync(1, 256);
      if (threadIdx.x == 0 && atomicAdd(departed, 1) == x.n_splits - 1) {
        *arrived = 0;
        *departed = 0;
      }
      if (threadIdx.x == 0 && ic == 0) trace_point(a.trace, 7);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_end(a.trace, 11);
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace vsd
