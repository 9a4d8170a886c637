// persistent.cuh -- the decoder layers and the head of one verify step in a
// single persistent, cooperative launch (one CTA per SM).
//
// The step's 5 * layers + 1 dependent phases (per layer: QKV GEMM with
// RoPE, block attention, O GEMM + residual, gate/up GEMM + SiLU, down GEMM
// + residual; then the head with its fused argmax) run inside one kernel.
// A phase starts once every CTA has finished the one before it: each CTA
// adds one to a global counter per phase, and whoever needs the previous
// phase's outputs waits (bounded) for that counter to reach the grid size.
// Launch gaps and per-kernel start-up (barrier set-up, TMEM allocation)
// disappear, and so does most of the weight latency: weights do not depend
// on activations ("The Inference Stack Behind OCRia", section "Why decoding
// dominates latency": decode time is weight reads), so the producer warp
// streams the raw FP8 / NVFP4 tiles of later phases into their ring while
// the current phase computes, and the expansion warps turn them into f16
// MMA tiles before the phase's activations exist.  Context K/V pages of the
// attention phase are likewise fetched as soon as the QKV MMAs have released
// the shared-memory region they use.
//
// Warp roles (320 threads) are fixed for the whole launch and walk the same
// phase list:
//   warp 8  producer: weight tiles (1-D bulk copies of pre-packed tiles),
//           activation tiles and attention q / K / V (TMA);
//   warp 9  MMA issue (tcgen05, accumulators in TMEM);
//   warps 0-7  weight expansion, GEMM epilogues, attention softmax / merge.
// Shared memory: a region shared by the GEMM rings (expanded f16 weight tiles
// A, activation tiles B) and the attention buffers (q, K/V stages, P), a ring
// of raw weight tiles W, and a control block.  Ring positions and barrier
// phases are counted across phases, so no barrier is re-initialised.
//
// GEMMs whose output tiles cannot fill the GPU split k over a group of
// consecutive CTAs; each writes its partial tile to global memory (L2), the
// group meets on a per-item counter, and each member then sums a share of the
// tile's 16-column groups over all members in member order (deterministic)
// before applying the epilogue.
#pragma once

#include "attention.cuh"
#include "gemm.cuh"

namespace vsd {

constexpr int kMkThreads = 320;
constexpr int kMkKinds = 5;               // GEMM kinds: QKV, O, gate/up, down, head
constexpr int kMaxSplitItems = 1024;      // items of one split-k phase (per-item counters)
constexpr int kMkMaxTok = 144;            // token rows per activation tile (MMA N)

template <int HD>
struct MkCfg {
  static constexpr int NS = HD == 64 ? 2 : 1;   // attention K/V stages
  static constexpr int DA = 3, DB = 3, RD = 5;  // slots of the A, B and W rings
  static constexpr uint32_t A_SLOT = 16384u, B_SLOT = kMkMaxTok * 256u, W_SLOT = 8192u;
  static constexpr uint32_t QB = 128u * HD * 2u;  // one 128-row bf16 tile
  // attention buffers: q (hi, lo), K and V stages, P (hi, lo)
  static constexpr uint32_t ATT_Q = 0, ATT_KV = 2u * QB, ATT_P = ATT_KV + NS * 2u * QB, ATT_END = ATT_P + 65536u;
  // GEMM rings in the same region
  static constexpr uint32_t RING_A = 0, RING_B = DA * A_SLOT, RINGS_END = RING_B + DB * B_SLOT;
  // control block: barriers and flags (1 KB), per-warp argmax keys (2 KB),
  // running argmax keys (8 KB), sums of squares (4 KB), token scales (1 KB),
  // positions (1 KB), attention row statistics (4 KB), attention item offsets
  static constexpr uint32_t C_BAR = 0, C_WBEST = 1024, C_BEST = 3072, C_SQ = 11264, C_RS = 15360, C_POS = 16384,
                            C_XSTAT = 17408, C_ITEMS = 21504, CTRL_BYTES = C_ITEMS + 4u * (kMaxReqs + 2);
  static constexpr uint32_t MAX_DYN = 232448u - 1024u;
  static constexpr uint32_t RU = ATT_END > RINGS_END ? ATT_END : RINGS_END;
  // the W ring sits after the attention buffers when everything fits, else
  // inside them (then no W tile is fetched while an attention phase runs)
  static constexpr bool W_OVERLAP = RU + RD * W_SLOT + CTRL_BYTES > MAX_DYN;
  static constexpr uint32_t RING_W = W_OVERLAP ? RINGS_END : RU;
  static constexpr uint32_t CTRL = RING_W + RD * W_SLOT > ATT_END ? RING_W + RD * W_SLOT : ATT_END;
  static constexpr uint32_t SMEM = 1024u + CTRL + CTRL_BYTES;
  static_assert(SMEM <= 232448u, "persistent step kernel: shared memory");
  static_assert(RING_W >= RINGS_END, "W ring overlaps the GEMM rings");
};

// barrier slots of the control block
enum : int {
  MB_WFULL = 0, MB_WEMPTY = 5, MB_AFULL = 10, MB_AEMPTY = 13, MB_BFULL = 16, MB_BEMPTY = 19, MB_TFULL = 22,
  MB_TEMPTY = 24, MB_KFULL = 26, MB_KEMPTY = 28, MB_VFULL = 30, MB_VEMPTY = 32, MB_QFULL = 34, MB_QEMPTY = 35,
  MB_SFULL = 36, MB_SFREE = 38, MB_PFULL = 40, MB_OFULL = 41, MB_OFREE = 42, MB_ATTDONE = 43, MB_DRAIN = 44,
  MB_COUNT = 45
};
// named barriers: 1 epilogue set, 2-5 attention row pairs / argmax sets,
// 6 expansion by 256 threads, 7 by 128, 8 phase end, 9 attention (256)
constexpr int NB_EPI = 1, NB_X256 = 6, NB_X128 = 7, NB_END = 8, NB_ATT = 9;

struct MkLayerW {
  const uint8_t* w[4];  // tiles of QKV, O, gate/up, down
  const float* s[4];    // their per-row scales (FP8 / NVFP4)
};

struct MkParams {
  CUtensorMap tm_act[3];  // GEMM inputs (box n_tok x 64): u (QKV, gate/up, head), act_o (O), act_a (down)
  CUtensorMap tm_q, tm_kc, tm_vc, tm_kn, tm_vn;
  GemmArgs g[kMkKinds];   // per kind; weights, scales and per-layer outputs come from `layers`
  int wf[kMkKinds];
  int act_of[kMkKinds];
  AttnArgs at;            // layer set per phase
  const MkLayerW* layers;
  int n_layers;
  int* sync;              // [n_phases] phase counters, then the exit counter and the abort flag
  float* part;            // split-k partials [item][member][n_tok][128]
  int* item_cnt;          // [2][kMaxSplitItems] arrivals / departures per item
  int* status;
  long long wait_limit;   // SM cycles after which a wait gives up (VSD_DEV_TIMEOUT)
  Trace trace;            // launch id = trace.id + phase; trace.id + n_phases: kernel start / end
};

__device__ __forceinline__ int mk_phases(int n_layers) { return 5 * n_layers + 1; }
// GEMM kind of phase q (-1: attention)
__device__ __forceinline__ int mk_kind(int q, int n_layers) {
  if (q >= 5 * n_layers) return 4;
  const int s = q % 5;
  return s == 0 ? 0 : (s == 1 ? -1 : s - 1);
}

// Members of a split-k group are consecutive CTAs; CTAs past the last full
// group sit the phase out.
struct MkUnits {
  int cluster, rank, n_clusters, total, kb, ke;
  __device__ explicit MkUnits(const GemmArgs& a) {
    n_clusters = static_cast<int>(gridDim.x) / a.cs;
    cluster = static_cast<int>(blockIdx.x) / a.cs;
    rank = static_cast<int>(blockIdx.x) % a.cs;
    total = a.n_tiles * a.tok_tiles;
    if (cluster >= n_clusters) cluster = total;
    kb = rank * a.kps;
    ke = min(a.k_tiles, kb + a.kps);
  }
  __device__ int items() const {
    return (cluster < total && kb < ke) ? (total - cluster + n_clusters - 1) / n_clusters : 0;
  }
  __device__ int tiles() const { return items() * max(0, ke - kb); }
};

// (item, k tile) sequence of this CTA in one GEMM phase
struct MkIter {
  int item, total, stride, kt, kb, ke, tok_tiles;
  __device__ void init(const GemmArgs& a) {
    const MkUnits u(a);
    item = u.cluster;
    total = u.total;
    stride = u.n_clusters;
    kb = u.kb;
    ke = u.ke;
    kt = kb;
    tok_tiles = a.tok_tiles;
  }
  __device__ bool done() const { return item >= total || kb >= ke; }
  __device__ bool last_k() const { return kt + 1 == ke; }
  __device__ int tile() const { return item / tok_tiles; }
  __device__ int tok_tile() const { return item % tok_tiles; }
  __device__ void next() {
    if (++kt >= ke) {
      item += stride;
      kt = kb;
    }
  }
};

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Arrival on an mbarrier without a transaction (count 1) after expect_tx.
__device__ __forceinline__ void mbar_expect_tx_only(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

template <int HD>
__global__ void __launch_bounds__(kMkThreads, 1) step_kernel(const __grid_constant__ MkParams p) {
  using C = MkCfg<HD>;
  constexpr int NS = C::NS, DA = C::DA, DB = C::DB, RD = C::RD;
  constexpr int NA = HD / 64;  // 64-wide swizzle atoms along head_dim
  constexpr int HH = HD / 2;   // output columns per softmax thread
  constexpr uint32_t QB = C::QB, KVB = C::QB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ctrl = smem + C::CTRL;
  uint64_t* bar = reinterpret_cast<uint64_t*>(ctrl + C::C_BAR);
  int* misc = reinterpret_cast<int*>(ctrl + 512);
  uint32_t* tmem_p = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = misc + 1;
  volatile int* n_items_s = misc + 2;
  volatile int* cps_s = misc + 3;
  volatile int* sum_s = misc + 4;
  volatile int* flag_s = misc + 5;  // broadcast of a dependency wait's result to the epilogue threads
  unsigned long long* wbest = reinterpret_cast<unsigned long long*>(ctrl + C::C_WBEST);
  unsigned long long* best = reinterpret_cast<unsigned long long*>(ctrl + C::C_BEST);
  float* sq_red = reinterpret_cast<float*>(ctrl + C::C_SQ);
  float* rs = reinterpret_cast<float*>(ctrl + C::C_RS);
  int* pos_s = reinterpret_cast<int*>(ctrl + C::C_POS);
  float* xstat = reinterpret_cast<float*>(ctrl + C::C_XSTAT);
  int* item_off = reinterpret_cast<int*>(ctrl + C::C_ITEMS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = p.n_layers;
  const int n_phases = mk_phases(L);
  const int G = static_cast<int>(gridDim.x);
  int* const sync = p.sync;
  volatile int* const g_abort = p.sync + n_phases + 1;
  const AttnArgs& at = p.at;

  Trace tk = p.trace;
  tk.id += n_phases;
  if (threadIdx.x == 0) trace_start(tk);
  auto phase_trace = [&](int q) {
    Trace t = p.trace;
    t.id += q;
    return t;
  };

  // attention: lengths first, so that their loads overlap the set-up
  auto chunks_of = [&](int b) { return (valid_len(at, b) + 127) / 128 + 1; };
  int mine = 0;
  for (int b = threadIdx.x; b < at.batch; b += blockDim.x) mine += chunks_of(b);

  if (threadIdx.x == 0) {
    for (int i = 0; i < RD; ++i) {
      mbar_init(&bar[MB_WFULL + i], 1);
      mbar_init(&bar[MB_WEMPTY + i], 1);
    }
    for (int i = 0; i < DA; ++i) {
      mbar_init(&bar[MB_AFULL + i], 1);
      mbar_init(&bar[MB_AEMPTY + i], 1);
    }
    for (int i = 0; i < DB; ++i) {
      mbar_init(&bar[MB_BFULL + i], 1);
      mbar_init(&bar[MB_BEMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[MB_TFULL + i], 1);
      mbar_init(&bar[MB_TEMPTY + i], 1);
      mbar_init(&bar[MB_SFULL + i], 1);
      mbar_init(&bar[MB_SFREE + i], 256);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar[MB_KFULL + s], 1);
      mbar_init(&bar[MB_KEMPTY + s], 1);
      mbar_init(&bar[MB_VFULL + s], 1);
      mbar_init(&bar[MB_VEMPTY + s], 1);
    }
    mbar_init(&bar[MB_QFULL], 1);
    mbar_init(&bar[MB_QEMPTY], 1);
    mbar_init(&bar[MB_PFULL], 256);
    mbar_init(&bar[MB_OFULL], 1);
    mbar_init(&bar[MB_OFREE], 256);
    mbar_init(&bar[MB_ATTDONE], 1);
    mbar_init(&bar[MB_DRAIN], 1);
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
  // Attention split plan (the same in every CTA and every layer): the
  // smallest number of 128-key chunks per split, at least the host's, whose
  // items fit in one round of the grid; items request-major, then KV head,
  // then split.
  {
    if (mine) atomicAdd(const_cast<int*>(sum_s), mine);
    __syncthreads();
    const int total_chunks = *sum_s * at.n_kv;
    int c = max(at.chunks_per_split, (total_chunks + G - 1) / G);
    for (;; ++c) {  // ends: at the longest request's chunk count every request is one split
      __syncthreads();
      if (threadIdx.x == 0) *sum_s = 0;
      __syncthreads();
      int items = 0;
      for (int b = threadIdx.x; b < at.batch; b += blockDim.x) items += (chunks_of(b) + c - 1) / c;
      if (items) atomicAdd(const_cast<int*>(sum_s), items);
      __syncthreads();
      if (*sum_s * at.n_kv <= G || *sum_s == at.batch) break;
    }
    if (warp == 0) {
      int base = 0;
      for (int b0 = 0; b0 < at.batch; b0 += 32) {
        const int b = b0 + lane;
        const int cnt = b < at.batch ? at.n_kv * ((chunks_of(b) + c - 1) / c) : 0;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        if (b < at.batch) item_off[b] = base + incl - cnt;
        base += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (lane == 0) {
        item_off[at.batch] = base;
        *n_items_s = base;
        *cps_s = c;
      }
    }
    __syncthreads();
  }
  const uint32_t tmem = *tmem_p;
  const int att_total = *n_items_s;
  const int cps = *cps_s;
  auto splits_of = [&](int b) { return (chunks_of(b) + cps - 1) / cps; };
  struct Item {
    int b, h, split, n_splits, L, n_ctx, c_begin, n;
  };
  auto decode = [&](int it) {
    Item x;
    int lo = 0, hi = at.batch - 1;  // last request whose first item is <= it
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
    x.L = valid_len(at, x.b);
    x.n_ctx = (x.L + 127) >> 7;
    x.c_begin = x.split * cps;
    x.n = min(x.n_ctx + 1, x.c_begin + cps) - x.c_begin;
    return x;
  };
  // chunks of this CTA's attention items in one layer (the same every layer)
  int att_chunks = 0, att_items = 0;
  for (int it = blockIdx.x; it < att_total; it += G) {
    att_chunks += decode(it).n;
    ++att_items;
  }

  // bounded waits -------------------------------------------------------------
  // raise the CTA's and the grid's abort flags and record the timeout
  auto give_up = [&](bool timed_out) {
    if (timed_out && !*abort_flag) atomicOr(p.status, VSD_DEV_TIMEOUT);
    *abort_flag = 1;
    *g_abort = 1;
  };
  auto aborted = [&]() { return *abort_flag != 0 || *g_abort != 0; };
  // phase q complete in every CTA (q < 0: nothing to wait for)
  auto phase_done = [&](int q) { return q < 0 || ld_acquire_gpu(sync + q) >= G; };
  auto wait_phase = [&](int q) -> bool {
    if (phase_done(q)) return *abort_flag == 0;
    const long long t0 = cycles();
    while (!phase_done(q)) {
      if (aborted()) {
        *abort_flag = 1;
        return false;
      }
      if (cycles() - t0 > p.wait_limit) {
        give_up(true);
        return false;
      }
    }
    return *abort_flag == 0;
  };
  // position n of a ring of depth D: its slot, and the parity of its fill
  auto slot_of = [](int n, int D) { return n % D; };
  auto par_of = [](int n, int D) { return static_cast<uint32_t>((n / D) & 1); };
  // an mbarrier wait that also gives up when another CTA has aborted; after
  // the barrier completes it still reports an abort of this CTA, so that the
  // threads of a group that meet at a named barrier next take one decision
  auto mwait = [&](uint64_t* b, uint32_t parity) -> bool {
    if (mbar_test_wait(b, parity)) return *abort_flag == 0;
    const long long t0 = cycles();
    while (true) {
#pragma unroll 1
      for (int i = 0; i < 32; ++i)
        if (mbar_test_wait(b, parity)) return *abort_flag == 0;
      if (aborted()) {
        *abort_flag = 1;
        return false;
      }
      if (cycles() - t0 > p.wait_limit) {
        give_up(true);
        return false;
      }
    }
  };

  // ring positions, counted across phases by every role alike
  int w_pos = 0, a_pos = 0, b_pos = 0, acc_pos = 0;
  int att_g = 0, att_ic = 0, att_seen = 0;

  if (warp == 8) {
    // ====================================================================== producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    // raw weight stream: phase, position in it, tiles issued (lane 0 only)
    int wq = -1, wn = 0;
    MkIter wit;
    wit.item = wit.total = 0;
    wit.kb = wit.ke = 0;
    auto w_advance = [&]() {
      ++wq;
      if (wq < n_phases) {
        const int k = mk_kind(wq, L);
        if (k >= 0) wit.init(p.g[k]);
      }
    };
    w_advance();
    // attention phases finished by this CTA's compute warps
    auto poll_att = [&]() {
      while (mbar_test_wait(&bar[MB_ATTDONE], static_cast<uint32_t>(att_seen & 1))) ++att_seen;
      return att_seen;
    };
    // issue the next raw weight tile if its slot is free; false if nothing was issued
    auto try_w = [&]() -> bool {
      while (wq < n_phases) {
        const int k = mk_kind(wq, L);
        if (k < 0) {
          if (C::W_OVERLAP && poll_att() <= wq / 5) return false;  // its buffers hold the W ring
          w_advance();
          continue;
        }
        if (p.wf[k] == W_BF16 || wit.done()) {
          w_advance();
          continue;
        }
        break;
      }
      if (wq >= n_phases) return false;
      const int s = slot_of(wn, RD);
      if (wn >= RD && !mbar_test_wait(&bar[MB_WEMPTY + s], par_of(wn - RD, RD))) return false;
      const int k = mk_kind(wq, L);
      const GemmArgs& a = p.g[k];
      const uint32_t bytes = p.wf[k] == W_FP8 ? kFp8TileBytes : kFp4TileBytes;
      const uint8_t* base = k == 4 ? a.w_tiles : p.layers[wq / 5].w[k];
      const uint8_t* src = base + (static_cast<size_t>(wit.tile()) * a.k_tiles + wit.kt) * bytes;
      mbar_expect_tx(&bar[MB_WFULL + s], bytes);
      bulk_load(smem + C::RING_W + s * C::W_SLOT, src, bytes, &bar[MB_WFULL + s], pol_w);
      ++wn;
      wit.next();
      return true;
    };
    // producer-side wait (the whole warp calls it): lane 0 polls the barrier
    // and keeps the weight stream going meanwhile; every lane gets its verdict
    auto pwait = [&](uint64_t* b, uint32_t parity) -> bool {
      int okw = 1;
      if (lane == 0) {
        const long long t0 = cycles();
        while (!mbar_test_wait(b, parity)) {
          if (try_w()) continue;
          if (aborted()) {
            *abort_flag = 1;
            okw = 0;
            break;
          }
          if (cycles() - t0 > p.wait_limit) {
            give_up(true);
            okw = 0;
            break;
          }
        }
      }
      return __shfl_sync(0xFFFFFFFFu, okw, 0) != 0;
    };
    auto pwait_phase = [&](int q) -> bool {  // lane 0
      const long long t0 = cycles();
      while (!phase_done(q)) {
        if (try_w()) continue;
        if (aborted()) {
          *abort_flag = 1;
          return false;
        }
        if (cycles() - t0 > p.wait_limit) {
          give_up(true);
          return false;
        }
      }
      fence_proxy_async_global();  // generic writes of the other CTAs -> this CTA's TMA reads
      return true;
    };
    bool ok = true;
    for (int q = 0; ok && q < n_phases; ++q) {
      const int kind = mk_kind(q, L);
      const Trace tq = phase_trace(q);
      if (kind >= 0) {
        // ---------------------------------------------------------------- GEMM phase
        const GemmArgs& a = p.g[kind];
        const bool bf16 = p.wf[kind] == W_BF16;
        const int n_tiles_cta = MkUnits(a).tiles();
        if (lane == 0) {
          const CUtensorMap* tm = &p.tm_act[p.act_of[kind]];
          const bool act_lo = a.act_lo_rows > 0;
          const uint32_t b_bytes = static_cast<uint32_t>(a.n_tok) * 128u * (act_lo ? 2u : 1u);
          MkIter ib, ia;
          ib.init(a);
          ia.init(a);
          // 16-bit weights go straight into the A ring, which shares its space
          // with the attention buffers: after an attention phase, only once
          // this CTA's attention work is over
          const int att_before = (q % 5 == 2 && q < 5 * L) ? q / 5 : -1;
          bool dep = q == 0, region = !bf16 || att_before < 0;
          int an = a_pos, bn = b_pos;
          long long t_last = cycles();
          while (!ib.done() || (bf16 && !ia.done())) {
            bool progress = false;
            if (bf16 && !ia.done()) {
              if (!region) region = poll_att() > att_before;
              const int s = slot_of(an, DA);
              if (region && (an < DA || mbar_test_wait(&bar[MB_AEMPTY + s], par_of(an - DA, DA)))) {
                const uint8_t* base = kind == 4 ? a.w_tiles : p.layers[q / 5].w[kind];
                const uint8_t* src = base + (static_cast<size_t>(ia.tile()) * a.k_tiles + ia.kt) * 16384u;
                mbar_expect_tx(&bar[MB_AFULL + s], 16384u);
                bulk_load(smem + C::RING_A + s * C::A_SLOT, src, 16384u, &bar[MB_AFULL + s], pol_w);
                ++an;
                ia.next();
                progress = true;
              }
            }
            if (!dep && phase_done(q - 1)) {
              dep = true;
              fence_proxy_async_global();
              trace_point(tq, 1);
            }
            if (dep && !ib.done()) {
              const int s = slot_of(bn, DB);
              if (bn < DB || mbar_test_wait(&bar[MB_BEMPTY + s], par_of(bn - DB, DB))) {
                uint8_t* dst = smem + C::RING_B + s * C::B_SLOT;
                mbar_expect_tx(&bar[MB_BFULL + s], b_bytes);
                const int r0 = ib.tok_tile() * a.n_tok;
                tma_load_2d_hint(dst, tm, &bar[MB_BFULL + s], ib.kt * kTileK, r0, pol_a);
                if (act_lo)
                  tma_load_2d_hint(dst + a.n_tok * 128, tm, &bar[MB_BFULL + s], ib.kt * kTileK, a.act_lo_rows + r0,
                                   pol_a);
                ++bn;
                ib.next();
                progress = true;
                if (ib.done()) trace_point(tq, 11);
              }
            }
            if (try_w()) progress = true;
            if (progress) {
              t_last = cycles();
              continue;
            }
            if (aborted()) {
              *abort_flag = 1;
              ok = false;
              break;
            }
            if (cycles() - t_last > p.wait_limit) {
              give_up(true);
              ok = false;
              break;
            }
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        a_pos += n_tiles_cta;
        b_pos += n_tiles_cta;
        if (!bf16) w_pos += n_tiles_cta;
      } else {
        // ---------------------------------------------------------------- attention phase
        const int layer = q / 5;
        // the attention buffers reuse the GEMM rings' space (and, W_OVERLAP,
        // the W ring's): wait until the MMAs have released the last A and B
        // slots and the expansion the last W slot
        ok = (a_pos == 0 || pwait(&bar[MB_AEMPTY + slot_of(a_pos - 1, DA)], par_of(a_pos - 1, DA))) &&
             (b_pos == 0 || pwait(&bar[MB_BEMPTY + slot_of(b_pos - 1, DB)], par_of(b_pos - 1, DB)));
        // (wn: lane 0's count of W tiles issued)
        const int wn_all = __shfl_sync(0xFFFFFFFFu, wn, 0);
        if (ok && C::W_OVERLAP && wn_all > 0)
          ok = pwait(&bar[MB_WEMPTY + slot_of(wn_all - 1, RD)], par_of(wn_all - 1, RD));
        if (!ok) break;
        const uint64_t pol = policy_evict_first();
        // chunk i of item x, global chunk number g: K then V, each once its slot is free
        auto issue = [&](const Item& x, int i, int g, int page_pre) -> bool {
          const int st = g % NS;
          uint8_t* ks = smem + C::ATT_KV + st * KVB;
          uint8_t* vs = smem + C::ATT_KV + (NS + st) * KVB;
          const int c = x.c_begin + i;
          const bool ctx = c < x.n_ctx;
          int row0 = 0;
          if (ctx && lane < 8) {  // lane p: page p of the chunk
            const int pi = min(c * 8 + lane, at.pages_per_req - 1);
            int page = page_pre >= 0 ? page_pre : at.page_table[x.b * at.pages_per_req + pi];
            if (page < 0 || page >= at.num_pages) {
              atomicOr(at.status, VSD_DEV_BAD_PAGE);
              page = 0;
            }
            row0 = ((layer * at.num_pages + page) * at.n_kv + x.h) * kPage;
          } else if (!ctx) {
            row0 = ((layer * at.batch_cap + x.b) * at.n_kv + x.h) * 32;
          }
          const uint32_t bytes = (ctx ? 128u : 32u) * HD * 2u;
          for (int part = 0; part < 2; ++part) {  // 0: K, 1: V
            uint64_t* full = part ? &bar[MB_VFULL + st] : &bar[MB_KFULL + st];
            uint64_t* empty = part ? &bar[MB_VEMPTY + st] : &bar[MB_KEMPTY + st];
            uint8_t* dst = part ? vs : ks;
            if (g >= NS && !pwait(empty, static_cast<uint32_t>(((g / NS) - 1) & 1))) return false;
            if (lane == 0) mbar_expect_tx(full, bytes);
            __syncwarp();
            if (ctx && lane < 8) {
#pragma unroll
              for (int t = 0; t < NA; ++t)
                tma_load_2d_hint(dst + t * 16384 + lane * 2048, part ? &p.tm_vc : &p.tm_kc, full, t * 64, row0, pol);
            } else if (!ctx && lane == 0) {
              for (int t = 0; t < NA; ++t)
                tma_load_2d(dst + t * 16384, part ? &p.tm_vn : &p.tm_kn, full, t * 64, row0);
            }
            __syncwarp();
          }
          return true;
        };
        // context chunks do not depend on this step: the first item's first
        // chunks go out before the QKV phase is complete
        int npre = 0;
        if (static_cast<int>(blockIdx.x) < att_total) {
          const Item x = decode(blockIdx.x);
          while (npre < min(x.n, NS) && x.c_begin + npre < x.n_ctx) ++npre;
          for (int i = 0; ok && i < npre; ++i) ok = issue(x, i, att_g + i, -1);
        }
        if (!ok) break;
        if (lane == 0) {
          ok = pwait_phase(q - 1);  // q tiles and the block's K/V come from the QKV phase
          if (ok) trace_point(tq, 1);
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        int g = att_g, ic = att_ic;
        for (int it = blockIdx.x; ok && it < att_total; it += G, ++ic) {
          const Item x = decode(it);
          if (ic > att_ic && !pwait(&bar[MB_QEMPTY], static_cast<uint32_t>((ic - 1) & 1))) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const int q_row = (x.b * at.n_kv + x.h) * 128;
            mbar_expect_tx(&bar[MB_QFULL], at.q_lo_rows ? 2 * QB : QB);
            for (int t = 0; t < NA; ++t) {
              tma_load_2d(smem + C::ATT_Q + t * 16384, &p.tm_q, &bar[MB_QFULL], t * 64, q_row);
              if (at.q_lo_rows)
                tma_load_2d(smem + C::ATT_Q + QB + t * 16384, &p.tm_q, &bar[MB_QFULL], t * 64, at.q_lo_rows + q_row);
            }
          }
          __syncwarp();
          for (int i = 0; i < x.n; ++i, ++g) {
            if (ic == att_ic && i < npre) continue;  // issued before the dependency wait
            if (!issue(x, i, g, -1)) {
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
        att_g += att_chunks;
        att_ic += att_items;
      }
    }
    if (!ok) {
      // let the copies in flight land before the CTA exits
      volatile int never = 0;
      if (lane == 0) {
        const long long t0 = cycles();
        while (cycles() - t0 < 200000) {
        }
        (void)never;
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ====================================================================== MMA issue
    bool ok = true;
    for (int q = 0; ok && q < n_phases; ++q) {
      const int kind = mk_kind(q, L);
      const Trace tq = phase_trace(q);
      if (kind >= 0) {
        const GemmArgs& a = p.g[kind];
        const int n_tiles_cta = MkUnits(a).tiles();
        const int n_items_cta = MkUnits(a).items();
        if (lane == 0) {
          const bool act_lo = a.act_lo_rows > 0;
          const bool stacked = act_lo && 2 * a.n_tok <= 256;
          const int acc_w = stacked ? 2 * a.n_tok : a.n_tok;
          const uint32_t idesc = idesc_f16(128, acc_w, false, false, false);
          const uint64_t a_desc0 = sw128_desc(smem_u32(smem + C::RING_A), 16, 1024);
          const uint64_t b_desc0 = sw128_desc(smem_u32(smem + C::RING_B), 16, 1024);
          const uint32_t lo_step = static_cast<uint32_t>(a.n_tok) * 8u;
          MkIter it;
          it.init(a);
          int an = a_pos, bn = b_pos, acc = acc_pos;
          bool first = true;
          while (ok && !it.done()) {
            const int ab = acc & 1;
            if (acc >= 2 && !mwait(&bar[MB_TEMPTY + ab], static_cast<uint32_t>(((acc >> 1) - 1) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem + static_cast<uint32_t>(ab * 256);
            uint32_t accum = 0;
            bool last = false;
            do {
              const int sa = slot_of(an, DA), sb = slot_of(bn, DB);
              if (!mwait(&bar[MB_AFULL + sa], par_of(an, DA)) || !mwait(&bar[MB_BFULL + sb], par_of(bn, DB))) {
                ok = false;
                break;
              }
              if (first) {
                trace_point(tq, 2);
                first = false;
              }
              tc_fence_after();
              const uint64_t ad = a_desc0 + static_cast<uint64_t>(sa) * (C::A_SLOT >> 4);
              const uint64_t bd = b_desc0 + static_cast<uint64_t>(sb) * (C::B_SLOT >> 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                umma_f16(d, ad + 2 * kk, bd + 2 * kk, idesc, accum | kk);
                if (act_lo && !stacked) umma_f16(d, ad + 2 * kk, bd + lo_step + 2 * kk, idesc, 1u);
              }
              accum = 1;
              umma_commit(&bar[MB_AEMPTY + sa]);
              umma_commit(&bar[MB_BEMPTY + sb]);
              ++an;
              ++bn;
              last = it.last_k();
              it.next();
            } while (!last);
            if (!ok) break;
            umma_commit(&bar[MB_TFULL + ab]);
            trace_point(tq, 10);
            ++acc;
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        a_pos += n_tiles_cta;
        b_pos += n_tiles_cta;
        acc_pos += n_items_cta;
      } else {
        if (lane == 0) {
          const uint32_t id_s128 = idesc_f16(128, 128, true, true, false);
          const uint32_t id_s32 = idesc_f16(128, 32, true, true, false);
          const uint32_t id_pv = idesc_f16(128, HD, true, true, true);
          const uint32_t qa = smem_u32(smem + C::ATT_Q), pa = smem_u32(smem + C::ATT_P);
          int g0 = att_g, ic = att_ic;
          bool first = true;
          for (int it = blockIdx.x; ok && it < att_total; it += G, ++ic) {
            const Item x = decode(it);
            if (!mwait(&bar[MB_QFULL], static_cast<uint32_t>(ic & 1))) {
              ok = false;
              break;
            }
            auto issue_s = [&](int i) -> bool {
              const int g = g0 + i, st = g % NS;
              if (!mwait(&bar[MB_KFULL + st], static_cast<uint32_t>((g / NS) & 1))) return false;
              if (g >= 2 && !mwait(&bar[MB_SFREE + (g & 1)], static_cast<uint32_t>(((g >> 1) - 1) & 1)))
                return false;
              tc_fence_after();
              if (first) {
                trace_point(tq, 2);
                first = false;
              }
              const uint32_t ka = smem_u32(smem + C::ATT_KV + st * KVB);
              const bool blk = (x.c_begin + i) >= x.n_ctx;
              const uint32_t d = tmem + (g & 1) * 128;
              // The lo product of each k step goes first and the hi product
              // follows.  Issued hi first (the hi tile sits at the start of
              // the region the GEMM rings share), the scores of up to a few
              // dozen q rows came out wrong on sm_103a while each product
              // alone was exact; lo first is exact in every measured case.
#pragma unroll
              for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                const uint64_t kd = sw128_desc(ka + off, 16, 1024);
                if (at.q_lo_rows) {
                  umma_f16(d, sw128_desc(qa + QB + off, 16, 1024), kd, blk ? id_s32 : id_s128, kk > 0 ? 1u : 0u);
                  umma_f16(d, sw128_desc(qa + off, 16, 1024), kd, blk ? id_s32 : id_s128, 1u);
                } else {
                  umma_f16(d, sw128_desc(qa + off, 16, 1024), kd, blk ? id_s32 : id_s128, kk > 0 ? 1u : 0u);
                }
              }
              umma_commit(&bar[MB_SFULL + (g & 1)]);
              umma_commit(&bar[MB_KEMPTY + st]);
              if (i + 1 == x.n) umma_commit(&bar[MB_QEMPTY]);  // last use of this item's q tile
              return true;
            };
            ok = issue_s(0);
            for (int i = 0; ok && i < x.n; ++i) {
              const int g = g0 + i;
              if (i + 1 < x.n && !issue_s(i + 1)) {
                ok = false;
                break;
              }
              if (!mwait(&bar[MB_PFULL], static_cast<uint32_t>(g & 1)) ||
                  (g >= 1 && !mwait(&bar[MB_OFREE], static_cast<uint32_t>((g - 1) & 1)))) {
                ok = false;
                break;
              }
              const int st = g % NS;
              if (!mwait(&bar[MB_VFULL + st], static_cast<uint32_t>((g / NS) & 1))) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t va = smem_u32(smem + C::ATT_KV + (NS + st) * KVB);
              const bool blk = (x.c_begin + i) >= x.n_ctx;
              const int ksteps = blk ? 2 : 8;
              for (int kk = 0; kk < ksteps; ++kk) {
                const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
                const uint64_t vd = sw128_desc(va + kk * 2048, 16384, 1024);
                umma_f16(tmem + 256, sw128_desc(pa + aoff, 16, 1024), vd, id_pv, kk > 0 ? 1u : 0u);
                umma_f16(tmem + 256, sw128_desc(pa + 32768 + aoff, 16, 1024), vd, id_pv, 1u);
              }
              umma_commit(&bar[MB_OFULL]);
              umma_commit(&bar[MB_VEMPTY + st]);
            }
            g0 += x.n;
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        att_g += att_chunks;
        att_ic += att_items;
      }
    }
    if (lane == 0) {
      // every MMA issued by this thread completes before the TMEM is freed
      umma_commit(&bar[MB_DRAIN]);
      volatile int never = 0;
      mbar_wait(&bar[MB_DRAIN], 0, &never, nullptr);
    }
    __syncwarp();
  } else {
    // ====================================================================== warps 0-7
    const int t = threadIdx.x;  // 0..255
    bool ok = true;
    for (int q = 0; q < n_phases; ++q) {
      const int kind = mk_kind(q, L);
      const Trace tq = phase_trace(q);
      if (t == 0) trace_point(tq, 3);
      if (ok && kind >= 0) {
        // ---------------------------------------------------------------- GEMM phase
        const GemmArgs& a = p.g[kind];
        const int wf = p.wf[kind];
        const bool raw = wf != W_BF16;
        const MkUnits u(a);
        const int items = u.items();
        const int n_tiles_cta = u.tiles();
        const int layer = kind == 4 ? 0 : q / 5;
        const float* row_scale = kind == 4 ? a.row_scale : p.layers[layer].s[kind];
        // one item: all eight warps expand, then all eight run the epilogue;
        // more items: warps 0-3 expand while warps 4-7 run the epilogues
        const bool wide = raw && items <= 1;
        const bool ep8 = !raw || wide;
        const int half = warp < 4 ? 1 : 0;
        if (raw && (wide || half)) {
          const int NT = wide ? 256 : 128;
          const int nb = wide ? NB_X256 : NB_X128;
          MkIter it;
          it.init(a);
          for (int i = 0; !it.done(); it.next(), ++i) {
            const int wn = w_pos + i, an = a_pos + i;
            const int sw = slot_of(wn, RD), sa = slot_of(an, DA);
            if (!mwait(&bar[MB_WFULL + sw], par_of(wn, RD)) ||
                (an >= DA && !mwait(&bar[MB_AEMPTY + sa], par_of(an - DA, DA)))) {
              ok = false;
              break;
            }
            uint8_t* at_ = smem + C::RING_A + sa * C::A_SLOT;
            const uint8_t* raw_ = smem + C::RING_W + sw * C::W_SLOT;
            if (wf == W_FP8) {
              expand_weights<W_FP8, 256>(at_, raw_, t);
              if (NT == 128) expand_weights<W_FP8, 256>(at_, raw_, t + 128);
            } else {
              expand_weights<W_NVFP4, 256>(at_, raw_, t);
              if (NT == 128) expand_weights<W_NVFP4, 256>(at_, raw_, t + 128);
            }
            fence_proxy_async();
            named_bar_sync(nb, NT);
            if ((t & (NT - 1)) == 0) {
              mbar_arrive(&bar[MB_AFULL + sa]);
              mbar_arrive(&bar[MB_WEMPTY + sw]);
            }
          }
          if (t == 0) trace_point(tq, 9);
        }
        if (ok && (!half || ep8)) {
          // -------------------------------------------------------------- epilogue
          const int we = warp & 3;                // TMEM lane quarter
          const int row = we * 32 + lane;
          const int et = t & 127;
          const int n_sets = ep8 ? 2 : 1;
          const int ep_n = 128 * n_sets;
          const int et2 = ep8 ? t : et;           // thread of the epilogue
          const int set = ep8 ? half : 0;         // which alternate column groups
          const int cs = a.cs, rank = u.rank;
          const int groups = a.n_tok / 16;
          // inputs of this phase (residual rows, sums of squares, lengths) come from earlier phases
          if (items > 0) {
            if (et2 == 0) *flag_s = wait_phase(q - 1) ? 1 : 0;
            named_bar_sync(NB_EPI, ep_n);
            ok = *flag_s != 0;
          }
          const bool keep_best = a.tok_tiles * a.n_tok <= kBestCap;
          if (kind == 4 && a.keys != nullptr)
            for (int c = et2; c < kBestCap; c += ep_n) best[c] = 0ull;
          int acc = acc_pos;
          for (int item = u.cluster; ok && items > 0 && item < u.total; item += u.n_clusters, ++acc) {
            const int ab = acc & 1;
            const int tile = item / a.tok_tiles, tt = item % a.tok_tiles;
            const int prow_s = tile * kTileN + row;
            const float scale = (raw && prow_s < a.n_rows) ? row_scale[prow_s] : 1.0f;
            // per-token scale of the normalised input rows (and positions / draft tokens)
            for (int c = et2; c < a.n_tok; c += ep_n) {
              float r = 1.0f;
              const int tok = tt * a.n_tok + c;
              if (a.ssq_in && tok < a.m_tokens) {
                float ss = 0.0f;
#pragma unroll 8
                for (int k = 0; k < a.n_ssq; ++k) ss += __ldcg(a.ssq_in + static_cast<size_t>(k) * a.ssq_ld + tok);
                r = 1.0f / sqrtf(ss * a.inv_hidden + a.eps);
              }
              rs[c] = r;
              if (kind == 0) {
                pos_s[c] = tok < a.m_tokens ? a.ctx_len[tok / kRows] + tok % kRows : 0;
              } else if (kind == 4 && a.drafts != nullptr) {
                const int j = tok % kRows;
                pos_s[c] = (tok < a.m_tokens && j < kBlock) ? a.drafts[(tok / kRows) * kBlock + j] : -1;
              }
            }
            named_bar_sync(NB_EPI, ep_n);
            if (et2 == 0 && acc == acc_pos) trace_point(tq, 4);
            if (!mwait(&bar[MB_TFULL + ab], static_cast<uint32_t>((acc >> 1) & 1))) {
              ok = false;
              break;
            }
            if (et2 == 0 && acc == acc_pos) trace_point(tq, 5);
            tc_fence_after();
            const bool act_lo = a.act_lo_rows > 0;
            const bool stacked = act_lo && 2 * a.n_tok <= 256;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(we * 32) << 16) + static_cast<uint32_t>(ab * 256);
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
            float* part_item = p.part + static_cast<size_t>(item) * cs * a.n_tok * 128;
            if (cs > 1) {
              // partial sums of this member's k range -> global [member][column][row]
              float* mine_p = part_item + static_cast<size_t>(rank) * a.n_tok * 128;
              for (int c0 = set * 16; c0 < a.n_tok; c0 += 16 * n_sets) {
                load_cols(c0, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) __stcg(mine_p + (c0 + i) * 128 + row, v[i]);
              }
              tc_fence_before();
              __threadfence();
              named_bar_sync(NB_EPI, ep_n);
              if (et2 == 0) {
                trace_point(tq, 6);
                mbar_arrive(&bar[MB_TEMPTY + ab]);
                int* arrived = p.item_cnt + item;
                red_release_add(arrived, 1);
                const long long t0 = cycles();
                int okw = 1;
                while (ld_acquire_gpu(arrived) < cs) {
                  if (aborted()) {
                    okw = 0;
                    break;
                  }
                  if (cycles() - t0 > p.wait_limit) {
                    give_up(true);
                    okw = 0;
                    break;
                  }
                }
                *flag_s = okw;
                trace_point(tq, 7);
              }
              named_bar_sync(NB_EPI, ep_n);
              if (!*flag_s) {
                ok = false;
                break;
              }
            }
            // column groups of this set: every n_sets-th of this member's
            // (every group when k is not split, every cs-th otherwise)
            int gi = 0;
            for (int gidx = rank + cs * set; gidx < groups; gidx += cs * n_sets, ++gi) {
              const int c0 = gidx * 16;
              if (cs == 1) {
                load_cols(c0, v);
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = 0.0f;
                for (int m = 0; m < cs; ++m) {  // member order: deterministic
                  const float* src = part_item + static_cast<size_t>(m) * a.n_tok * 128 + c0 * 128 + row;
                  float x[16];
#pragma unroll
                  for (int i = 0; i < 16; ++i) x[i] = __ldcg(src + i * 128);
#pragma unroll
                  for (int i = 0; i < 16; ++i) v[i] += x[i];
                }
              }
              unsigned long long* wb = wbest + set * 128 + (gi & 1) * 64;
              switch (kind) {
                case 0:
                  epilogue_cols<EPI_QKV, W_FP8>(a, tile, tt, row, c0, v, scale, rs, pos_s, wb, sq_red, we, lane,
                                                layer);
                  break;
                case 1:
                case 3:
                  epilogue_cols<EPI_RESID, W_FP8>(a, tile, tt, row, c0, v, scale, rs, pos_s, wb, sq_red, we, lane,
                                                  layer);
                  break;
                case 2:
                  epilogue_cols<EPI_SILU, W_FP8>(a, tile, tt, row, c0, v, scale, rs, pos_s, wb, sq_red, we, lane,
                                                 layer);
                  break;
                default:
                  if (a.keys != nullptr)
                    epilogue_cols<EPI_ARGMAX, W_FP8>(a, tile, tt, row, c0, v, scale, rs, pos_s, wb, sq_red, we,
                                                     lane, layer);
                  else
                    epilogue_cols<EPI_SAMPLE, W_FP8>(a, tile, tt, row, c0, v, scale, rs, pos_s, wb, sq_red, we,
                                                     lane, layer);
                  break;
              }
              if (kind == 4) {
                named_bar_sync(4 + set, 128);  // this set's four warps only
                if (et < 16) {
                  const int col = tt * a.n_tok + c0 + et;
                  if (a.keys != nullptr) {
                    unsigned long long k = wb[et];
#pragma unroll
                    for (int w = 1; w < 4; ++w) k = wb[w * 16 + et] > k ? wb[w * 16 + et] : k;
                    if (keep_best) {
                      if (k > best[col]) best[col] = k;
                    } else if (col < a.m_tokens && k) {
                      atomicMax(a.keys + col, k);
                    }
                  } else {  // the tile's (max, sum), warps in fixed order (deterministic)
                    const unsigned long long r =
                        ms_merge(ms_merge(ms_merge(wb[et], wb[16 + et]), wb[32 + et]), wb[48 + et]);
                    if (col < a.m_tokens) {
                      a.tile_max[static_cast<size_t>(col) * a.n_tiles + tile] = ms_max(r);
                      a.tile_sum[static_cast<size_t>(col) * a.n_tiles + tile] = ms_sum(r);
                    }
                  }
                }
              }
            }
            if (cs == 1) {
              tc_fence_before();
              named_bar_sync(NB_EPI, ep_n);
              if (et2 == 0) mbar_arrive(&bar[MB_TEMPTY + ab]);
            } else {
              named_bar_sync(NB_EPI, ep_n);
            }
            if (et2 == 0 && acc == acc_pos) trace_point(tq, 8);
            if (kind == 1 || kind == 3) {  // RESID: sums of squares of the updated rows, per token
              for (int c = et2; c < a.n_tok; c += ep_n) {
                const int tok = tt * a.n_tok + c;
                if ((c / 16) % cs == rank && tok < a.m_tokens)
                  a.ssq_out[static_cast<size_t>(tile) * a.ssq_ld + tok] =
                      sq_red[c] + sq_red[256 + c] + sq_red[512 + c] + sq_red[768 + c];
              }
            }
            if (cs > 1 && et2 == 0) {
              // the last member to finish resets the item's counters for the next split phase
              int* arrived = p.item_cnt + item;
              int* departed = p.item_cnt + kMaxSplitItems + item;
              if (atomicAdd(departed, 1) == cs - 1) {
                *arrived = 0;
                *departed = 0;
              }
            }
            named_bar_sync(NB_EPI, ep_n);
          }
          if (ok && kind == 4 && a.keys != nullptr && keep_best && items > 0)
            for (int c = et2; c < a.tok_tiles * a.n_tok; c += ep_n)
              if (c < a.m_tokens && best[c]) atomicMax(a.keys + c, best[c]);
        }
        a_pos += n_tiles_cta;
        b_pos += n_tiles_cta;
        if (raw) w_pos += n_tiles_cta;
        acc_pos += items;
      } else if (ok) {
        // ---------------------------------------------------------------- attention phase
        const int layer = q / 5;
        (void)layer;
        const int q4 = warp & 3, hf = warp >> 2;  // TMEM lane quarter, column half
        const int r = q4 * 32 + lane;             // row == TMEM lane
        const bool row_ok = r < at.rows_valid;
        const int jr = row_ok ? r / at.group : 0;
        const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
        const int bar_id = 2 + q4;  // the 64 threads that share these rows
        uint8_t* p_s = smem + C::ATT_P;
        int g0 = att_g, ic = att_ic;
        for (int it = blockIdx.x; ok && it < att_total; it += G, ++ic) {
          const Item x = decode(it);
          float o[HH];
#pragma unroll
          for (int d = 0; d < HH; ++d) o[d] = 0.0f;
          float m = -INFINITY, l = 0.0f;
          for (int i = 0; i < x.n; ++i) {
            const int g = g0 + i;
            if (!mwait(&bar[MB_SFULL + (g & 1)], static_cast<uint32_t>((g >> 1) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int c = x.c_begin + i;
            const bool blk = c >= x.n_ctx;
            const bool need_mask = blk || (c * 128 + 128 > x.L) || !row_ok;
            const int ncol = blk ? 16 : 64;  // this thread's columns of the chunk
            const int col0 = hf * ncol;
            const uint32_t sa = tmem + lane_base + (g & 1) * 128 + col0;
            float s[64];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              if (qq * 16 < ncol) tmem_ld16(sa + qq * 16, s + qq * 16);
            tmem_ld_wait();
            int lim = ncol;
            if (need_mask) lim = !row_ok ? 0 : min(ncol, blk ? jr + 1 - col0 : x.L - c * 128 - col0);
            const float sl = at.scale_log2;
            float cm = -INFINITY;
#pragma unroll
            for (int tt = 0; tt < 64; ++tt) {
              s[tt] = tt < lim ? s[tt] * sl : -INFINITY;
              cm = fmaxf(cm, s[tt]);
            }
            float* xs = xstat + (g & 1) * 256;
            xs[hf * 128 + r] = cm;
            named_bar_sync(bar_id, 64);
            cm = fmaxf(xs[r], xs[128 + r]);
            const float m_new = fmaxf(m, cm);
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            const float alpha = ex2(m - m_use);
            float psum = 0.0f;
#pragma unroll
            for (int tt = 0; tt < 64; tt += 8) {
              if (tt < ncol) {
                uint32_t w[4], wl[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                  const float p0 = ex2(s[tt + e] - m_use), p1 = ex2(s[tt + e + 1] - m_use);
                  w[e >> 1] = f32x2_to_bf16x2(p0, p1);
                  const float h0 = __uint_as_float(w[e >> 1] << 16), h1 = __uint_as_float(w[e >> 1] & 0xFFFF0000u);
                  wl[e >> 1] = f32x2_to_bf16x2(p0 - h0, p1 - h1);
                  psum += p0 + p1;
                }
                const int key = col0 + tt;
                const uint32_t off = (key >> 6) * 16384 + sw128_off(r, (key & 63) >> 3);
                *reinterpret_cast<uint4*>(p_s + off) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(p_s + 32768 + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
              }
            }
            tc_fence_before();
            mbar_arrive(&bar[MB_SFREE + (g & 1)]);
            fence_proxy_async();
            mbar_arrive(&bar[MB_PFULL]);
            l = l * alpha + psum;
            m = m_new;
            if (!mwait(&bar[MB_OFULL], static_cast<uint32_t>(g & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            float vv[16];
#pragma unroll
            for (int d0 = 0; d0 < HH; d0 += 16) {
              tmem_ld16(tmem + lane_base + 256 + hf * HH + d0, vv);
              tmem_ld_wait();
#pragma unroll
              for (int tt = 0; tt < 16; ++tt) o[d0 + tt] = o[d0 + tt] * alpha + vv[tt];
            }
            tc_fence_before();
            mbar_arrive(&bar[MB_OFREE]);
          }
          g0 += x.n;
          if (!ok) break;
          float* xl = xstat + 512 + (ic & 1) * 256;
          xl[hf * 128 + r] = l;
          named_bar_sync(bar_id, 64);
          const float lt = xl[r] + xl[128 + r];
          const size_t pair = static_cast<size_t>(x.b) * at.n_kv + x.h;
          const int hq = row_ok ? r % at.group : 0;
          __half* dst = at.out + (static_cast<size_t>(x.b) * kRows + jr) * (at.n_q * HD) + (x.h * at.group + hq) * HD +
                        hf * HH;
          if (x.n_splits == 1) {
            if (row_ok) {
              const float inv = 1.0f / lt;
#pragma unroll
              for (int d = 0; d < HH; d += 8) {
                uint32_t hw[4], lw[4];
                f16_pairs8(o + d, inv, hw, lw);
                *reinterpret_cast<uint4*>(dst + d) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                if (at.out_lo) *reinterpret_cast<uint4*>(dst + at.out_lo + d) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
              }
            }
            continue;
          }
          // split partial, staged through shared memory for coalesced stores
          constexpr int Q4 = HH / 4;
          constexpr int NF4 = 128 * Q4;
          float4* stage = reinterpret_cast<float4*>(p_s);
          auto slot = [&](int rr, int d4) { return rr * Q4 + (d4 ^ (rr & 7)); };
          const size_t split_idx = pair * at.max_splits + x.split;
          float4* po = reinterpret_cast<float4*>(at.part_o + split_idx * 128 * HD);
          for (int hh = 0; hh < 2; ++hh) {
            if (hf == hh) {
#pragma unroll
              for (int d4 = 0; d4 < Q4; ++d4)
                stage[slot(r, d4)] = make_float4(o[4 * d4], o[4 * d4 + 1], o[4 * d4 + 2], o[4 * d4 + 3]);
            }
            named_bar_sync(NB_ATT, 256);
            for (int j = t; j < NF4; j += 256) __stcg(po + hh * NF4 + j, stage[slot(j / Q4, j % Q4)]);
            named_bar_sync(NB_ATT, 256);
          }
          if (hf == 0) __stcg(reinterpret_cast<float2*>(at.part_ml) + split_idx * 128 + r, make_float2(m, lt));
          __threadfence();
          named_bar_sync(NB_ATT, 256);
          int* arrived = at.counters + pair;
          int* departed = at.counters + static_cast<size_t>(at.batch_cap) * at.n_kv + pair;
          if (t == 0) {
            atomicAdd(arrived, 1);
            const long long t0 = cycles();
            int okw = 1;
            while (ld_acquire_gpu(arrived) < x.n_splits) {
              if (aborted()) {
                okw = 0;
                break;
              }
              if (cycles() - t0 > p.wait_limit) {
                give_up(true);
                okw = 0;
                break;
              }
            }
            *flag_s = okw;
          }
          named_bar_sync(NB_ATT, 256);
          if (!*flag_s) {
            ok = false;
            break;
          }
          {
            const int r0 = x.split * at.rows_valid / x.n_splits, r1 = (x.split + 1) * at.rows_valid / x.n_splits;
            constexpr int Q = HD / 4;
            const size_t first = pair * at.max_splits;
            const float2* pml = reinterpret_cast<const float2*>(at.part_ml) + first * 128;
            const float4* pbase = reinterpret_cast<const float4*>(at.part_o + first * 128 * HD);
            for (int idx = t; idx < (r1 - r0) * Q; idx += 256) {
              const int rw = r0 + idx / Q, d4 = idx % Q;
              const int hh = d4 / Q4, w4 = d4 % Q4;
              const float4* po_row = pbase + hh * NF4 + rw * Q4 + w4;
              float mm = -INFINITY, ls = 0.0f;
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int s0 = 0; s0 < x.n_splits; s0 += 8) {
                float2 ml[8];
                float4 ov[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const bool in = s0 + j < x.n_splits;
                  ml[j] = in ? __ldcg(pml + (s0 + j) * 128 + rw) : make_float2(-INFINITY, 0.0f);
                  ov[j] = in ? __ldcg(po_row + static_cast<size_t>(s0 + j) * 2 * NF4) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                float bm = mm;
#pragma unroll
                for (int j = 0; j < 8; ++j) bm = fmaxf(bm, ml[j].x);
                const float bu = bm == -INFINITY ? 0.0f : bm;
                const float sc = ex2(mm - bu);
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
              __half* o_dst = at.out + (static_cast<size_t>(x.b) * kRows + rw / at.group) * (at.n_q * HD) +
                              (x.h * at.group + rw % at.group) * HD + d;
              const float y[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
              uint32_t hw[2], lw[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                hw[e] = f32x2_to_f16x2(y[2 * e], y[2 * e + 1]);
                const __half2 h2 = *reinterpret_cast<const __half2*>(&hw[e]);
                lw[e] = f32x2_to_f16x2(y[2 * e] - __low2float(h2), y[2 * e + 1] - __high2float(h2));
              }
              *reinterpret_cast<uint2*>(o_dst) = make_uint2(hw[0], hw[1]);
              if (at.out_lo) *reinterpret_cast<uint2*>(o_dst + at.out_lo) = make_uint2(lw[0], lw[1]);
            }
          }
          named_bar_sync(NB_ATT, 256);
          if (t == 0 && atomicAdd(departed, 1) == x.n_splits - 1) {
            *arrived = 0;
            *departed = 0;
          }
        }
        att_g += att_chunks;
        att_ic += att_items;
        // the attention buffers are free again (the producer may refill the region)
        named_bar_sync(NB_END, 256);
        if (t == 0) mbar_arrive(&bar[MB_ATTDONE]);
      }
      // ------------------------------------------------------------------ phase end
      // every compute thread's global writes, then one release per CTA
      fence_proxy_async_global();
      named_bar_sync(NB_END, 256);
      if (t == 0) {
        trace_point(tq, 0);
        __threadfence();
        red_release_add(sync + q, 1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) trace_end(tk, 1);
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) {
    // the last CTA out resets the phase counters for the next launch (every
    // CTA has passed all of its waits by the time it counts itself out)
    __threadfence();
    if (atomicAdd(sync + n_phases, 1) == G - 1) {
      for (int i = 0; i < n_phases; ++i) sync[i] = 0;
      sync[n_phases] = 0;
      sync[n_phases + 1] = 0;
      __threadfence();
    }
  }
}

}  // namespace vsd
