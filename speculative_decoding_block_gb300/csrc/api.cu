// api.cu -- the C ABI of include/vsd.h: model and cache objects, weight
// repacking, tensor maps, argument checks, and the kernel sequence of the
// greedy block-verify step.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "host_util.h"
#include "launch.h"
#include "quant_kernels.cuh"
#include "step_kernels.cuh"

using namespace vsd;

namespace {
thread_local std::string g_err;
}  // namespace

vsd_status vsd::fail(vsd_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D tiled tensor map over a row-major [outer, inner] matrix of 2-byte elements.
vsd_status tmap_2d(CUtensorMap* tm, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer,
                   uint32_t box_inner, uint32_t box_outer) {
  if (!get_encoder()) return fail(VSD_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(VSD_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu] box %u x %u", (int)r,
                (unsigned long long)outer, (unsigned long long)inner, box_outer, box_inner);
  return VSD_OK;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }
int ceil_div(int x, int m) { return (x + m - 1) / m; }


int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// One packed weight matrix of the GEMM kernel.
struct Linear {
  int fmt = 0;
  int n_rows = 0;   // packed rows with data (tile rows beyond are zero)
  int k = 0;
  int n_tiles = 0, k_tiles = 0;
  void* data = nullptr;        // tiles [n_tiles][k_tiles]: f16 (BF16 weights, MMA layout) | FP8 | NVFP4
  float* row_scale = nullptr;  // FP8 / NVFP4
  bool owns = true;
};

void free_linear(Linear& l) {
  if (l.owns && l.data) cudaFree(l.data);
  if (l.row_scale) cudaFree(l.row_scale);
  l.data = nullptr;
  l.row_scale = nullptr;
}

}  // namespace

struct vsd_model {
  vsd_model_config cfg{};
  uint16_t* embed = nullptr;
  Linear lm;
  std::vector<Linear> qkv, o, gu, down;
  float2* rope = nullptr;
  int sms = 1;
  int max_clusters[4] = {1, 1, 1, 1};  // resident GEMM clusters of 1, 2, 4, 8 CTAs
  uint64_t uid = 0;                     // distinct per created model (keys the cached step graphs)
  MkLayerW* mk_layers = nullptr;        // device [layers]: tile and scale pointers of every layer
};

struct vsd_kv {
  const vsd_model* m = nullptr;
  int max_batch = 0, max_tokens = 0, num_pages = 0, ppr = 0, m_alloc = 0;
  __nv_bfloat16 *k_pool = nullptr, *v_pool = nullptr;
  int* page_table = nullptr;
  float* x = nullptr;
  __half *u = nullptr, *act_o = nullptr, *act_a = nullptr;
  __nv_bfloat16 *q_tile = nullptr, *k_new = nullptr, *v_new = nullptr;
  unsigned long long* keys = nullptr;
  int* ctx_len = nullptr;
  int* req_ok = nullptr;
  float* ssq = nullptr;  // [ceil(H/128)][m_alloc] sums of squares of the residual rows
  float *attn_o = nullptr, *attn_ml = nullptr;
  int* attn_counters = nullptr;
  size_t attn_items_cap = 0;
  float* anchor = nullptr;  // [max_batch][H] residual row of the last accepted position (drafter input)
  int* zeros = nullptr;     // [max_batch] zero context lengths (the draft pass reads no cache)
  int* probe_flag = nullptr;  // one int nothing ever sets (the wait probe's flag)
  long long wait_limit = kWaitLimitCycles;  // SM cycles a persistent-kernel wait may take
  int step_kernel = VSD_STEP_LAYERED;       // how the decoder layers and the head are launched
  // slot state of the device-resident loop: lengths, pending, drafts, accepted [max_batch], outputs [max_batch][17]
  int *loop_seq = nullptr, *loop_pend = nullptr, *loop_drafts = nullptr, *loop_acc = nullptr, *loop_out = nullptr;
  // stochastic verification: per (row, vocabulary tile) sums, the drafts' logits, the decisions [max_batch][18]
  float *tile_max = nullptr, *tile_sum = nullptr, *draft_logit = nullptr;
  int* decided = nullptr;
  // vsd_verify_step replays a graph of the step captured on its first call
  // with the same arguments (a few kept, oldest replaced)
  struct StepGraph {
    uint64_t model_uid;
    int batch;
    const void* args[5];
    cudaGraphExec_t exec;
  };
  std::vector<StepGraph> graphs;
  cudaStream_t capture_stream = nullptr;
  // host-buffer step: [drafts 16B | seq B | pending B | accepted B | out 17B]
  // on the device and in pinned host memory (allocated on first use)
  int* io_dev = nullptr;
  int* io_host = nullptr;
  int* status = nullptr;
  // persistent step kernel: phase counters (+ exit counter, abort flag), split-k partial sums, per-item counters
  int* mk_sync = nullptr;
  float* mk_part = nullptr;
  int* mk_item_cnt = nullptr;
  unsigned long long* trace = nullptr;  // optional phase timestamps [launch][CTA][tag]
  int trace_launches = 0;
  int trace_seq = 0;
  // GEMM activation maps, one per token-tile height 16, 32, ..., 256 rows
  CUtensorMap tm_u[kActBoxes]{}, tm_o[kActBoxes]{}, tm_a[kActBoxes]{};
  CUtensorMap tm_q{}, tm_kc{}, tm_vc{}, tm_kn{}, tm_vn{};
};

namespace {

Trace next_trace(vsd_kv* kv) {
  Trace t{};
  if (kv && kv->trace) {
    t.buf = kv->trace;
    t.max_launches = kv->trace_launches;
    t.id = kv->trace_seq++;
  }
  return t;
}

// ------------------------------------------------------------------ weight packing
// Builds a Linear from canonical matrices stacked in order (all the same
// format and K); perm[p] = stacked source row of packed row p (-1 = zero row).
vsd_status build_linear(const vsd_weight* const* parts, const int* part_rows, int n_parts, int K,
                        const std::vector<int>& perm, cudaStream_t st, Linear* out) {
  const int fmt = parts[0]->fmt;
  int rows = 0;
  for (int i = 0; i < n_parts; ++i) {
    if (parts[i]->fmt != fmt) return fail(VSD_ERR_ARG, "stacked matrices must share one format");
    if (!parts[i]->data_dev) return fail(VSD_ERR_ARG, "weight data pointer is NULL");
    if (fmt != VSD_FMT_BF16 && !parts[i]->scale_dev) return fail(VSD_ERR_ARG, "weight scale pointer is NULL");
    if (fmt == VSD_FMT_NVFP4 && !parts[i]->tensor_scale_dev) return fail(VSD_ERR_ARG, "NVFP4 tensor scale is NULL");
    rows += part_rows[i];
  }
  if (fmt == VSD_FMT_NVFP4 && K % 16) return fail(VSD_ERR_ARG, "NVFP4 needs K %% 16 == 0 (K = %d)", K);
  const int np = static_cast<int>(perm.size());
  Linear L;
  L.fmt = fmt;
  L.n_rows = np;
  L.k = K;
  L.n_tiles = ceil_div(np, kTileN);
  L.k_tiles = ceil_div(K, kTileK);
  int* perm_d = nullptr;
  vsd_status s = dalloc(&perm_d, np, false);
  if (s) return s;
  CK(cudaMemcpyAsync(perm_d, perm.data(), np * sizeof(int), cudaMemcpyHostToDevice, st));
  if (fmt == VSD_FMT_BF16) {
    uint16_t* stacked = nullptr;
    if ((s = dalloc(&stacked, static_cast<size_t>(rows) * K, false))) return s;
    size_t off = 0;
    for (int i = 0; i < n_parts; ++i) {
      CK(cudaMemcpyAsync(stacked + off, parts[i]->data_dev, static_cast<size_t>(part_rows[i]) * K * 2,
                         cudaMemcpyDeviceToDevice, st));
      off += static_cast<size_t>(part_rows[i]) * K;
    }
    uint16_t* packed = nullptr;
    if ((s = dalloc(&packed, static_cast<size_t>(L.n_tiles) * L.k_tiles * 8192, false))) return s;
    pack_bf16_tiles_kernel<<<dim3(L.k_tiles, L.n_tiles), 256, 0, st>>>(stacked, perm_d, np, K, L.k_tiles, packed);
    CK(cudaGetLastError());
    CK(cudaStreamSynchronize(st));
    cudaFree(stacked);
    L.data = packed;
  } else {
    const size_t vbytes_row = fmt == VSD_FMT_FP8 ? K : K / 2;
    uint8_t* stacked = nullptr;
    uint8_t* stacked_sb = nullptr;
    float* src_scale = nullptr;
    if ((s = dalloc(&stacked, static_cast<size_t>(rows) * vbytes_row, false))) return s;
    if ((s = dalloc(&src_scale, rows, false))) return s;
    if (fmt == VSD_FMT_NVFP4 && (s = dalloc(&stacked_sb, static_cast<size_t>(rows) * (K / 16), false))) return s;
    size_t off = 0;
    for (int i = 0; i < n_parts; ++i) {
      const size_t r = part_rows[i];
      CK(cudaMemcpyAsync(stacked + off * vbytes_row, parts[i]->data_dev, r * vbytes_row, cudaMemcpyDeviceToDevice, st));
      if (fmt == VSD_FMT_FP8) {
        CK(cudaMemcpyAsync(src_scale + off, parts[i]->scale_dev, r * 4, cudaMemcpyDeviceToDevice, st));
      } else {
        CK(cudaMemcpyAsync(stacked_sb + off * (K / 16), parts[i]->scale_dev, r * (K / 16), cudaMemcpyDeviceToDevice, st));
        float S = 0.0f;  // every row of this matrix gets its tensor scale
        CK(cudaMemcpyAsync(&S, parts[i]->tensor_scale_dev, 4, cudaMemcpyDeviceToHost, st));
        CK(cudaStreamSynchronize(st));
        std::vector<float> rep(r, S);
        CK(cudaMemcpyAsync(src_scale + off, rep.data(), r * 4, cudaMemcpyHostToDevice, st));
        CK(cudaStreamSynchronize(st));
      }
      off += r;
    }
    const uint32_t tile_bytes = fmt == VSD_FMT_FP8 ? kFp8TileBytes : kFp4TileBytes;
    uint8_t* tiles = nullptr;
    if ((s = dalloc(&tiles, static_cast<size_t>(L.n_tiles) * L.k_tiles * tile_bytes, false))) return s;
    if ((s = dalloc(&L.row_scale, static_cast<size_t>(L.n_tiles) * kTileN))) return s;
    dim3 grid(L.k_tiles, L.n_tiles);
    if (fmt == VSD_FMT_FP8) {
      pack_fp8_kernel<<<grid, 256, 0, st>>>(stacked, src_scale, perm_d, np, K, L.k_tiles, tiles, L.row_scale);
    } else {
      pack_fp4_kernel<<<grid, 256, 0, st>>>(stacked, stacked_sb, perm_d, np, K, L.k_tiles, tiles);
      pack_row_scale_kernel<<<ceil_div(np, 256), 256, 0, st>>>(src_scale, perm_d, np, L.row_scale);
    }
    CK(cudaGetLastError());
    CK(cudaStreamSynchronize(st));
    cudaFree(stacked);
    cudaFree(src_scale);
    if (stacked_sb) cudaFree(stacked_sb);
    L.data = tiles;
  }
  cudaFree(perm_d);
  *out = L;
  return VSD_OK;
}

// Packed QKV rows: within every head, row pairs (i, i + hd/2) become
// neighbours (2i, 2i+1) so that the RoPE partner sits in the adjacent lane.
std::vector<int> rope_pair_perm(int rows, int hd) {
  std::vector<int> p(rows);
  for (int r = 0; r < rows; ++r) {
    const int head = r / hd, w = r % hd;
    p[r] = head * hd + ((w & 1) ? (w >> 1) + hd / 2 : (w >> 1));
  }
  return p;
}

// Packed gate/up rows: tile t holds 64 features, gate row of feature f at
// 2(f - 64t), up row right after it.  Stacked source: [wg; wu].
std::vector<int> gate_up_perm(int ffn) {
  const int fp = round_up(ffn, 64);
  std::vector<int> p(2 * fp);
  for (int r = 0; r < 2 * fp; ++r) {
    const int t = r / 128, w = r % 128, f = t * 64 + (w >> 1);
    p[r] = f < ffn ? ((w & 1) ? ffn + f : f) : -1;
  }
  return p;
}

std::vector<int> identity_perm(int n) {
  std::vector<int> p(n);
  for (int i = 0; i < n; ++i) p[i] = i;
  return p;
}

// ------------------------------------------------------------------ GEMM planning

struct Plan {
  int n_tok, tok_tiles, cs, kps, rd, da, db, grid;
  bool r_alias;
};

// Chooses token tiles (MMA N <= 256) and the k split (cluster of 1..8 CTAs)
// with a latency model fitted to traced steps (microseconds): each CTA pays
// a fixed launch / start-up / drain cost, about 0.6 us per k tile (weight
// expansion and MMA pipeline; 0.5 for 16-bit weights), and its share of the
// epilogue's 16-column groups; a split adds the cluster reduction, which
// grows with the columns exchanged.  Clusters beyond what can be resident
// at once run in further waves.
Plan plan_gemm(const vsd_model* m, const Linear& w, int M, int epi, bool lo) {
  const bool no_split = epi == EPI_ARGMAX || epi == EPI_SAMPLE;  // the epilogue needs the finished dot products
  const double t_group = epi == EPI_QKV ? 1.5 : (epi == EPI_ARGMAX || epi == EPI_SAMPLE || epi == EPI_STORE ? 0.3 : 0.5);
  Plan best{};
  double best_cost = 1e30;
  const int max_t = std::max(1, ceil_div(M, 16));
  for (int t = ceil_div(M, 256); t <= max_t; ++t) {
    const int n_tok = std::max(16, round_up(ceil_div(M, t), 16));
    if (n_tok > 256 || (t > 1 && round_up(ceil_div(M, t - 1), 16) == n_tok)) continue;
    // MMA instructions per k tile: 4, or 8 when lo rows do not fit beside the hi rows (N <= 256)
    const int n_mma = (lo && 2 * n_tok > 256) ? 8 : 4;
    const double t_tile = (w.fmt == VSD_FMT_BF16 ? 0.26 : 0.36) + 0.06 * n_mma;
    for (int li = 0; li < 4; ++li) {
      const int want = 1 << li;
      if (no_split && want > 1) break;
      if (want > w.k_tiles) break;
      const int kps = ceil_div(w.k_tiles, want);
      const int cs = ceil_div(w.k_tiles, kps);  // every rank gets at least one k tile
      const int csi = cs <= 1 ? 0 : (cs <= 2 ? 1 : (cs <= 4 ? 2 : 3));
      const int items = w.n_tiles * t;
      const int resident = std::max(1, std::min(m->max_clusters[csi], m->sms / cs));
      const int waves = ceil_div(items, resident);
      const int groups = ceil_div(ceil_div(n_tok, 16), cs);
      double cost = waves * (6.0 + kps * t_tile + groups * t_group);
      if (cs > 1) cost += 2.5 + 0.035 * n_tok + 0.1 * cs;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best.tok_tiles = t;
        best.n_tok = n_tok;
        best.kps = kps;
        best.cs = cs;
      }
    }
  }
  const int csi = best.cs <= 1 ? 0 : (best.cs <= 2 ? 1 : (best.cs <= 4 ? 2 : 3));
  const int items = w.n_tiles * best.tok_tiles;
  const int clusters = std::max(1, std::min({items, m->sms / best.cs, std::max(1, m->max_clusters[csi])}));
  best.grid = clusters * best.cs;
  // ring depths: as deep as the CTA's k stream, trimmed until the shared
  // memory fits -- weights beyond 6 slots first, then activations beyond 4
  const int ki = ceil_div(items, clusters) * best.kps;  // k iterations of one CTA
  best.r_alias = best.cs > 1 && items <= clusters;
  auto fits = [&](int da, int db, int rd) {
    return gemm_smem_bytes(w.fmt, best.n_tok, rd, da, db, best.cs, lo, best.r_alias) <= 232448;
  };
  if (w.fmt == VSD_FMT_BF16) {
    best.da = 1;
    int d = std::max(2, std::min(8, ki));
    while (d > 2 && !fits(1, d, d)) --d;
    best.rd = best.db = d;
  } else {
    int da = std::max(2, std::min(kMaxDa, ki)), db = std::max(2, std::min(kMaxDb, ki));
    int rd = std::max(2, std::min(kMaxRd, ki));
    while (!fits(da, db, rd)) {
      if (rd > 6) --rd;
      else if (db > 4) --db;
      else if (rd > 4) --rd;
      else if (db > 3) --db;
      else if (da > 2) --da;
      else if (rd > 2) --rd;
      else if (db > 2) --db;
      else break;
    }
    best.da = da;
    best.db = db;
    best.rd = rd;
  }
  return best;
}

// Per-token RMSNorm scale of the GEMM input (rows held unnormalised).
void set_norm_input(GemmArgs& a, const vsd_kv* kv) {
  const vsd_model_config& c = kv->m->cfg;
  a.ssq_in = kv->ssq;
  a.n_ssq = ceil_div(c.hidden, kTileN);
  a.ssq_ld = kv->m_alloc;
  a.inv_hidden = 1.0f / static_cast<float>(c.hidden);
  a.eps = c.eps;
}

vsd_status run_gemm(const vsd_model* m, const Linear& w, int epi, const CUtensorMap* tm_acts, int M, GemmArgs a,
                    int* status, cudaStream_t st, Trace trace = Trace{}) {
  const bool lo = a.act_lo_rows > 0;
  const Plan p = plan_gemm(m, w, M, epi, lo);
  a.w_tiles = static_cast<const uint8_t*>(w.data);
  a.row_scale = w.row_scale;
  a.n_rows = w.n_rows;
  a.n_tiles = w.n_tiles;
  a.k_tiles = w.k_tiles;
  a.tok_tiles = p.tok_tiles;
  a.n_tok = p.n_tok;
  a.cs = p.cs;
  a.kps = p.kps;
  a.m_tokens = M;
  a.rd = p.rd;
  a.da = p.da;
  a.db = p.db;
  a.status = status;
  a.trace = trace;
  a.r_alias = p.r_alias ? 1 : 0;
  if (gemm_smem_bytes(w.fmt, p.n_tok, p.rd, p.da, p.db, p.cs, lo, p.r_alias) > 232448)
    return fail(VSD_ERR_UNSUPPORTED, "GEMM tile does not fit in shared memory");
  const cudaError_t e = launch_gemm(w.fmt, epi, tm_acts[p.n_tok / 16 - 1], a, p.grid, st, use_pdl(st));
  if (e != cudaSuccess) return fail(VSD_ERR_CUDA, "gemm launch: %s", cudaGetErrorString(e));
  return VSD_OK;
}

// lo: the q tiles carry lo halves and the output gets its lo copy (the step);
// otherwise hi only (the single-layer entry point, whose inputs are BF16)
vsd_status run_attention(vsd_kv* kv, int layer, int B, const int* seq_lens, cudaStream_t st, bool lo) {
  const vsd_model* m = kv->m;
  const vsd_model_config& c = m->cfg;
  if (B > kMaxReqs) return fail(VSD_ERR_UNSUPPORTED, "at most %d requests per step", kMaxReqs);
  const int max_chunks = ceil_div(kv->max_tokens, 128) + 1;
  // about two work items per SM at the longest contexts
  int cps = std::max(1, ceil_div(B * c.n_kv * max_chunks, 2 * m->sms));
  const int max_splits = ceil_div(max_chunks, cps);
  if (static_cast<size_t>(B) * c.n_kv * max_splits > kv->attn_items_cap)
    return fail(VSD_ERR_UNSUPPORTED, "attention workspace too small");
  const int grid = std::min(B * c.n_kv * max_splits, m->sms);
  AttnArgs a{};
  a.batch = B;
  a.batch_cap = kv->max_batch;
  a.n_q = c.n_q;
  a.n_kv = c.n_kv;
  a.hd = c.head_dim;
  a.group = c.n_q / c.n_kv;
  a.rows_valid = kRows * a.group;
  a.chunks_per_split = cps;
  a.max_splits = max_splits;
  a.layer = layer;
  a.num_pages = kv->num_pages;
  a.pages_per_req = kv->ppr;
  a.max_tokens = kv->max_tokens;
  a.seq_lens = seq_lens;
  a.page_table = kv->page_table;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c.head_dim)));
  a.part_o = kv->attn_o;
  a.part_ml = kv->attn_ml;
  a.counters = kv->attn_counters;
  a.out = kv->act_o;
  if (lo) {
    a.out_lo = static_cast<size_t>(kv->m_alloc) * c.n_q * c.head_dim;
    a.q_lo_rows = kv->max_batch * c.n_kv * 128;
  }
  a.status = kv->status;
  a.trace = next_trace(kv);
  const cudaError_t e = launch_attn(c.head_dim, kv->tm_q, kv->tm_kc, kv->tm_vc, kv->tm_kn, kv->tm_vn, a,
                                    dim3(grid), st, use_pdl(st));
  if (e != cudaSuccess) return fail(VSD_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  return VSD_OK;
}

CommitArgs commit_args(const vsd_kv* kv, const int* drafts, int* seq_lens, int* pending, int* accepted,
                       int* out_tokens) {
  const vsd_model_config& c = kv->m->cfg;
  CommitArgs ca{};
  ca.vocab = c.vocab;
  ca.layers = c.layers;
  ca.n_kv = c.n_kv;
  ca.hd = c.head_dim;
  ca.batch_cap = kv->max_batch;
  ca.num_pages = kv->num_pages;
  ca.pages_per_req = kv->ppr;
  ca.keys = kv->keys;
  ca.drafts = drafts;
  ca.ctx_len = kv->ctx_len;
  ca.req_ok = kv->req_ok;
  ca.seq_lens = seq_lens;
  ca.pending = pending;
  ca.accepted = accepted;
  ca.out_tokens = out_tokens;
  ca.page_table = kv->page_table;
  ca.k_new = kv->k_new;
  ca.v_new = kv->v_new;
  ca.k_pool = kv->k_pool;
  ca.v_pool = kv->v_pool;
  ca.status = kv->status;
  return ca;
}

vsd_status check_model_config(const vsd_model_config* c) {
  if (!c) return fail(VSD_ERR_ARG, "config is NULL");
  if (c->layers < 1 || c->hidden < 64 || c->n_q < 1 || c->n_kv < 1 || c->ffn < 16 || c->vocab < 2 ||
      c->max_positions < vsd::kRows)
    return fail(VSD_ERR_ARG, "config has a non-positive or too small dimension");
  if (c->head_dim != 64 && c->head_dim != 128) return fail(VSD_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c->n_q % c->n_kv) return fail(VSD_ERR_ARG, "n_q must be a multiple of n_kv");
  if (kRows * (c->n_q / c->n_kv) > 128)
    return fail(VSD_ERR_UNSUPPORTED, "17 * (n_q / n_kv) must fit a 128-row attention tile");
  if (c->hidden % 8 || c->ffn % 8 || (c->n_q * c->head_dim) % 8)
    return fail(VSD_ERR_UNSUPPORTED, "hidden, ffn and n_q*head_dim must be multiples of 8");
  if (c->hidden > 16384) return fail(VSD_ERR_UNSUPPORTED, "hidden above 16384");
  for (int f : {c->attn_fmt, c->mlp_fmt})
    if (f < VSD_FMT_BF16 || f > VSD_FMT_NVFP4) return fail(VSD_ERR_ARG, "unknown weight format %d", f);
  if (!(c->eps > 0.0f) || !(c->rope_theta > 0.0f)) return fail(VSD_ERR_ARG, "eps and rope_theta must be > 0");
  return VSD_OK;
}

}  // namespace

extern "C" {

const char* vsd_version(void) { return "vsd 0.1 sm_103a"; }
const char* vsd_last_error(void) { return g_err.c_str(); }

// ------------------------------------------------------------------ quantisers
vsd_status vsd_quantize_fp8_rowwise(const uint16_t* w, int32_t n, int32_t k, uint8_t* q, float* scale,
                                    vsd_stream stream) {
  if (!w || !q || !scale) return fail(VSD_ERR_ARG, "NULL pointer");
  if (n < 1 || k < 2 || (k & 1)) return fail(VSD_ERR_ARG, "need n >= 1 and an even k >= 2");
  quant_fp8_rowwise_kernel<<<n, 256, 0, stream>>>(w, k, q, scale);
  CK(cudaGetLastError());
  return VSD_OK;
}

vsd_status vsd_quantize_nvfp4(const uint16_t* w, int32_t n, int32_t k, uint8_t* q, uint8_t* sb, float* S,
                              vsd_stream stream) {
  if (!w || !q || !sb || !S) return fail(VSD_ERR_ARG, "NULL pointer");
  if (n < 1 || k < 16 || (k % 16)) return fail(VSD_ERR_ARG, "need n >= 1 and k a positive multiple of 16");
  const size_t total = static_cast<size_t>(n) * k;
  CK(cudaMemsetAsync(S, 0, 4, stream));
  amax_kernel<<<std::min<size_t>(1024, (total + 255) / 256), 256, 0, stream>>>(w, total,
                                                                               reinterpret_cast<unsigned int*>(S));
  const size_t nb = total / 16;
  quant_nvfp4_kernel<<<(nb + 255) / 256, 256, 0, stream>>>(w, nb, S, q, sb);
  nvfp4_tensor_scale_kernel<<<1, 1, 0, stream>>>(S);
  CK(cudaGetLastError());
  return VSD_OK;
}

// ------------------------------------------------------------------ model
vsd_status vsd_model_create(const vsd_model_config* cfg, const vsd_weights* w, vsd_stream stream, vsd_model** out) {
  if (!out) return fail(VSD_ERR_ARG, "out is NULL");
  *out = nullptr;
  vsd_status s = check_model_config(cfg);
  if (s) return s;
  if (!w || !w->embed_dev || !w->layers) return fail(VSD_ERR_ARG, "weights are NULL");
  if (!cfg->tied && !w->lm_head_dev) return fail(VSD_ERR_ARG, "untied model needs lm_head");
  int dev_count = 0;
  if (cudaGetDeviceCount(&dev_count) != cudaSuccess || dev_count < 1) return fail(VSD_ERR_CUDA, "no CUDA device");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const vsd_model_config& c = *cfg;
  vsd_model* m = new vsd_model();
  static std::atomic<uint64_t> next_uid{1};
  m->uid = next_uid++;
  m->cfg = c;
  m->sms = sm_count();
  for (int i = 0; i < 4; ++i) m->max_clusters[i] = gemm_max_clusters(1 << i);
  auto cleanup = [&](vsd_status e) {
    vsd_model_destroy(m);
    return e;
  };
  const int H = c.hidden, hd = c.head_dim, F = c.ffn;
  if ((s = dalloc(&m->embed, static_cast<size_t>(c.vocab) * H, false))) return cleanup(s);
  if (cudaMemcpyAsync(m->embed, w->embed_dev, static_cast<size_t>(c.vocab) * H * 2, cudaMemcpyDeviceToDevice, st))
    return cleanup(fail(VSD_ERR_CUDA, "embedding copy failed"));
  // lm_head: BF16 rows of the vocabulary
  vsd_weight lmw{VSD_FMT_BF16, c.tied ? m->embed : w->lm_head_dev, nullptr, nullptr};
  const vsd_weight* lmp = &lmw;
  int vrows = c.vocab;
  if ((s = build_linear(&lmp, &vrows, 1, H, identity_perm(c.vocab), st, &m->lm))) return cleanup(s);
  const int nq = c.n_q * hd, nk = c.n_kv * hd;
  for (int l = 0; l < c.layers; ++l) {
    const vsd_weight* L = w->layers + static_cast<size_t>(l) * 7;
    for (int i = 0; i < 7; ++i) {
      const int want = i < 4 ? c.attn_fmt : c.mlp_fmt;
      if (L[i].fmt != want) return cleanup(fail(VSD_ERR_ARG, "layer %d matrix %d has format %d, config says %d", l, i, L[i].fmt, want));
    }
    Linear lin;
    const vsd_weight* qkv[3] = {&L[0], &L[1], &L[2]};
    int qkv_rows[3] = {nq, nk, nk};
    if ((s = build_linear(qkv, qkv_rows, 3, H, rope_pair_perm(nq + 2 * nk, hd), st, &lin))) return cleanup(s);
    m->qkv.push_back(lin);
    const vsd_weight* op = &L[3];
    int orows = H;
    if ((s = build_linear(&op, &orows, 1, nq, identity_perm(H), st, &lin))) return cleanup(s);
    m->o.push_back(lin);
    const vsd_weight* gu[2] = {&L[4], &L[5]};
    int gu_rows[2] = {F, F};
    if ((s = build_linear(gu, gu_rows, 2, H, gate_up_perm(F), st, &lin))) return cleanup(s);
    m->gu.push_back(lin);
    const vsd_weight* dp = &L[6];
    if ((s = build_linear(&dp, &orows, 1, F, identity_perm(H), st, &lin))) return cleanup(s);
    m->down.push_back(lin);
  }
  {
    std::vector<MkLayerW> tab(c.layers);
    for (int l = 0; l < c.layers; ++l) {
      const Linear* ls[4] = {&m->qkv[l], &m->o[l], &m->gu[l], &m->down[l]};
      for (int k = 0; k < 4; ++k) {
        tab[l].w[k] = static_cast<const uint8_t*>(ls[k]->data);
        tab[l].s[k] = ls[k]->row_scale;
      }
    }
    if ((s = dalloc(&m->mk_layers, tab.size(), false))) return cleanup(s);
    if (cudaMemcpy(m->mk_layers, tab.data(), tab.size() * sizeof(MkLayerW), cudaMemcpyHostToDevice))
      return cleanup(fail(VSD_ERR_CUDA, "layer table copy failed"));
  }
  // RoPE table: angle = pos * theta^(-2i/hd), evaluated in double, stored as fp32 (cos, sin)
  {
    const int half = hd / 2;
    std::vector<float2> tab(static_cast<size_t>(c.max_positions) * half);
    for (int p = 0; p < c.max_positions; ++p)
      for (int i = 0; i < half; ++i) {
        const double ang = p * std::pow(static_cast<double>(c.rope_theta), -2.0 * i / hd);
        tab[static_cast<size_t>(p) * half + i] = make_float2(static_cast<float>(std::cos(ang)), static_cast<float>(std::sin(ang)));
      }
    if ((s = dalloc(&m->rope, tab.size(), false))) return cleanup(s);
    if (cudaMemcpy(m->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice))
      return cleanup(fail(VSD_ERR_CUDA, "RoPE table copy failed"));
  }
  if (cudaStreamSynchronize(st) != cudaSuccess) return cleanup(fail(VSD_ERR_CUDA, "model creation failed"));
  *out = m;
  return VSD_OK;
}

void vsd_model_destroy(vsd_model* m) {
  if (!m) return;
  free_linear(m->lm);
  for (auto* v : {&m->qkv, &m->o, &m->gu, &m->down})
    for (auto& l : *v) free_linear(l);
  if (m->embed) cudaFree(m->embed);
  if (m->rope) cudaFree(m->rope);
  if (m->mk_layers) cudaFree(m->mk_layers);
  delete m;
}

// ------------------------------------------------------------------ KV cache + workspace
vsd_status vsd_kv_create(const vsd_model* m, int32_t max_batch, int32_t max_tokens, int32_t page_size,
                         int32_t num_pages, vsd_kv** out) {
  if (!m || !out) return fail(VSD_ERR_ARG, "NULL pointer");
  *out = nullptr;
  if (page_size != kPage) return fail(VSD_ERR_UNSUPPORTED, "page_size must be 16");
  if (max_batch < 1 || max_batch > 4096) return fail(VSD_ERR_ARG, "max_batch out of range");
  if (max_tokens < kRows || max_tokens > m->cfg.max_positions)
    return fail(VSD_ERR_ARG, "max_tokens_per_req must lie in [17, max_positions]");
  const vsd_model_config& c = m->cfg;
  vsd_kv* kv = new vsd_kv();
  auto cleanup = [&](vsd_status e) {
    vsd_kv_destroy(kv);
    return e;
  };
  kv->m = m;
  kv->max_batch = max_batch;
  kv->max_tokens = max_tokens;
  kv->ppr = ceil_div(max_tokens, kPage);
  kv->num_pages = num_pages > 0 ? num_pages : max_batch * kv->ppr;
  const int hd = c.head_dim, H = c.hidden, F = c.ffn, nqd = c.n_q * hd;
  const size_t pool = static_cast<size_t>(c.layers) * kv->num_pages * c.n_kv * kPage * hd;
  vsd_status s;
  if ((s = dalloc(&kv->k_pool, pool)) || (s = dalloc(&kv->v_pool, pool))) return cleanup(s);
  {
    std::vector<int> ident(static_cast<size_t>(max_batch) * kv->ppr);
    for (size_t i = 0; i < ident.size(); ++i) ident[i] = static_cast<int>(i % kv->num_pages);
    if ((s = dalloc(&kv->page_table, ident.size(), false))) return cleanup(s);
    if (cudaMemcpy(kv->page_table, ident.data(), ident.size() * 4, cudaMemcpyHostToDevice))
      return cleanup(fail(VSD_ERR_CUDA, "page table copy failed"));
  }
  const int M = kRows * max_batch;
  kv->m_alloc = round_up(M, 16);
  // GEMM inputs and the attention's q tiles are hi / lo pairs: [2][rows][cols]
  if ((s = dalloc(&kv->x, static_cast<size_t>(kv->m_alloc) * H)) ||
      (s = dalloc(&kv->u, static_cast<size_t>(2) * kv->m_alloc * H)) ||
      (s = dalloc(&kv->act_o, static_cast<size_t>(2) * kv->m_alloc * nqd)) ||
      (s = dalloc(&kv->act_a, static_cast<size_t>(2) * kv->m_alloc * F)) ||
      (s = dalloc(&kv->q_tile, static_cast<size_t>(2) * max_batch * c.n_kv * 128 * hd)) ||
      (s = dalloc(&kv->k_new, static_cast<size_t>(c.layers) * max_batch * c.n_kv * 32 * hd)) ||
      (s = dalloc(&kv->v_new, static_cast<size_t>(c.layers) * max_batch * c.n_kv * 32 * hd)) ||
      (s = dalloc(&kv->keys, M)) || (s = dalloc(&kv->ctx_len, max_batch)) || (s = dalloc(&kv->req_ok, max_batch)) ||
      (s = dalloc(&kv->anchor, static_cast<size_t>(max_batch) * H)) || (s = dalloc(&kv->zeros, max_batch)) ||
      (s = dalloc(&kv->probe_flag, 1)) ||
      (s = dalloc(&kv->loop_seq, max_batch)) || (s = dalloc(&kv->loop_pend, max_batch)) ||
      (s = dalloc(&kv->loop_drafts, static_cast<size_t>(max_batch) * kBlock)) ||
      (s = dalloc(&kv->loop_acc, max_batch)) || (s = dalloc(&kv->loop_out, static_cast<size_t>(max_batch) * kRows)) ||
      (s = dalloc(&kv->tile_max, static_cast<size_t>(kv->m_alloc) * m->lm.n_tiles)) ||
      (s = dalloc(&kv->tile_sum, static_cast<size_t>(kv->m_alloc) * m->lm.n_tiles)) ||
      (s = dalloc(&kv->draft_logit, kv->m_alloc)) ||
      (s = dalloc(&kv->decided, static_cast<size_t>(max_batch) * (kRows + 1))) ||
      (s = dalloc(&kv->status, 1)))
    return cleanup(s);
  if ((s = dalloc(&kv->ssq, static_cast<size_t>(ceil_div(H, kTileN)) * kv->m_alloc))) return cleanup(s);
  // persistent step kernel: counters zero between launches (the kernel resets them on exit)
  if ((s = dalloc(&kv->mk_sync, static_cast<size_t>(5) * c.layers + 3)) ||
      (s = dalloc(&kv->mk_item_cnt, static_cast<size_t>(2) * kMaxSplitItems)) ||
      (s = dalloc(&kv->mk_part, static_cast<size_t>(m->sms) * kMkMaxTok * kTileN, false)))
    return cleanup(s);
  kv->attn_items_cap = static_cast<size_t>(4) * m->sms + static_cast<size_t>(2) * max_batch * c.n_kv;
  if ((s = dalloc(&kv->attn_o, kv->attn_items_cap * 128 * hd, false)) ||
      (s = dalloc(&kv->attn_ml, kv->attn_items_cap * 128 * 2, false)) ||
      (s = dalloc(&kv->attn_counters, static_cast<size_t>(2) * max_batch * c.n_kv)))
    return cleanup(s);
  const auto F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16, BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  for (int j = 0; j < kActBoxes; ++j) {
    const uint32_t rows = 16u * (j + 1);
    if ((s = tmap_2d(&kv->tm_u[j], kv->u, F16, H, 2 * kv->m_alloc, 64, rows)) ||
        (s = tmap_2d(&kv->tm_o[j], kv->act_o, F16, nqd, 2 * kv->m_alloc, 64, rows)) ||
        (s = tmap_2d(&kv->tm_a[j], kv->act_a, F16, F, 2 * kv->m_alloc, 64, rows)))
      return cleanup(s);
  }
  if ((s = tmap_2d(&kv->tm_q, kv->q_tile, BF16, hd, static_cast<uint64_t>(2) * max_batch * c.n_kv * 128, 64, 128)) ||
      (s = tmap_2d(&kv->tm_kc, kv->k_pool, BF16, hd, pool / hd, 64, 16)) ||
      (s = tmap_2d(&kv->tm_vc, kv->v_pool, BF16, hd, pool / hd, 64, 16)) ||
      (s = tmap_2d(&kv->tm_kn, kv->k_new, BF16, hd, static_cast<uint64_t>(c.layers) * max_batch * c.n_kv * 32, 64, 32)) ||
      (s = tmap_2d(&kv->tm_vn, kv->v_new, BF16, hd, static_cast<uint64_t>(c.layers) * max_batch * c.n_kv * 32, 64, 32)))
    return cleanup(s);
  if (cudaDeviceSynchronize() != cudaSuccess) return cleanup(fail(VSD_ERR_CUDA, "cache creation failed"));
  *out = kv;
  return VSD_OK;
}

void vsd_kv_destroy(vsd_kv* kv) {
  if (!kv) return;
  for (auto& g : kv->graphs) cudaGraphExecDestroy(g.exec);
  if (kv->capture_stream) cudaStreamDestroy(kv->capture_stream);
  if (kv->io_dev) cudaFree(kv->io_dev);
  if (kv->io_host) cudaFreeHost(kv->io_host);
  void* ptrs[] = {kv->k_pool, kv->v_pool, kv->page_table, kv->x, kv->u, kv->act_o, kv->act_a, kv->q_tile,
                  kv->k_new, kv->v_new, kv->keys, kv->ctx_len, kv->req_ok, kv->ssq, kv->attn_o,
                  kv->attn_ml, kv->attn_counters, kv->anchor, kv->zeros, kv->probe_flag, kv->loop_seq, kv->loop_pend,
                  kv->loop_drafts, kv->loop_acc, kv->loop_out, kv->tile_max, kv->tile_sum, kv->draft_logit, kv->decided,
                  kv->status, kv->trace, kv->mk_sync, kv->mk_part, kv->mk_item_cnt};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  delete kv;
}

int32_t vsd_kv_pages_per_req(const vsd_kv* kv) { return kv ? kv->ppr : -1; }
int32_t vsd_kv_num_pages(const vsd_kv* kv) { return kv ? kv->num_pages : -1; }

vsd_status vsd_kv_set_page_table(vsd_kv* kv, const int32_t* table, vsd_stream stream) {
  if (!kv || !table) return fail(VSD_ERR_ARG, "NULL pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t n = static_cast<size_t>(kv->max_batch) * kv->ppr;
  CK(cudaMemcpyAsync(kv->page_table, table, n * 4, cudaMemcpyDeviceToDevice, st));
  check_pages_kernel<<<64, 256, 0, st>>>(kv->page_table, n, kv->num_pages, kv->status);
  CK(cudaGetLastError());
  return VSD_OK;
}

static vsd_status kv_rows(const vsd_kv* kv, int req, int start, int count, uint16_t* k, uint16_t* v, int write,
                          cudaStream_t st) {
  if (!kv || !k || !v) return fail(VSD_ERR_ARG, "NULL pointer");
  if (req < 0 || req >= kv->max_batch) return fail(VSD_ERR_ARG, "request slot out of range");
  if (start < 0 || count < 0 || start + count > kv->max_tokens) return fail(VSD_ERR_CAPACITY, "rows outside the cache");
  if (count == 0) return VSD_OK;
  const vsd_model_config& c = kv->m->cfg;
  const size_t n = static_cast<size_t>(c.layers) * count * c.n_kv * c.head_dim;
  const int grid = static_cast<int>(std::min<size_t>(4096, (n + 255) / 256));
  for (int pass = 0; pass < 2; ++pass)
    kv_rows_kernel<<<grid, 256, 0, st>>>(pass ? kv->v_pool : kv->k_pool, kv->page_table, kv->ppr, kv->num_pages,
                                         c.layers, c.n_kv, c.head_dim, req, start, count,
                                         reinterpret_cast<__nv_bfloat16*>(pass ? v : k), write, kv->status);
  CK(cudaGetLastError());
  return VSD_OK;
}

vsd_status vsd_kv_write(vsd_kv* kv, int32_t req, int32_t start, int32_t count, const uint16_t* k, const uint16_t* v,
                        vsd_stream stream) {
  return kv_rows(kv, req, start, count, const_cast<uint16_t*>(k), const_cast<uint16_t*>(v), 1,
                 reinterpret_cast<cudaStream_t>(stream));
}

vsd_status vsd_kv_read(const vsd_kv* kv, int32_t req, int32_t start, int32_t count, uint16_t* k, uint16_t* v,
                       vsd_stream stream) {
  return kv_rows(kv, req, start, count, k, v, 0, reinterpret_cast<cudaStream_t>(stream));
}

vsd_status vsd_trace_enable(vsd_kv* kv, int32_t max_launches) {
  if (!kv || max_launches < 0) return fail(VSD_ERR_ARG, "bad arguments");
  if (kv->trace) cudaFree(kv->trace);
  kv->trace = nullptr;
  kv->trace_launches = 0;
  kv->trace_seq = 0;
  if (max_launches == 0) return VSD_OK;
  vsd_status s;
  if ((s = dalloc(&kv->trace, static_cast<size_t>(max_launches) * kTraceCtas * kTraceTags))) return s;
  kv->trace_launches = max_launches;
  return VSD_OK;
}

vsd_status vsd_trace_read(vsd_kv* kv, uint64_t* slots_host, int32_t max_launches, int32_t* n_launches,
                          vsd_stream stream) {
  if (!kv || !slots_host || !n_launches || max_launches < 0) return fail(VSD_ERR_ARG, "bad arguments");
  if (!kv->trace) {
    *n_launches = 0;
    return VSD_OK;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int n = std::min(kv->trace_launches, max_launches);  // graph replays keep their capture-time ids
  const size_t bytes = static_cast<size_t>(n) * kTraceCtas * kTraceTags * 8;
  CK(cudaStreamSynchronize(st));
  if (n > 0) CK(cudaMemcpy(slots_host, kv->trace, bytes, cudaMemcpyDeviceToHost));
  CK(cudaMemset(kv->trace, 0, static_cast<size_t>(kv->trace_launches) * kTraceCtas * kTraceTags * 8));
  kv->trace_seq = 0;
  *n_launches = n;
  return VSD_OK;
}

vsd_status vsd_kv_set_step_kernel(vsd_kv* kv, int32_t mode) {
  if (!kv || (mode != VSD_STEP_LAYERED && mode != VSD_STEP_PERSISTENT)) return fail(VSD_ERR_ARG, "bad arguments");
  if (kv->step_kernel != mode) {
    // the cached step graphs hold the other mode's launches
    for (auto& g : kv->graphs) cudaGraphExecDestroy(g.exec);
    kv->graphs.clear();
    kv->step_kernel = mode;
  }
  return VSD_OK;
}

vsd_status vsd_debug_wait_probe(vsd_kv* kv, int64_t limit_cycles, vsd_stream stream) {
  if (!kv) return fail(VSD_ERR_ARG, "NULL pointer");
  if (limit_cycles < 1 || limit_cycles > kWaitLimitCycles) return fail(VSD_ERR_ARG, "limit out of range");
  wait_probe_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(kv->probe_flag, limit_cycles, kv->status);
  CK(cudaGetLastError());
  return VSD_OK;
}

vsd_status vsd_get_device_status(vsd_kv* kv, vsd_stream stream, int32_t* out) {
  if (!kv || !out) return fail(VSD_ERR_ARG, "NULL pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  CK(cudaMemcpyAsync(&v, kv->status, 4, cudaMemcpyDeviceToHost, st));
  CK(cudaMemsetAsync(kv->status, 0, 4, st));
  CK(cudaStreamSynchronize(st));
  *out = v;
  return VSD_OK;
}

// ------------------------------------------------------------------ the step
// Optional per-launch event timing of one step.
struct LaunchTimer {
  std::vector<cudaEvent_t> ev;
  std::vector<int> kinds;
  cudaStream_t st = nullptr;
  void before(int kind) {
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    ev.push_back(a);
    ev.push_back(b);
    kinds.push_back(kind);
    cudaEventRecord(a, st);
  }
  void after() { cudaEventRecord(ev.back(), st); }
  ~LaunchTimer() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
};

#define TIMED(kind, ...)          \
  do {                            \
    if (timer) timer->before(kind); \
    __VA_ARGS__;                  \
    if (timer) timer->after();    \
  } while (0)

// Stochastic verification inputs of one step (nullptr: greedy).
struct SampleIn {
  float inv_temp;
  const float* u_accept;  // [B][16]
  const float* u_sample;  // [B][17]
};

// The decoder layers of model m over the M = 17 B rows already in the
// residual scratch, then the final RMSNorm + head: per-row argmax keys
// (kv->keys; greedy) or, with `smp`, the per-tile exp sums and the drafts'
// logits; logits and hidden rows optional.  Attention reads attn_lens[b]
// cached rows per request.  One persistent launch (persistent.cuh).
static vsd_status run_persistent(const vsd_model* m, vsd_kv* kv, int B, const int* attn_lens, float* hidden,
                                 float* logits, const int* drafts, const SampleIn* smp, cudaStream_t st) {
  const vsd_model_config& c = m->cfg;
  const int M = kRows * B, H = c.hidden, G = m->sms;
  if (B > kMaxReqs) return fail(VSD_ERR_UNSUPPORTED, "at most %d requests per step", kMaxReqs);
  if (c.layers > kv->m->cfg.layers) return fail(VSD_ERR_ARG, "model deeper than the cache's target");
  MkParams p{};
  const int tok_tiles = ceil_div(M, kMkMaxTok);
  const int n_tok = round_up(ceil_div(M, tok_tiles), 16);
  p.tm_act[0] = kv->tm_u[n_tok / 16 - 1];
  p.tm_act[1] = kv->tm_o[n_tok / 16 - 1];
  p.tm_act[2] = kv->tm_a[n_tok / 16 - 1];
  p.tm_q = kv->tm_q;
  p.tm_kc = kv->tm_kc;
  p.tm_vc = kv->tm_vc;
  p.tm_kn = kv->tm_kn;
  p.tm_vn = kv->tm_vn;
  const Linear* lin[kMkKinds] = {&m->qkv[0], &m->o[0], &m->gu[0], &m->down[0], &m->lm};
  const int act_of[kMkKinds] = {0, 1, 0, 2, 0};
  for (int k = 0; k < kMkKinds; ++k) {
    GemmArgs& a = p.g[k];
    const Linear& w = *lin[k];
    a.n_rows = w.n_rows;
    a.n_tiles = w.n_tiles;
    a.k_tiles = w.k_tiles;
    a.tok_tiles = tok_tiles;
    a.n_tok = n_tok;
    a.m_tokens = M;
    // k split over consecutive CTAs when the output tiles alone leave most
    // SMs idle: as many members as fit the grid in one round, each with at
    // least one k tile and one 16-column group to finish
    const int items = w.n_tiles * tok_tiles;
    a.cs = 1;
    a.kps = w.k_tiles;
    if (k != 4 && 2 * items <= G) {
      const int cs_max = std::min({G / items, w.k_tiles, n_tok / 16});
      a.kps = ceil_div(w.k_tiles, cs_max);
      a.cs = ceil_div(w.k_tiles, a.kps);
    }
    if (a.cs > 1 && (items > kMaxSplitItems || static_cast<size_t>(items) * a.cs > static_cast<size_t>(G)))
      return fail(VSD_ERR_UNSUPPORTED, "split-k plan outside the workspace");
    a.act_lo_rows = kv->m_alloc;
    a.status = kv->status;
    p.wf[k] = w.fmt;
    p.act_of[k] = act_of[k];
  }
  {  // QKV: RoPE, q tile, block K / V scratch
    GemmArgs& a = p.g[0];
    set_norm_input(a, kv);
    a.q_tile = kv->q_tile;
    a.out_lo = static_cast<size_t>(kv->max_batch) * c.n_kv * 128 * c.head_dim;
    a.k_new = kv->k_new;
    a.v_new = kv->v_new;
    a.kv_layer_stride = static_cast<size_t>(kv->max_batch) * c.n_kv * 32 * c.head_dim;
    a.ctx_len = kv->ctx_len;
    a.rope = m->rope;
    a.n_q = c.n_q;
    a.n_kv = c.n_kv;
    a.head_dim = c.head_dim;
  }
  for (int k : {1, 3}) {  // O and down: residual update, f16 copy, sums of squares
    GemmArgs& a = p.g[k];
    a.out_f32 = kv->x;
    a.ld_out = H;
    a.x16_out = kv->u;
    a.out_lo = static_cast<size_t>(kv->m_alloc) * H;
    a.ssq_out = kv->ssq;
    a.ssq_ld = kv->m_alloc;
  }
  if (hidden) {  // layer l's output rows at hidden + (l + 1) M H
    p.g[3].hidden_out = hidden + static_cast<size_t>(M) * H;
    p.g[3].hidden_layer_stride = static_cast<size_t>(M) * H;
  }
  {  // gate/up: SiLU(gate) * up
    GemmArgs& a = p.g[2];
    set_norm_input(a, kv);
    a.act_out = kv->act_a;
    a.out_lo = static_cast<size_t>(kv->m_alloc) * c.ffn;
    a.ffn = c.ffn;
  }
  {  // head
    GemmArgs& a = p.g[4];
    set_norm_input(a, kv);
    a.w_tiles = static_cast<const uint8_t*>(m->lm.data);
    a.row_scale = m->lm.row_scale;
    a.logits = logits;
    if (smp) {
      a.inv_temp = smp->inv_temp;
      a.drafts = drafts;
      a.tile_max = kv->tile_max;
      a.tile_sum = kv->tile_sum;
      a.draft_logit = kv->draft_logit;
    } else {
      a.keys = kv->keys;
    }
  }
  {  // attention (every layer; the layer is the phase's)
    AttnArgs& a = p.at;
    const int max_chunks = ceil_div(kv->max_tokens, 128) + 1;
    const int cps = std::max(1, ceil_div(B * c.n_kv * max_chunks, 2 * G));
    const int max_splits = ceil_div(max_chunks, cps);
    if (static_cast<size_t>(B) * c.n_kv * max_splits > kv->attn_items_cap)
      return fail(VSD_ERR_UNSUPPORTED, "attention workspace too small");
    a.batch = B;
    a.batch_cap = kv->max_batch;
    a.n_q = c.n_q;
    a.n_kv = c.n_kv;
    a.hd = c.head_dim;
    a.group = c.n_q / c.n_kv;
    a.rows_valid = kRows * a.group;
    a.chunks_per_split = cps;
    a.max_splits = max_splits;
    a.num_pages = kv->num_pages;
    a.pages_per_req = kv->ppr;
    a.max_tokens = kv->max_tokens;
    a.seq_lens = attn_lens;
    a.page_table = kv->page_table;
    a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c.head_dim)));
    a.part_o = kv->attn_o;
    a.part_ml = kv->attn_ml;
    a.counters = kv->attn_counters;
    a.out = kv->act_o;
    a.out_lo = static_cast<size_t>(kv->m_alloc) * c.n_q * c.head_dim;
    a.q_lo_rows = kv->max_batch * c.n_kv * 128;
    a.status = kv->status;
  }
  p.layers = m->mk_layers;
  p.n_layers = c.layers;
  p.wait_limit = kv->wait_limit;
  p.sync = kv->mk_sync;
  p.part = kv->mk_part;
  p.item_cnt = kv->mk_item_cnt;
  p.status = kv->status;
  // launch ids: one per phase, one more for the kernel's start / end stamps
  p.trace = next_trace(kv);
  if (kv->trace) kv->trace_seq += 5 * c.layers + 1;
  const cudaError_t e = launch_step(c.head_dim, p, G, st);
  if (e != cudaSuccess) return fail(VSD_ERR_CUDA, "step launch: %s", cudaGetErrorString(e));
  return VSD_OK;
}

// The decoder layers of model m as separate launches: per layer the QKV
// GEMM (+ RoPE, block K / V to scratch), attention, O GEMM (+ residual),
// gate/up GEMM (+ SiLU), down GEMM (+ residual); programmatic dependent
// launch lets each kernel's set-up overlap the previous one's tail, and a
// CUDA graph of the step removes the host from the chain.  Attention reads
// attn_lens[b] cached rows per request.
static vsd_status run_layers(const vsd_model* m, vsd_kv* kv, int B, const int* attn_lens, float* hidden,
                             cudaStream_t st, LaunchTimer* timer) {
  const vsd_model_config& c = m->cfg;
  const int M = kRows * B, H = c.hidden;
  vsd_status s;
  const size_t layer_scratch = static_cast<size_t>(kv->max_batch) * c.n_kv * 32 * c.head_dim;
  for (int l = 0; l < c.layers; ++l) {
    GemmArgs a{};
    set_norm_input(a, kv);
    a.q_tile = kv->q_tile;
    a.act_lo_rows = kv->m_alloc;
    a.out_lo = static_cast<size_t>(kv->max_batch) * c.n_kv * 128 * c.head_dim;
    a.k_new = kv->k_new + l * layer_scratch;
    a.v_new = kv->v_new + l * layer_scratch;
    a.ctx_len = kv->ctx_len;
    a.rope = m->rope;
    a.n_q = c.n_q;
    a.n_kv = c.n_kv;
    a.head_dim = c.head_dim;
    TIMED(VSD_K_QKV, if ((s = run_gemm(m, m->qkv[l], EPI_QKV, kv->tm_u, M, a, kv->status, st, next_trace(kv)))) return s);
    TIMED(VSD_K_ATTENTION, if ((s = run_attention(kv, l, B, attn_lens, st, true))) return s);
    GemmArgs r{};
    r.out_f32 = kv->x;
    r.ld_out = H;
    r.x16_out = kv->u;
    r.act_lo_rows = kv->m_alloc;
    r.out_lo = static_cast<size_t>(kv->m_alloc) * H;
    r.ssq_out = kv->ssq;
    r.ssq_ld = kv->m_alloc;
    TIMED(VSD_K_O_PROJ, if ((s = run_gemm(m, m->o[l], EPI_RESID, kv->tm_o, M, r, kv->status, st, next_trace(kv)))) return s);
    GemmArgs g{};
    set_norm_input(g, kv);
    g.act_out = kv->act_a;
    g.act_lo_rows = kv->m_alloc;
    g.out_lo = static_cast<size_t>(kv->m_alloc) * c.ffn;
    g.ffn = c.ffn;
    TIMED(VSD_K_GATE_UP, if ((s = run_gemm(m, m->gu[l], EPI_SILU, kv->tm_u, M, g, kv->status, st, next_trace(kv)))) return s);
    r.hidden_out = hidden ? hidden + static_cast<size_t>(l + 1) * M * H : nullptr;
    TIMED(VSD_K_DOWN, if ((s = run_gemm(m, m->down[l], EPI_RESID, kv->tm_a, M, r, kv->status, st, next_trace(kv)))) return s);
  }
  return VSD_OK;
}

// Final RMSNorm + head as its own launch: per-row argmax keys (kv->keys;
// greedy) or, with `smp`, the per-tile (max, sum) partials and the drafts'
// logits; logits optional.
static vsd_status run_head(const vsd_model* m, vsd_kv* kv, int M, float* logits, cudaStream_t st, LaunchTimer* timer,
                           const int* drafts, const SampleIn* smp) {
  vsd_status s;
  GemmArgs a{};
  set_norm_input(a, kv);
  a.keys = smp ? nullptr : kv->keys;
  a.logits = logits;
  a.act_lo_rows = kv->m_alloc;
  if (smp) {
    a.inv_temp = smp->inv_temp;
    a.drafts = drafts;
    a.tile_max = kv->tile_max;
    a.tile_sum = kv->tile_sum;
    a.draft_logit = kv->draft_logit;
  }
  TIMED(VSD_K_LM_HEAD, if ((s = run_gemm(m, m->lm, smp ? EPI_SAMPLE : EPI_ARGMAX, kv->tm_u, M, a, kv->status, st,
                                         next_trace(kv)))) return s);
  return VSD_OK;
}

// The decoder layers and the head of one step, as the cache's mode says.
static vsd_status run_body(const vsd_model* m, vsd_kv* kv, int B, const int* attn_lens, float* hidden, float* logits,
                           const int* drafts, const SampleIn* smp, cudaStream_t st, LaunchTimer* timer) {
  vsd_status s;
  if (kv->step_kernel == VSD_STEP_PERSISTENT) {
    TIMED(VSD_K_STEP, if ((s = run_persistent(m, kv, B, attn_lens, hidden, logits, drafts, smp, st))) return s);
    return VSD_OK;
  }
  if ((s = run_layers(m, kv, B, attn_lens, hidden, st, timer))) return s;
  return run_head(m, kv, kRows * B, logits, st, timer, drafts, smp);
}

static vsd_status verify_impl(const vsd_model* m, vsd_kv* kv, int B, int* seq_lens, int* pending, const int* drafts,
                              int* accepted, int* out_tokens, float* logits, float* hidden, cudaStream_t st,
                              LaunchTimer* timer = nullptr, const SampleIn* smp = nullptr) {
  if (!m || !kv || !seq_lens || !pending || !drafts || !accepted || !out_tokens)
    return fail(VSD_ERR_ARG, "NULL pointer");
  if (kv->m != m) return fail(VSD_ERR_ARG, "the cache was created for another model");
  if (B < 1 || B > kv->max_batch) return fail(VSD_ERR_ARG, "batch %d outside [1, %d]", B, kv->max_batch);
  const vsd_model_config& c = m->cfg;
  const int M = kRows * B, H = c.hidden;
  vsd_status s;
  {
    EmbedArgs e{};
    e.embed = m->embed;
    e.vocab = c.vocab;
    e.hidden = H;
    e.seq_lens = seq_lens;
    e.pending = pending;
    e.drafts = drafts;
    e.max_tokens = kv->max_tokens;
    e.x = kv->x;
    e.x16 = kv->u;
    e.x16_lo = static_cast<size_t>(kv->m_alloc) * H;
    e.ssq = kv->ssq;
    e.ssq_ld = kv->m_alloc;
    e.ctx_len = kv->ctx_len;
    e.req_ok = kv->req_ok;
    e.keys = kv->keys;
    e.hidden0 = hidden;
    e.status = kv->status;
    e.trace = next_trace(kv);
    TIMED(VSD_K_EMBED, CK(launch_ex(embed_kernel, dim3(M), dim3(128), 0, st, use_pdl(st), false, e)));
  }
  if ((s = run_body(m, kv, B, seq_lens, hidden, logits, drafts, smp, st, timer))) return s;
  if (smp) {
    SampleArgs sa{};
    sa.vocab = c.vocab;
    sa.hidden = H;
    sa.n_tiles = m->lm.n_tiles;
    sa.m_alloc = kv->m_alloc;
    sa.ssq_slices = ceil_div(H, kTileN);
    sa.inv_temp = smp->inv_temp;
    sa.inv_hidden = 1.0f / static_cast<float>(H);
    sa.eps = c.eps;
    sa.tile_max = kv->tile_max;
    sa.tile_sum = kv->tile_sum;
    sa.draft_logit = kv->draft_logit;
    sa.drafts = drafts;
    sa.u_accept = smp->u_accept;
    sa.u_sample = smp->u_sample;
    sa.head = static_cast<const __half*>(m->lm.data);
    sa.head_k_tiles = m->lm.k_tiles;
    sa.x16 = kv->u;
    sa.ssq = kv->ssq;
    sa.decided = kv->decided;
    TIMED(VSD_K_COMMIT, CK(launch_ex(sample_decide_kernel, dim3(B), dim3(256), 0, st, use_pdl(st), false, sa)));
  }
  CommitArgs ca = commit_args(kv, drafts, seq_lens, pending, accepted, out_tokens);
  if (smp) ca.decided = kv->decided;
  ca.x = kv->x;  // the drafter's next conditioning row
  ca.anchor = kv->anchor;
  ca.hidden = H;
  ca.trace = next_trace(kv);
  TIMED(VSD_K_COMMIT, CK(launch_ex(accept_commit_kernel, dim3(B, c.layers), dim3(256), 0, st, use_pdl(st), false, ca)));
  return VSD_OK;
}

// One draft pass: the drafter's layers over rows [anchor_b, mask x 16] at
// positions L_b .. L_b+16 with no cached context (block-causal attention
// among the 17 rows only), then the head; drafts[b][j] = argmax of row 1+j.
// Runs in the target cache's scratch (its staging K/V of layers 0..layers-1
// included), which no other call uses meanwhile on the stream.
static vsd_status draft_impl(const vsd_model* d, vsd_kv* kv, int B, const int* seq_lens, int mask_token,
                             const float* anchor, int* drafts, float* logits, float* hidden, cudaStream_t st,
                             LaunchTimer* timer = nullptr) {
  if (!d || !kv || !seq_lens || !drafts) return fail(VSD_ERR_ARG, "NULL pointer");
  if (B < 1 || B > kv->max_batch) return fail(VSD_ERR_ARG, "batch %d outside [1, %d]", B, kv->max_batch);
  const vsd_model_config& c = d->cfg;
  const vsd_model_config& t = kv->m->cfg;
  if (c.hidden != t.hidden || c.n_q != t.n_q || c.n_kv != t.n_kv || c.head_dim != t.head_dim || c.ffn != t.ffn ||
      c.vocab != t.vocab || c.layers > t.layers || c.attn_fmt != t.attn_fmt || c.mlp_fmt != t.mlp_fmt)
    return fail(VSD_ERR_ARG, "the drafter's shape does not fit the target cache's scratch");
  if (mask_token < 0 || mask_token >= c.vocab) return fail(VSD_ERR_ARG, "mask token %d outside the vocabulary", mask_token);
  const int M = kRows * B, H = c.hidden;
  vsd_status s;
  {
    EmbedArgs e{};
    e.embed = d->embed;
    e.vocab = c.vocab;
    e.hidden = H;
    e.seq_lens = seq_lens;
    e.max_tokens = kv->max_tokens;
    e.x = kv->x;
    e.x16 = kv->u;
    e.x16_lo = static_cast<size_t>(kv->m_alloc) * H;
    e.ssq = kv->ssq;
    e.ssq_ld = kv->m_alloc;
    e.ctx_len = kv->ctx_len;  // positions L_b + j for RoPE
    e.req_ok = kv->req_ok;
    e.keys = kv->keys;
    e.hidden0 = hidden;
    e.anchor = anchor ? anchor : kv->anchor;
    e.mask_token = mask_token;
    e.status = kv->status;
    e.trace = next_trace(kv);
    TIMED(VSD_K_EMBED, CK(launch_ex(embed_kernel, dim3(M), dim3(128), 0, st, use_pdl(st), false, e)));
  }
  if ((s = run_body(d, kv, B, kv->zeros, hidden, logits, nullptr, nullptr, st, timer))) return s;
  TIMED(VSD_K_COMMIT, CK(launch_ex(draft_pick_kernel, dim3(ceil_div(B * kBlock, 128)), dim3(128), 0, st, use_pdl(st),
                                   false, static_cast<const unsigned long long*>(kv->keys), B, c.vocab, drafts,
                                   kv->status)));
  return VSD_OK;
}
#undef TIMED

vsd_status vsd_verify_step_profiled(const vsd_model* m, vsd_kv* kv, int32_t batch, int32_t* seq_lens,
                                    int32_t* pending, const int32_t* drafts, int32_t* accepted,
                                    int32_t* out_tokens, int32_t max_launches, int32_t* kinds, float* ms,
                                    int32_t* n_launches, vsd_stream stream) {
  if (!kinds || !ms || !n_launches || max_launches < 1) return fail(VSD_ERR_ARG, "NULL pointer or no room");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  LaunchTimer t;
  t.st = st;
  vsd_status s = verify_impl(m, kv, batch, seq_lens, pending, drafts, accepted, out_tokens, nullptr, nullptr, st, &t);
  if (s) return s;
  CK(cudaStreamSynchronize(st));
  const int n = std::min<int>(max_launches, static_cast<int>(t.kinds.size()));
  for (int i = 0; i < n; ++i) {
    kinds[i] = t.kinds[i];
    CK(cudaEventElapsedTime(&ms[i], t.ev[2 * i], t.ev[2 * i + 1]));
  }
  *n_launches = static_cast<int>(t.kinds.size());
  return VSD_OK;
}

// The step as one graph launch: its ~5 launches per layer cost more host time
// than the GPU takes for the step.  Captured on a library stream the first
// time these arguments are seen, replayed on the caller's stream after.  Not
// while the caller's stream is itself being captured (its graph then holds
// the launches), nor with phase tracing on, nor with VSD_NO_STEP_GRAPH set.
static bool step_graphs_enabled() {
  static const bool on = getenv("VSD_NO_STEP_GRAPH") == nullptr;
  return on;
}

vsd_status vsd_verify_step(const vsd_model* m, vsd_kv* kv, int32_t batch, int32_t* seq_lens, int32_t* pending,
                           const int32_t* drafts, int32_t* accepted, int32_t* out_tokens, vsd_stream stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (!m || !kv || kv->trace || !step_graphs_enabled() || cudaStreamIsCapturing(st, &cap) != cudaSuccess ||
      cap != cudaStreamCaptureStatusNone)
    return verify_impl(m, kv, batch, seq_lens, pending, drafts, accepted, out_tokens, nullptr, nullptr, st);
  const void* args[5] = {seq_lens, pending, drafts, accepted, out_tokens};
  cudaGraphExec_t exec = nullptr;
  for (auto& g : kv->graphs)
    if (g.model_uid == m->uid && g.batch == batch && std::equal(args, args + 5, g.args)) exec = g.exec;
  if (!exec) {
    if (!kv->capture_stream) CK(cudaStreamCreateWithFlags(&kv->capture_stream, cudaStreamNonBlocking));
    CK(cudaStreamBeginCapture(kv->capture_stream, cudaStreamCaptureModeThreadLocal));
    const vsd_status s = verify_impl(m, kv, batch, seq_lens, pending, drafts, accepted, out_tokens, nullptr, nullptr,
                                     kv->capture_stream);
    cudaGraph_t graph = nullptr;
    const cudaError_t e = cudaStreamEndCapture(kv->capture_stream, &graph);
    if (s) {
      if (graph) cudaGraphDestroy(graph);
      return s;
    }
    if (e != cudaSuccess) return fail(VSD_ERR_CUDA, "step capture: %s", cudaGetErrorString(e));
    const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ei != cudaSuccess) return fail(VSD_ERR_CUDA, "step graph: %s", cudaGetErrorString(ei));
    if (kv->graphs.size() >= 4) {
      cudaGraphExecDestroy(kv->graphs.front().exec);
      kv->graphs.erase(kv->graphs.begin());
    }
    vsd_kv::StepGraph g{m->uid, batch, {}, exec};
    std::copy(args, args + 5, g.args);
    kv->graphs.push_back(g);
  }
  CK(cudaGraphLaunch(exec, st));
  return VSD_OK;
}

// One packed copy each way through library-owned staging: the step's inputs
// go up as one block, its outputs (lengths, pending tokens, accepted counts,
// output rows, laid out contiguously) come back as one block.
vsd_status vsd_verify_step_host(const vsd_model* m, vsd_kv* kv, int32_t batch, int32_t* seq_lens, int32_t* pending,
                                const int32_t* drafts, int32_t* accepted, int32_t* out_tokens, vsd_stream stream) {
  if (!m || !kv || !seq_lens || !pending || !drafts || !accepted || !out_tokens || batch < 1 ||
      batch > kv->max_batch)
    return fail(VSD_ERR_ARG, "bad arguments");
  // every check the step itself makes on the host comes before the input copy is queued
  if (kv->m != m) return fail(VSD_ERR_ARG, "the cache was created for another model");
  const size_t cap = static_cast<size_t>(kv->max_batch) * (kBlock + 3 + kRows);
  if (!kv->io_dev || !kv->io_host) {
    // both staging buffers are published together or not at all
    int* dev = nullptr;
    int* host = nullptr;
    vsd_status s;
    if ((s = dalloc(&dev, cap))) return s;
    if (cudaHostAlloc(reinterpret_cast<void**>(&host), cap * sizeof(int), cudaHostAllocDefault) != cudaSuccess) {
      cudaFree(dev);
      return fail(VSD_ERR_OOM, "pinned staging of %zu bytes", cap * sizeof(int));
    }
    if (kv->io_dev) cudaFree(kv->io_dev);
    if (kv->io_host) cudaFreeHost(kv->io_host);
    kv->io_dev = dev;
    kv->io_host = host;
  }
  // the layout depends on the batch; the step graph is keyed by the pointers, so each batch size gets its own
  const size_t B = static_cast<size_t>(batch);
  int* h = kv->io_host;
  int* d = kv->io_dev;
  memcpy(h, drafts, B * kBlock * sizeof(int));
  memcpy(h + B * kBlock, seq_lens, B * sizeof(int));
  memcpy(h + B * (kBlock + 1), pending, B * sizeof(int));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t n_in = B * (kBlock + 2), n_out = B * (3 + kRows);
  CK(cudaMemcpyAsync(d, h, n_in * sizeof(int), cudaMemcpyHostToDevice, st));
  const vsd_status s = vsd_verify_step(m, kv, batch, d + B * kBlock, d + B * (kBlock + 1), d, d + B * (kBlock + 2),
                                       d + B * (kBlock + 3), stream);
  if (s) {
    // the queued copy still reads the pinned staging: let it finish before
    // the next call may overwrite it (the step's own error message stands)
    cudaStreamSynchronize(st);
    return s;
  }
  CK(cudaMemcpyAsync(h + B * kBlock, d + B * kBlock, n_out * sizeof(int), cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  memcpy(seq_lens, h + B * kBlock, B * sizeof(int));
  memcpy(pending, h + B * (kBlock + 1), B * sizeof(int));
  memcpy(accepted, h + B * (kBlock + 2), B * sizeof(int));
  memcpy(out_tokens, h + B * (kBlock + 3), B * kRows * sizeof(int));
  return VSD_OK;
}

vsd_status vsd_verify_step_debug(const vsd_model* m, vsd_kv* kv, int32_t batch, int32_t* seq_lens, int32_t* pending,
                                 const int32_t* drafts, int32_t* accepted, int32_t* out_tokens, float* logits,
                                 float* hidden, vsd_stream stream) {
  return verify_impl(m, kv, batch, seq_lens, pending, drafts, accepted, out_tokens, logits, hidden,
                     reinterpret_cast<cudaStream_t>(stream));
}

vsd_status vsd_verify_step_sampled(const vsd_model* m, vsd_kv* kv, int32_t batch, int32_t* seq_lens, int32_t* pending,
                                   const int32_t* drafts, int32_t* accepted, int32_t* out_tokens,
                                   const float* u_accept, const float* u_sample, float temperature, float* logits,
                                   vsd_stream stream) {
  if (!u_accept || !u_sample) return fail(VSD_ERR_ARG, "NULL pointer");
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return fail(VSD_ERR_ARG, "temperature must be > 0");
  if (m && m->lm.fmt != VSD_FMT_BF16) return fail(VSD_ERR_UNSUPPORTED, "sampling needs a 16-bit head");
  if (m && (m->cfg.hidden % 16)) return fail(VSD_ERR_UNSUPPORTED, "sampling needs hidden %% 16 == 0");
  SampleIn smp{1.0f / temperature, u_accept, u_sample};
  return verify_impl(m, kv, batch, seq_lens, pending, drafts, accepted, out_tokens, logits, nullptr,
                     reinterpret_cast<cudaStream_t>(stream), nullptr, &smp);
}

vsd_status vsd_draft_step(const vsd_model* drafter, vsd_kv* kv, int32_t batch, const int32_t* seq_lens,
                          int32_t mask_token, int32_t* drafts, vsd_stream stream) {
  return draft_impl(drafter, kv, batch, seq_lens, mask_token, nullptr, drafts, nullptr, nullptr,
                    reinterpret_cast<cudaStream_t>(stream));
}

vsd_status vsd_draft_step_debug(const vsd_model* drafter, vsd_kv* kv, int32_t batch, const int32_t* seq_lens,
                                int32_t mask_token, const float* anchor, int32_t* drafts, float* logits,
                                float* hidden, vsd_stream stream) {
  return draft_impl(drafter, kv, batch, seq_lens, mask_token, anchor, drafts, logits, hidden,
                    reinterpret_cast<cudaStream_t>(stream));
}

vsd_status vsd_spec_loop(const vsd_model* target, const vsd_model* drafter, vsd_kv* kv, int32_t slots,
                         int32_t queued, const int32_t* req_len, const int32_t* req_pending,
                         const int32_t* req_budget, const float* req_anchor, int32_t* slot_req, int32_t* next_req,
                         int32_t* iter, int32_t* req_generated, int32_t* req_admit_iter, int32_t* req_out,
                         int32_t out_cap, int32_t n_iters, int32_t mask_token, vsd_stream stream) {
  if (!target || !drafter || !kv || !req_len || !req_pending || !req_budget || !req_anchor || !slot_req ||
      !next_req || !iter || !req_generated || !req_admit_iter || !req_out)
    return fail(VSD_ERR_ARG, "NULL pointer");
  if (kv->m != target) return fail(VSD_ERR_ARG, "the cache was created for another model");
  if (slots < 1 || slots > kMaxLoopSlots || queued < 0 || out_cap < 1 || n_iters < 0)
    return fail(VSD_ERR_ARG, "slots in [1, %d], queued >= 0, out_cap >= 1, n_iters >= 0", kMaxLoopSlots);
  if (static_cast<int64_t>(slots) + queued > kv->max_batch)
    return fail(VSD_ERR_ARG, "%d slots + %d queued requests exceed the cache's %d", slots, queued, kv->max_batch);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  LoopArgs la{};
  la.B = slots;
  la.Q = queued;
  la.out_cap = out_cap;
  la.hidden = target->cfg.hidden;
  la.pages_per_req = kv->ppr;
  la.first_queued = slots;
  la.slot_req = slot_req;
  la.next_req = next_req;
  la.req_len = req_len;
  la.req_pending = req_pending;
  la.req_budget = req_budget;
  la.req_anchor = req_anchor;
  la.req_generated = req_generated;
  la.req_admit_iter = req_admit_iter;
  la.req_out = req_out;
  la.seq_lens = kv->loop_seq;
  la.pending = kv->loop_pend;
  la.accepted = kv->loop_acc;
  la.out_tokens = kv->loop_out;
  la.page_table = kv->page_table;
  la.anchor = kv->anchor;
  la.iter = iter;
  la.status = kv->status;
  vsd_status s;
  for (int i = 0; i < n_iters; ++i) {
    CK(launch_ex(loop_schedule_kernel, dim3(1), dim3(256), 0, st, use_pdl(st), false, la));
    if ((s = draft_impl(drafter, kv, slots, kv->loop_seq, mask_token, nullptr, kv->loop_drafts, nullptr, nullptr, st)))
      return s;
    if ((s = verify_impl(target, kv, slots, kv->loop_seq, kv->loop_pend, kv->loop_drafts, kv->loop_acc, kv->loop_out,
                         nullptr, nullptr, st)))
      return s;
    CK(launch_ex(loop_collect_kernel, dim3(slots), dim3(32), 0, st, use_pdl(st), false, la));
  }
  return VSD_OK;
}

vsd_status vsd_kv_get_anchor(const vsd_kv* kv, int32_t batch, float* dst, vsd_stream stream) {
  if (!kv || !dst) return fail(VSD_ERR_ARG, "NULL pointer");
  if (batch < 1 || batch > kv->max_batch) return fail(VSD_ERR_ARG, "batch %d outside [1, %d]", batch, kv->max_batch);
  CK(cudaMemcpyAsync(dst, kv->anchor, static_cast<size_t>(batch) * kv->m->cfg.hidden * sizeof(float),
                     cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)));
  return VSD_OK;
}

// ------------------------------------------------------------------ components
vsd_status vsd_linear(const vsd_weight* w, int32_t n, int32_t k, const uint16_t* x, int32_t mtok, float* y,
                      vsd_stream stream) {
  if (!w || !x || !y) return fail(VSD_ERR_ARG, "NULL pointer");
  if (n < 1 || k < 8 || mtok < 1 || (k % 8)) return fail(VSD_ERR_ARG, "need n >= 1, m >= 1 and k a multiple of 8");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Linear L;
  vsd_status s = build_linear(&w, &n, 1, k, identity_perm(n), st, &L);
  if (s) return s;
  CUtensorMap tm[kActBoxes]{};
  for (int j = 0; j < kActBoxes; ++j) {
    if ((s = tmap_2d(&tm[j], x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, k, mtok, 64, 16u * (j + 1)))) {
      free_linear(L);
      return s;
    }
  }
  int* status = nullptr;
  if ((s = dalloc(&status, 1))) {
    free_linear(L);
    return s;
  }
  vsd_model mm;
  mm.sms = sm_count();
  for (int i = 0; i < 4; ++i) mm.max_clusters[i] = gemm_max_clusters(1 << i);
  GemmArgs a{};
  a.out_f32 = y;
  a.ld_out = n;
  s = run_gemm(&mm, L, EPI_STORE, tm, mtok, a, status, st);
  cudaStreamSynchronize(st);
  cudaFree(status);
  free_linear(L);
  return s;
}

vsd_status vsd_block_attention(const vsd_model* m, vsd_kv* kv, int32_t layer, int32_t B, const int32_t* seq_lens,
                               const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new, uint16_t* out,
                               vsd_stream stream) {
  if (!m || !kv || !seq_lens || !q || !k_new || !v_new || !out) return fail(VSD_ERR_ARG, "NULL pointer");
  if (kv->m != m) return fail(VSD_ERR_ARG, "the cache was created for another model");
  const vsd_model_config& c = m->cfg;
  if (B < 1 || B > kv->max_batch || layer < 0 || layer >= c.layers) return fail(VSD_ERR_ARG, "batch or layer out of range");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  scatter_q_kernel<<<256, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(q), B, c.n_q, c.n_kv, c.head_dim,
                                        kv->q_tile);
  scatter_block_rows_kernel<<<256, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(k_new), 1, B, c.n_kv,
                                                 c.head_dim, kv->max_batch, layer, kv->k_new);
  scatter_block_rows_kernel<<<256, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(v_new), 1, B, c.n_kv,
                                                 c.head_dim, kv->max_batch, layer, kv->v_new);
  CK(cudaGetLastError());
  vsd_status s = run_attention(kv, layer, B, seq_lens, st, false);
  if (s) return s;
  CK(cudaMemcpyAsync(out, kv->act_o, static_cast<size_t>(B) * kRows * c.n_q * c.head_dim * 2,
                     cudaMemcpyDeviceToDevice, st));
  return VSD_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ attention without allocation
// Scratch memory of vsd_block_attention_static: one fixed array in every
// device's copy of this library's module, present from load until the
// process exits, shared by all calls on that device.  Host code must not
// hand `g_static_scratch` itself to a kernel (on the host it names a
// stand-in, not device memory); it uses the device address looked up below.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(16) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device, looked up with
// cudaGetSymbolAddress on the first call per device (no allocation).
vsd_status static_scratch_address(void** out) {
  int dev = -1;
  CK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return fail(VSD_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return fail(VSD_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s", cudaGetErrorString(e));
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return VSD_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

extern "C" {

vsd_status vsd_block_attention_static(const vsd_model* m, vsd_kv* kv, int32_t layer, int32_t B,
                                      const int32_t* seq_lens, const uint16_t* q, const uint16_t* k_new,
                                      const uint16_t* v_new, uint16_t* out, vsd_stream stream) {
  if (!m || !kv || !seq_lens || !q || !k_new || !v_new || !out) return fail(VSD_ERR_ARG, "NULL pointer");
  if (kv->m != m) return fail(VSD_ERR_ARG, "the cache was created for another model");
  const vsd_model_config& c = m->cfg;
  if (B < 1 || B > kv->max_batch || layer < 0 || layer >= c.layers) return fail(VSD_ERR_ARG, "batch or layer out of range");
  if (B > kMaxReqs) return fail(VSD_ERR_UNSUPPORTED, "at most %d requests per call", kMaxReqs);
  const int hd = c.head_dim;
  const size_t pairs = static_cast<size_t>(B) * c.n_kv;
  // scratch layout: split counters | q tiles | block K rows | block V rows | split partials (O, then m / l)
  const size_t o_cnt = 0;
  const size_t o_q = align256(o_cnt + 2 * pairs * sizeof(int));  // arrived / done counters per pair
  const size_t o_k = align256(o_q + pairs * 128 * hd * 2);
  const size_t o_v = align256(o_k + pairs * 32 * hd * 2);
  const size_t o_part = align256(o_v + pairs * 32 * hd * 2);
  const size_t per_split = align256(pairs * 128 * hd * 4) + align256(pairs * 128 * 2 * 4);
  const int max_chunks = ceil_div(kv->max_tokens, 128) + 1;
  // same work split as the step's attention, coarsened until the partials fit
  int cps = std::max(1, ceil_div(B * c.n_kv * max_chunks, 2 * m->sms));
  while (o_part + static_cast<size_t>(ceil_div(max_chunks, cps)) * per_split > kStaticScratchBytes && cps < max_chunks)
    ++cps;
  const int max_splits = ceil_div(max_chunks, cps);
  const size_t need = o_part + static_cast<size_t>(max_splits) * per_split;
  if (need > kStaticScratchBytes)
    return fail(VSD_ERR_UNSUPPORTED,
                "%d requests x %d KV heads x head_dim %d need %zu bytes of scratch; the static array holds %zu",
                B, c.n_kv, hd, need, kStaticScratchBytes);
  void* base_v = nullptr;
  vsd_status s = static_scratch_address(&base_v);
  if (s) return s;
  uint8_t* base = static_cast<uint8_t*>(base_v);
  auto* q_tile = reinterpret_cast<__nv_bfloat16*>(base + o_q);
  auto* k_stage = reinterpret_cast<__nv_bfloat16*>(base + o_k);
  auto* v_stage = reinterpret_cast<__nv_bfloat16*>(base + o_v);
  float* part_o = reinterpret_cast<float*>(base + o_part);
  float* part_ml = reinterpret_cast<float*>(base + o_part + static_cast<size_t>(max_splits) * align256(pairs * 128 * hd * 4));
  // tensor maps: the layer's slice of the cache pool (so the kernel's layer index is 0), the staged tiles
  const auto BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const size_t layer_rows = static_cast<size_t>(kv->num_pages) * c.n_kv * kPage;
  CUtensorMap tm_q, tm_kc, tm_vc, tm_kn, tm_vn;
  if ((s = tmap_2d(&tm_q, q_tile, BF16, hd, pairs * 128, 64, 128)) ||
      (s = tmap_2d(&tm_kc, kv->k_pool + layer * layer_rows * hd, BF16, hd, layer_rows, 64, 16)) ||
      (s = tmap_2d(&tm_vc, kv->v_pool + layer * layer_rows * hd, BF16, hd, layer_rows, 64, 16)) ||
      (s = tmap_2d(&tm_kn, k_stage, BF16, hd, pairs * 32, 64, 32)) ||
      (s = tmap_2d(&tm_vn, v_stage, BF16, hd, pairs * 32, 64, 32)))
    return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // what must start at zero: the split counters, and the staged block rows
  // 17..31 of every 32-row group (loaded with the block, masked by the kernel)
  CK(cudaMemsetAsync(base + o_cnt, 0, 2 * pairs * sizeof(int), st));
  CK(cudaMemsetAsync(base + o_k, 0, o_part - o_k, st));
  scatter_q_kernel<<<256, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(q), B, c.n_q, c.n_kv, hd, q_tile);
  scatter_block_rows_kernel<<<256, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(k_new), 1, B, c.n_kv, hd, B,
                                                 0, k_stage);
  scatter_block_rows_kernel<<<256, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(v_new), 1, B, c.n_kv, hd, B,
                                                 0, v_stage);
  CK(cudaGetLastError());
  AttnArgs a{};
  a.batch = B;
  a.batch_cap = B;
  a.n_q = c.n_q;
  a.n_kv = c.n_kv;
  a.hd = hd;
  a.group = c.n_q / c.n_kv;
  a.rows_valid = kRows * a.group;
  a.chunks_per_split = cps;
  a.max_splits = max_splits;
  a.layer = 0;
  a.num_pages = kv->num_pages;
  a.pages_per_req = kv->ppr;
  a.max_tokens = kv->max_tokens;
  a.seq_lens = seq_lens;
  a.page_table = kv->page_table;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(hd)));
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.counters = reinterpret_cast<int*>(base + o_cnt);
  a.out = reinterpret_cast<__half*>(out);
  a.status = kv->status;
  const int grid = std::min(static_cast<int>(pairs) * max_splits, m->sms);
  const cudaError_t e = launch_attn(hd, tm_q, tm_kc, tm_vc, tm_kn, tm_vn, a, dim3(grid), st, false);
  if (e != cudaSuccess) return fail(VSD_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  return VSD_OK;
}

vsd_status vsd_accept_commit(const vsd_model* m, vsd_kv* kv, int32_t B, const float* logits, const uint16_t* k_new,
                             const uint16_t* v_new, int32_t* seq_lens, int32_t* pending, const int32_t* drafts,
                             int32_t* accepted, int32_t* out_tokens, vsd_stream stream) {
  if (!m || !kv || !logits || !k_new || !v_new || !seq_lens || !pending || !drafts || !accepted || !out_tokens)
    return fail(VSD_ERR_ARG, "NULL pointer");
  if (kv->m != m) return fail(VSD_ERR_ARG, "the cache was created for another model");
  const vsd_model_config& c = m->cfg;
  if (B < 1 || B > kv->max_batch) return fail(VSD_ERR_ARG, "batch out of range");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  scatter_block_rows_kernel<<<512, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(k_new), c.layers, B, c.n_kv,
                                                 c.head_dim, kv->max_batch, 0, kv->k_new);
  scatter_block_rows_kernel<<<512, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(v_new), c.layers, B, c.n_kv,
                                                 c.head_dim, kv->max_batch, 0, kv->v_new);
  logits_argmax_kernel<<<B * kRows, 256, 0, st>>>(logits, c.vocab, kv->keys);
  CK(cudaGetLastError());
  validate_requests_kernel<<<ceil_div(B, 128), 128, 0, st>>>(seq_lens, pending, B, c.vocab, kv->max_tokens,
                                                            kv->ctx_len, kv->req_ok, kv->status);
  CommitArgs ca = commit_args(kv, drafts, seq_lens, pending, accepted, out_tokens);
  CK(launch_ex(accept_commit_kernel, dim3(B, c.layers), dim3(256), 0, st, false, false, ca));
  return VSD_OK;
}

}  // extern "C"
