/*
 * vsd.h -- C ABI of the GB300 greedy block-verify library.
 *
 * One call, vsd_verify_step, runs the target-model verification step of
 * block speculative decoding on the GPU: for every request, the pending token
 * and a block of 16 drafted tokens pass through the decoder-only target in
 * one forward over the request's KV cache (causal inside the block); the
 * greedy token of every row is compared with the drafts; the longest
 * matching prefix plus one target token is accepted; only the accepted rows'
 * K and V are committed to the cache.
 *
 * Where the method is defined:
 *   - one target pass verifies a whole drafted block: "The Inference Stack
 *     Behind OCRia", section "Generate more tokens per target pass:
 *     speculative decoding"; HunyuanOCR-1.5 summary, section one, inference
 *     steps 2-3 (block size B = 16);
 *   - accept the longest valid prefix, cutting at the first mismatch from the
 *     left, then append the target's own token (correction or bonus):
 *     HunyuanOCR-1.5 summary, section one, inference step 4; the accept /
 *     correct / bonus branch of the speculative decoder in "LLM inference
 *     acceleration", section 3.2;
 *   - the output equals the target's own greedy output: OCRia post,
 *     speculative-decoding section ("100% lossless");
 *   - BF16 / FP8 / NVFP4 weights: OCRia post, section "Reducing the data
 *     moved: workload-aware quantization";
 *   - KV cache (no recomputation of earlier tokens), GQA, paged KV:
 *     OCRia post, speculative-decoding section; "LLM inference
 *     acceleration", section two;
 *   - per-step batch metadata (sequence lengths, cache locations) kept where
 *     the kernels read it, no host round trip per step: OCRia post, section
 *     "Fixing CPU-side preparation".
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are CUDA device pointers; *_host are host memory.
 *     The caller owns every pointer it passes; the library owns what it
 *     allocates inside vsd_model / vsd_kv and frees it in *_destroy.
 *   - Work is enqueued on the given stream and is asynchronous unless the
 *     comment says the call synchronises.  vsd_verify_step never synchronises
 *     and never copies to the host, so it can be captured in a CUDA graph.
 *   - Errors the host can see (null pointers, sizes out of range, a missing
 *     CUDA device) return a nonzero vsd_status before anything is enqueued;
 *     vsd_last_error() then describes it (per thread).  Errors only the
 *     device can see (a token id >= vocab, a sequence length beyond the
 *     cache, a page id outside the pool, a bounded wait that ran out) set a
 *     bit in the cache's device status word (vsd_get_device_status); an
 *     affected request is left unchanged (no commit, accepted = -1).  A
 *     page outside the pool anywhere in a request's rows [0, L + 17)
 *     rejects that request; a wait that ran out (VSD_DEV_TIMEOUT, sticky
 *     until the status word is read) rejects every request of the step.
 *   - Token ids, lengths and counts are int32.  BF16 is raw 16-bit storage
 *     (uint16_t bit patterns); FP8 is E4M3 ("fn": max 448, no infinities);
 *     FP4 is E2M1, two per byte with the even element in the low nibble.
 */
#ifndef VSD_H
#define VSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* vsd_stream; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  VSD_OK = 0,
  VSD_ERR_ARG = 1,        /* bad pointer / size / enum */
  VSD_ERR_CUDA = 2,       /* a CUDA runtime call failed */
  VSD_ERR_OOM = 3,        /* device allocation failed */
  VSD_ERR_CAPACITY = 4,   /* request does not fit the cache that was created */
  VSD_ERR_DEVICE = 5,     /* the device status word has bits set */
  VSD_ERR_UNSUPPORTED = 6 /* shape the kernels do not cover */
} vsd_status;

/* Bits of the device status word. */
#define VSD_DEV_BAD_TOKEN   0x1  /* token id outside [0, vocab) */
#define VSD_DEV_BAD_SEQLEN  0x2  /* seq_len < 0 or seq_len + 17 > max_tokens_per_req */
#define VSD_DEV_BAD_PAGE    0x4  /* page-table entry outside [0, num_pages) */
#define VSD_DEV_TIMEOUT     0x8  /* a bounded device-side wait ran out */

typedef enum { VSD_FMT_BF16 = 0, VSD_FMT_FP8 = 1, VSD_FMT_NVFP4 = 2 } vsd_weight_format;

/* Decoder-only target: pre-norm layers, RMSNorm (weight 1), rotate-half
 * RoPE, GQA attention (query head h reads KV head h / (n_q / n_kv)), SwiGLU
 * MLP, final RMSNorm, lm_head (tied to the embedding or separate). */
typedef struct {
  int32_t layers, hidden, n_q, n_kv, head_dim, ffn, vocab;
  float rope_theta;
  float eps;
  int32_t tied;          /* 1: lm_head is the embedding matrix */
  int32_t attn_fmt;      /* vsd_weight_format of wq, wk, wv, wo */
  int32_t mlp_fmt;       /* vsd_weight_format of wg, wu, wd */
  int32_t max_positions; /* length of the RoPE table; positions must stay below it */
} vsd_model_config;

/* One weight matrix W [N, K] (y = x W^T) in canonical form, device memory:
 *   BF16 : data = uint16 [N, K] row-major; scale unused
 *   FP8  : data = e4m3 [N, K] row-major; scale = float [N], w = e4m3 * scale[n]
 *   NVFP4: data = packed e2m1 [N, K/2]; scale = e4m3 [N, K/16] (one per 16
 *          consecutive k of a row); tensor_scale = float [1];
 *          w = e2m1 * e4m3(scale) * tensor_scale
 * (the quantised forms are what vsd_quantize_* write). */
typedef struct {
  int32_t fmt;
  const void* data_dev;
  const void* scale_dev;
  const float* tensor_scale_dev;
} vsd_weight;

/* All weights.  layers points to layers*7 entries, per layer in the order
 * wq [n_q*hd, H], wk [n_kv*hd, H], wv [n_kv*hd, H], wo [H, n_q*hd],
 * wg [F, H], wu [F, H], wd [H, F]. */
typedef struct {
  const uint16_t* embed_dev;   /* BF16 [vocab, hidden] */
  const uint16_t* lm_head_dev; /* BF16 [vocab, hidden], or NULL when tied */
  const vsd_weight* layers;    /* host array of layers*7 entries */
} vsd_weights;

typedef struct vsd_model vsd_model;
typedef struct vsd_kv vsd_kv;

/* Library build string, e.g. "vsd 0.1 sm_103a". */
const char* vsd_version(void);
/* Description of the last error returned on this thread ("" if none). */
const char* vsd_last_error(void);

/* ---------------------------------------------------------------- quantisers
 * Round-to-nearest (ties to even, saturating) quantisation of a BF16 matrix,
 * the weight recipe of "The Inference Stack Behind OCRia", section "Reducing
 * the data moved" (BF16 master -> FP8 / NVFP4; the pages' calibration set is
 * replaced by plain rounding).  Scale arithmetic is float32, one rounding per
 * operation:
 *   FP8  : s[n] = amax_row / 448;  q = e4m3(w / s[n]);  s == 0 -> q = 0
 *   NVFP4: S = amax / 2688;  s_blk = e4m3(amax_blk / (6 S));
 *          q = e2m1(w / (e4m3(s_blk) * S));  a zero scale -> q = 0
 * w_dev BF16 [N, K] row-major; outputs as in vsd_weight.  NVFP4 needs
 * K % 16 == 0.  Asynchronous on the stream; no allocation. */
vsd_status vsd_quantize_fp8_rowwise(const uint16_t* w_dev, int32_t n, int32_t k,
                                    uint8_t* q_dev, float* scale_dev, vsd_stream stream);
vsd_status vsd_quantize_nvfp4(const uint16_t* w_dev, int32_t n, int32_t k,
                              uint8_t* q_dev, uint8_t* block_scale_dev,
                              float* tensor_scale_dev, vsd_stream stream);

/* ---------------------------------------------------------------- model
 * Repacks the caller's canonical weights into the kernels' tile layout
 * (library-owned copies) and builds the RoPE table.  Synchronises the stream
 * before returning; the caller's buffers may be freed afterwards. */
vsd_status vsd_model_create(const vsd_model_config* cfg, const vsd_weights* w,
                            vsd_stream stream, vsd_model** out);
void vsd_model_destroy(vsd_model* m);

/* ---------------------------------------------------------------- KV cache
 * Paged BF16 KV cache for up to max_batch requests (request slot b = row b
 * of every per-request array), each holding up to max_tokens_per_req tokens
 * including the 17 rows of an in-flight block.  page_size must be 16.
 * num_pages = 0 gives max_batch * ceil(max_tokens_per_req / 16) pages.  The
 * page table starts as the identity (slot b, page i -> b * pages_per_req + i).
 * Also owns the step's device workspace.  Synchronises. */
vsd_status vsd_kv_create(const vsd_model* m, int32_t max_batch, int32_t max_tokens_per_req,
                         int32_t page_size, int32_t num_pages, vsd_kv** out);
void vsd_kv_destroy(vsd_kv* kv);
int32_t vsd_kv_pages_per_req(const vsd_kv* kv);
int32_t vsd_kv_num_pages(const vsd_kv* kv);

/* Replaces the page table: table_dev int32 [max_batch, pages_per_req], every
 * entry in [0, num_pages) (checked on the device; a bad entry sets
 * VSD_DEV_BAD_PAGE).  Pages of one request must be distinct and not shared. */
vsd_status vsd_kv_set_page_table(vsd_kv* kv, const int32_t* table_dev, vsd_stream stream);

/* Writes (read) cache rows [start, start+count) of request slot req, all
 * layers: k_dev / v_dev BF16 [layers, count, n_kv, head_dim].  Asynchronous. */
vsd_status vsd_kv_write(vsd_kv* kv, int32_t req, int32_t start, int32_t count,
                        const uint16_t* k_dev, const uint16_t* v_dev, vsd_stream stream);
vsd_status vsd_kv_read(const vsd_kv* kv, int32_t req, int32_t start, int32_t count,
                       uint16_t* k_dev, uint16_t* v_dev, vsd_stream stream);

/* Phase tracing for profiling.  With max_launches > 0, the kernels of later
 * steps store globaltimer (ns) at their phase boundaries into a library-owned
 * table [launch][CTA < 1024][tag < 64] (0 = not reached); 0 turns tracing
 * off.  Launch ids count kernel launches in order from 0 after each read.
 * vsd_trace_read copies the table rows of up to max_launches launches to
 * slots_host (max_launches * 1024 * 64 words), clears the table, restarts the
 * launch ids and returns the number of table rows copied; it synchronises
 * the stream.  A step captured in a CUDA graph keeps the launch ids it was
 * captured with. */
vsd_status vsd_trace_enable(vsd_kv* kv, int32_t max_launches);
vsd_status vsd_trace_read(vsd_kv* kv, uint64_t* slots_host, int32_t max_launches, int32_t* n_launches,
                          vsd_stream stream);

/* Reads and clears the device status word (VSD_DEV_* bits).  Synchronises
 * the stream. */
vsd_status vsd_get_device_status(vsd_kv* kv, vsd_stream stream, int32_t* status_host);

/* How a step launches the decoder layers and the head (per cache; the
 * default is VSD_STEP_LAYERED):
 *   VSD_STEP_LAYERED     one launch per GEMM and per attention of every
 *                        layer, then the head (5 * layers + 1 launches,
 *                        chained with programmatic dependent launch);
 *   VSD_STEP_PERSISTENT  one cooperative launch of a persistent kernel (one
 *                        CTA per SM) that runs the same phases in order,
 *                        separated by grid-wide counters with bounded waits.
 * Both compute the same step (same kernels' arithmetic, the same results up
 * to the order of floating-point sums).  Changing the mode drops the step
 * graphs the cache holds.  VSD_ERR_ARG for a NULL cache or an unknown mode. */
#define VSD_STEP_LAYERED    0
#define VSD_STEP_PERSISTENT 1
vsd_status vsd_kv_set_step_kernel(vsd_kv* kv, int32_t mode);

/* ------------------------------------------------------ ReplaySSM rollback
 * A recurrent (gated delta rule) layer's state under block speculative
 * decoding, kept the ReplaySSM way ("The Inference Stack Behind OCRia",
 * section "Make speculative verification cheaper"): per request and head a
 * checkpoint S (d x d fp32) plus a buffer of up to `window` recent tokens;
 * outputs come from the checkpoint and the buffered tokens; rejected drafts
 * are dropped by moving the buffer pointer; the checkpoint is rewritten only
 * at flushes.  The pages give no update rule; the gated delta rule is used,
 * per token
 *     S <- alpha S (I - beta k k^T) + beta v k^T,   o = S q.
 * The buffer holds per token its key, its corrected value
 * u = beta (v - alpha S_prev k) and the sum of log alpha since the
 * checkpoint, so that S = e^{L} S_ckpt + sum_s e^{L - L_s} u_s k_s^T in
 * closed form (log alpha is floored at -200, where e^{L} underflows).
 * The checkpoint and the retained keys are kept as f16 hi / lo pairs with a
 * power-of-2 scale per row (about 22 significant bits of each row's
 * largest value), the form the tensor cores read.
 * The library owns every state buffer; d is 64 or 128, 17 <= window <= 128
 * for d = 64 and <= 64 for d = 128 (VSD_ERR_UNSUPPORTED above: shared
 * memory).
 * Errors as elsewhere: host-visible ones return before any launch; a commit
 * count outside [-1, 16] (its block is then rejected) or a corrupted pointer
 * sets VSD_DEV_BAD_SEQLEN in the object's own status word. */
typedef struct vsd_ssm vsd_ssm;
vsd_status vsd_ssm_create(int32_t max_batch, int32_t heads, int32_t d, int32_t window, vsd_ssm** out);
void vsd_ssm_destroy(vsd_ssm* ssm);
/* Request req's state := state_dev ([heads][d][d] fp32, device; row-major
 * S[i][j] multiplies k[j]), with an empty buffer.  Asynchronous. */
vsd_status vsd_ssm_set_state(vsd_ssm* ssm, int32_t req, const float* state_dev, vsd_stream stream);
/* Request req's effective state (the checkpoint replayed through the
 * retained buffer) into state_dev ([heads][d][d], device).  Asynchronous. */
vsd_status vsd_ssm_get_state(vsd_ssm* ssm, int32_t req, float* state_dev, vsd_stream stream);
/* One verify block for requests 0..B-1: inputs q, k, v [B][heads][17][d]
 * and alpha, beta [B][heads][17] (device, fp32; k is used as given, the
 * caller normalises it); out [B][heads][17][d] receives o for each row, the
 * state after the retained buffer and rows 0..t applied to q_t.  The block's
 * tokens are staged in the buffer after the pointer.  q, k, v and out must be
 * 16-byte aligned (VSD_ERR_ARG otherwise).  Asynchronous. */
vsd_status vsd_ssm_verify(vsd_ssm* ssm, int32_t batch, const float* q, const float* k, const float* v,
                          const float* alpha, const float* beta, float* out, vsd_stream stream);
/* Commit of the last verify block: accepted_dev[B] (device int32) holds each
 * request's accepted drafts a (rows 0..a stay in the buffer; -1 keeps none,
 * as for a request the step rejected).  A request whose next block would
 * not fit (pointer + 17 > window) folds its buffer into the checkpoint.
 * Asynchronous. */
vsd_status vsd_ssm_commit(vsd_ssm* ssm, int32_t batch, const int32_t* accepted_dev, vsd_stream stream);
/* Reads and clears the object's device status word.  Synchronises. */
vsd_status vsd_ssm_get_device_status(vsd_ssm* ssm, vsd_stream stream, int32_t* status_host);

/* Test-only; the method has no counterpart.  Enqueues one CTA that waits,
 * with the same bounded-wait pattern as the step's kernels, on a device flag
 * that nothing sets and on a shared-memory mbarrier that nothing completes.
 * Each wait gives up after limit_cycles SM cycles (1 .. 2e9), sets
 * VSD_DEV_TIMEOUT in kv's device status word and the kernel returns; the
 * context stays usable.  Returns VSD_ERR_ARG for a NULL cache or a limit out
 * of range.  Asynchronous. */
vsd_status vsd_debug_wait_probe(vsd_kv* kv, int64_t limit_cycles, vsd_stream stream);

/* ---------------------------------------------------------------- the step
 * Greedy block verification of B requests (slots 0..B-1), 1 <= B <= max_batch.
 *   seq_lens_dev   int32 [B] in/out: committed length L_b; += accepted+1
 *   pending_dev    int32 [B] in/out: last emitted token (its K/V not yet
 *                  cached); becomes the target's token after the accepted
 *                  prefix (correction or bonus)
 *   drafts_dev     int32 [B, 16]: drafted tokens
 *   accepted_dev   int32 [B] out: a_b in 0..16 = index of the first draft
 *                  that differs from the target's greedy token (16 if none)
 *   out_tokens_dev int32 [B, 17] out: the target's greedy tokens g_0..g_a,
 *                  -1 beyond (g_i = d_i for i < a)
 * Rows [pending, d_0..d_15] run at positions L_b..L_b+16.  Rows 0..a_b (the
 * pending token and the accepted drafts) have their K (after RoPE) and V
 * committed at positions L_b..L_b+a_b; no other cache row changes.  argmax
 * ties go to the lowest token id.  Needs L_b + 17 <= max_tokens_per_req.
 * The step's kernel launches (about five per layer) are recorded once into a CUDA graph for
 * each new (model, batch, five device pointers) combination (up to four kept
 * per cache, oldest replaced; the first call of a combination captures on a
 * library-owned stream, costing some milliseconds) and replayed on `stream`
 * afterwards, so reuse the same device buffers across steps.  Launches go
 * straight to `stream` instead while that stream is itself being captured,
 * while phase tracing is on, or when the environment sets VSD_NO_STEP_GRAPH. */
vsd_status vsd_verify_step(const vsd_model* m, vsd_kv* kv, int32_t batch,
                           int32_t* seq_lens_dev, int32_t* pending_dev,
                           const int32_t* drafts_dev, int32_t* accepted_dev,
                           int32_t* out_tokens_dev, vsd_stream stream);

/* The same step for a caller holding its state in host memory (any host
 * buffers, pageable or pinned; same shapes and meanings as above).  The
 * inputs travel to the device as one copy through library-owned staging
 * (device and pinned host, max_batch * 36 words each, allocated on the first
 * call and freed with the cache), the step runs as above (the staging
 * addresses are fixed, so its graph is reused), and lengths, pending tokens,
 * accepted counts and output rows come back as one copy.  Synchronous: it
 * returns after the outputs are in the caller's buffers.  VSD_ERR_OOM if the
 * staging cannot be allocated. */
vsd_status vsd_verify_step_host(const vsd_model* m, vsd_kv* kv, int32_t batch,
                                int32_t* seq_lens_host, int32_t* pending_host,
                                const int32_t* drafts_host, int32_t* accepted_host,
                                int32_t* out_tokens_host, vsd_stream stream);

/* The same step, also writing float32 logits [B*17, vocab] and the residual
 * stream hidden [layers+1, B*17, hidden] (entry 0 = embeddings, entry l+1 =
 * after layer l); either pointer may be NULL.  Row index = b*17 + j. */
vsd_status vsd_verify_step_debug(const vsd_model* m, vsd_kv* kv, int32_t batch,
                                 int32_t* seq_lens_dev, int32_t* pending_dev,
                                 const int32_t* drafts_dev, int32_t* accepted_dev,
                                 int32_t* out_tokens_dev, float* logits_dev,
                                 float* hidden_dev, vsd_stream stream);

/* Stochastic verification at temperature T > 0: the pages require that the
 * accepted tokens keep the target's output distribution ("The Inference
 * Stack Behind OCRia", speculative-decoding section) and print a sampler at
 * temperature 0.7 with accept / correction / bonus branches ("LLM inference
 * acceleration", section 3.2).  The rule (from the speculative-sampling
 * literature, for a drafter proposing single tokens): draft d_j is accepted
 * iff u_accept[b][j] < p_j(d_j), p_j = softmax(logits_j / T); the first
 * rejected row a gives out[a] = a sample of p_a without d_a; after 16
 * acceptances out[16] = a sample of p_16.  Samples are drawn by inverse CDF
 * over token ids in increasing order at u_sample[b][a] (the smallest id whose
 * cumulative mass reaches u times the total).  Weights are float32 and taken
 * relative to each row's largest logit, exp((logit - max) / T), so any logit
 * magnitude and any T > 0 give the softmax (no overflow, no clamp).  Commits
 * as the greedy step.
 *   u_accept_dev float32 [B, 16], u_sample_dev float32 [B, 17]: uniforms in
 *                (0, 1), the caller's random numbers
 *   logits_dev   optional float32 [B*17, vocab]
 * VSD_ERR_UNSUPPORTED for a head that is not 16-bit or hidden % 16 != 0. */
vsd_status vsd_verify_step_sampled(const vsd_model* m, vsd_kv* kv, int32_t batch,
                                   int32_t* seq_lens_dev, int32_t* pending_dev,
                                   const int32_t* drafts_dev, int32_t* accepted_dev,
                                   int32_t* out_tokens_dev, const float* u_accept_dev,
                                   const float* u_sample_dev, float temperature,
                                   float* logits_dev, vsd_stream stream);

/* Kernel kinds reported by vsd_verify_step_profiled. */
#define VSD_K_EMBED      0  /* embedding gather (+ f16 copy, sums of squares) */
#define VSD_K_QKV        1  /* QKV GEMM + RMSNorm scale + RoPE + block K/V to scratch */
#define VSD_K_ATTENTION  2  /* verify attention */
#define VSD_K_O_PROJ     3  /* O GEMM + residual */
#define VSD_K_GATE_UP    4  /* gate/up GEMM + RMSNorm scale + SiLU * up */
#define VSD_K_DOWN       5  /* down GEMM + residual */
#define VSD_K_LM_HEAD    6  /* lm_head GEMM + RMSNorm scale + argmax */
#define VSD_K_COMMIT     7  /* accept + KV commit */
#define VSD_K_STEP       8  /* the decoder layers and the head in one persistent launch */

/* The same step with a CUDA event recorded before and after every kernel
 * launch (which keeps each launch from overlapping its neighbours).  Writes,
 * for each launch i < *n_launches_host (at most max_launches), its kind
 * (VSD_K_*) to kinds_host[i] and its duration in milliseconds to
 * ms_host[i].  Synchronises the stream; for measurement, not for serving. */
vsd_status vsd_verify_step_profiled(const vsd_model* m, vsd_kv* kv, int32_t batch,
                                    int32_t* seq_lens_dev, int32_t* pending_dev,
                                    const int32_t* drafts_dev, int32_t* accepted_dev,
                                    int32_t* out_tokens_dev, int32_t max_launches,
                                    int32_t* kinds_host, float* ms_host,
                                    int32_t* n_launches_host, vsd_stream stream);

/* ---------------------------------------------------------------- drafting
 * One forward pass of a block drafter proposes the next 16 tokens of every
 * request at once, conditioned on the target's hidden state at the anchor
 * (the last accepted position) -- HunyuanOCR-1.5 summary, section one (the
 * DFlash drafter: a 5-layer transformer initialised from the target's last
 * five decoder layers, input the target's hidden state at the anchor, one
 * pass per block of 16); "The Inference Stack Behind OCRia", section
 * "Generate more tokens per target pass" (one drafter pass per block).
 * Readings where the pages are silent: the drafter has the target's layer
 * shapes and formats (any number of layers up to the target's); its input
 * rows are [anchor_b, E[mask], ..., E[mask]] (16 mask rows) at positions
 * L_b .. L_b+16, where anchor_b is the target's residual row (before the
 * final norm) at the last accepted position; attention is causal among
 * these 17 rows and reads no cache; draft j is the argmax (ties to the
 * lowest id) of row 1+j of the drafter's head.  The drafter's weights are
 * the caller's (random in this library's tests and benchmark).
 *
 * The pass runs in the target cache's scratch (activations, staging K/V of
 * the first `layers` layers, argmax keys), so it must not overlap a verify
 * step of the same cache on the GPU; vsd_verify_step leaves the anchor rows
 * of its requests in the cache for the next draft pass.  */

/* drafter: a model whose shape and formats equal the target's except for a
 * layer count <= the target's (else VSD_ERR_ARG).
 *   seq_lens_dev int32 [B]: committed lengths L_b (positions of row 0)
 *   mask_token   id whose embedding fills rows 1..16
 *   drafts_dev   int32 [B, 16] out: the proposed tokens (-1 and
 *                VSD_DEV_BAD_TOKEN in the status word if a row had no key)
 * Needs L_b + 17 <= max_tokens_per_req (else VSD_DEV_BAD_SEQLEN). */
vsd_status vsd_draft_step(const vsd_model* drafter, vsd_kv* kv, int32_t batch,
                          const int32_t* seq_lens_dev, int32_t mask_token,
                          int32_t* drafts_dev, vsd_stream stream);

/* The same pass with an explicit anchor (anchor_dev float32 [B, hidden], or
 * NULL for the rows the last verify step left) and optional float32 logits
 * [B*17, vocab] and residual stream [layers+1, B*17, hidden] outputs. */
vsd_status vsd_draft_step_debug(const vsd_model* drafter, vsd_kv* kv, int32_t batch,
                                const int32_t* seq_lens_dev, int32_t mask_token,
                                const float* anchor_dev, int32_t* drafts_dev,
                                float* logits_dev, float* hidden_dev, vsd_stream stream);

/* ---------------------------------------------------------------- device-resident loop
 * n_iters iterations of draft -> verify -> commit without the host: each
 * iteration (1) retires the requests that have generated their budget and
 * admits queued requests into empty slots in queue order, (2) runs the
 * drafter pass on every slot's anchor row, (3) runs the verify step on the
 * slots, (4) appends each slot's accepted tokens (the target's greedy
 * tokens g_0..g_a) to its request's output.  The pages' serving loop:
 * "LLM inference acceleration", section three (continuous batching: finished
 * requests leave the running batch, waiting ones take their places, first
 * come first served); "The Inference Stack Behind OCRia", "Fixing CPU-side
 * preparation" (no host round trips between steps).  Everything is
 * asynchronous on `stream` and capturable in one CUDA graph.
 *
 * Layout: the cache holds >= slots + queued requests; slots 0..slots-1 run,
 * cache slot slots+q holds queued request q's context (written by the
 * caller, e.g. vsd_kv_write at that index, with its page-table row).  On
 * admission, slot b takes that page-table row, length req_len[q], pending
 * token req_pending[q] and anchor row req_anchor[q] (float32 [queued,
 * hidden]: the target's residual row at the request's last context
 * position).  An empty slot runs with length -1: computed, never committed,
 * not an error.  Requires req_len[q] + req_budget[q] + 16 + 17 <=
 * max_tokens_per_req (not checked on the device beyond the step's own
 * VSD_DEV_BAD_SEQLEN).
 *   slot_req_dev   int32 [slots] in/out: request in each slot, -1 empty
 *                  (start: all -1)
 *   next_req_dev   int32 [1] in/out: first request not yet admitted (start 0)
 *   iter_dev       int32 [1] in/out: iteration counter (start 0)
 *   req_generated  int32 [queued] in/out: tokens generated (start 0)
 *   req_admit_iter int32 [queued] out: iteration of admission (start -1)
 *   req_out        int32 [queued, out_cap] out: generated tokens, in order
 *                  (the first out_cap of them)
 * A request stays in its slot until it has generated >= req_budget[q]
 * tokens; the tokens of its last step beyond out_cap are not stored. */
vsd_status vsd_spec_loop(const vsd_model* target, const vsd_model* drafter, vsd_kv* kv,
                         int32_t slots, int32_t queued, const int32_t* req_len_dev,
                         const int32_t* req_pending_dev, const int32_t* req_budget_dev,
                         const float* req_anchor_dev, int32_t* slot_req_dev,
                         int32_t* next_req_dev, int32_t* iter_dev, int32_t* req_generated_dev,
                         int32_t* req_admit_iter_dev, int32_t* req_out_dev, int32_t out_cap,
                         int32_t n_iters, int32_t mask_token, vsd_stream stream);

/* Copies the anchor rows [B, hidden] float32 that the last verify step left
 * (request b: the residual row of its last accepted position) to dst_dev. */
vsd_status vsd_kv_get_anchor(const vsd_kv* kv, int32_t batch, float* dst_dev, vsd_stream stream);

/* ---------------------------------------------------------------- components
 * Single kernels of the step, exposed so that each can be checked alone.  */

/* y = x W^T for one weight in any format (the step's GEMM kernel with a
 * plain float32 store): x_dev f16 [m, K] row-major, y_dev float32 [m, N].
 * W as in vsd_weight, repacked inside the call (allocates; test use). */
vsd_status vsd_linear(const vsd_weight* w, int32_t n, int32_t k, const uint16_t* x_f16_dev,
                      int32_t m, float* y_dev, vsd_stream stream);

/* Block attention of one layer for B requests: q_dev BF16 [B, 17, n_q, hd]
 * (RoPE already applied), k_new_dev / v_new_dev BF16 [B, 17, n_kv, hd] (the
 * block's own rows), cache rows [0, seq_lens[b]) of the layer; row j sees the
 * cached rows and block rows 0..j.  out_dev f16 [B*17, n_q*hd].  The block
 * rows go to the step's scratch, not to the cache. */
vsd_status vsd_block_attention(const vsd_model* m, vsd_kv* kv, int32_t layer, int32_t batch,
                               const int32_t* seq_lens_dev, const uint16_t* q_dev,
                               const uint16_t* k_new_dev, const uint16_t* v_new_dev,
                               uint16_t* out_dev, vsd_stream stream);

/* vsd_block_attention without any device allocation (no counterpart in the
 * method's description; an addition for callers that cannot allocate).
 * Some callers must not call cudaMalloc once they are running: a serving
 * process whose device memory is handed out up front by another allocator,
 * or code that runs where allocation is forbidden or would synchronise the
 * device.  This entry point takes the same arguments and computes the same
 * result as vsd_block_attention, but its scratch (query tiles, the block's
 * staged K/V rows, split partials and their counters) lives in one static
 * device array of 16 MiB that every device loading this library holds from
 * load until the process exits; the cache's own step workspace is not
 * touched.  It calls no allocating routine.
 *   - Limit: B * n_kv tiles of 128 x head_dim query rows plus the split
 *     partials must fit in 16 MiB (the call coarsens the context split until
 *     the partials fit); beyond that it returns VSD_ERR_UNSUPPORTED and
 *     names the bytes it needed.
 *   - The array is shared by all calls on a device and keeps the last
 *     call's contents; each call clears what must start at zero (split
 *     counters, padding rows of the staged block).  Calls whose work
 *     overlaps on the GPU (other streams, other threads) race on it: order
 *     them on one stream.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, no allocation); make that first call before
 *     any stream capture.
 * Device-side errors (bad page numbers) go to the cache's status word, as
 * for vsd_block_attention. */
vsd_status vsd_block_attention_static(const vsd_model* m, vsd_kv* kv, int32_t layer, int32_t batch,
                                      const int32_t* seq_lens_dev, const uint16_t* q_dev,
                                      const uint16_t* k_new_dev, const uint16_t* v_new_dev,
                                      uint16_t* out_dev, vsd_stream stream);

/* The accept-and-commit tail of the step driven by given float32 logits
 * [B*17, vocab] and block K/V rows k_new_dev / v_new_dev BF16
 * [layers, B, 17, n_kv, hd]: per-row argmax, prefix accept, outputs, KV
 * commit, seq_lens / pending update -- exactly as in vsd_verify_step. */
vsd_status vsd_accept_commit(const vsd_model* m, vsd_kv* kv, int32_t batch,
                             const float* logits_dev, const uint16_t* k_new_dev,
                             const uint16_t* v_new_dev, int32_t* seq_lens_dev,
                             int32_t* pending_dev, const int32_t* drafts_dev,
                             int32_t* accepted_dev, int32_t* out_tokens_dev,
                             vsd_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* VSD_H */
