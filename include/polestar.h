/*
 * polestar.h -- C ABI of the GB300 (sm_103a) Polestar calibration + commit path.
 *
 * The operations follow "Polestar: Drift-Aware Cache Calibration and Token
 * Commitment for Efficient Inference of Diffusion LLMs" (arXiv 2607.14107):
 *   - Polestar-Cache, §4.1 (block entry, spherical K-means, residual NVFP4 of
 *     App. C.3, proxy attention + KL drift of Eq. 4, top-k clusters, sparse
 *     layer-wise update packets, update schedule) and Algorithm 1;
 *   - Polestar-Commit, §4.2 (drift history, dynamic threshold, current- and
 *     suffix-block commit) and the commit phases of Algorithm 1;
 *   - the system design of §4.3 (pinned-host NVFP4 store, side-stream prefetch).
 *
 * Conventions (all entry points):
 *   - No call throws; every failure is a polestar_status, with a message kept
 *     for polestar_last_error().  Argument errors are detected on the host
 *     before any launch and leave the context unchanged.
 *   - All device work is issued asynchronously on the context's main stream
 *     (given at init).  Device outputs are valid once that stream is
 *     synchronised.  The side stream carries host<->device traffic of the
 *     NVFP4 store only.
 *   - "device" pointers are CUDA device (or managed) memory of the current
 *     device; "host" pointers are ordinary host memory.  Caller-provided
 *     buffers stay owned by the caller; the context never frees them.
 *   - Layouts are dense, row-major, innermost index last.
 *   - A context is not thread-safe; use one context per host thread.
 */
#ifndef POLESTAR_H
#define POLESTAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct polestar_ctx polestar_ctx; /* opaque; owned by the library */

typedef enum {
  POLESTAR_OK = 0,
  POLESTAR_ERR_INVALID_ARG = 1, /* bad pointer, size or configuration          */
  POLESTAR_ERR_CUDA = 2,        /* a CUDA runtime/driver call failed            */
  POLESTAR_ERR_OOM = 3,         /* device or pinned-host allocation failed      */
  POLESTAR_ERR_STATE = 4,       /* call out of order (e.g. commit before step)  */
  POLESTAR_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up           */
  POLESTAR_ERR_UNSUPPORTED = 6  /* shape outside what the kernels implement     */
} polestar_status;

typedef enum { POLESTAR_FP32 = 0, POLESTAR_BF16 = 1 } polestar_dtype;

/* Model shape and Polestar hyper-parameters (Table 5 defaults in brackets). */
typedef struct {
  int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim;
  float rope_base; /* rotary base theta                                        */
  float rms_eps;   /* RMSNorm epsilon                                          */
  int32_t dtype;   /* polestar_dtype: storage of weights, x0, K/V cache         */
  int32_t batch;   /* independent sequences decoded in lockstep blocks          */
  int32_t prompt_len, gen_len;        /* N = prompt_len + gen_len positions     */
  int32_t block;                      /* B [32]                                 */
  int32_t prefix_win, suffix_win;     /* |Omega^p| [2B], |Omega^s| [B]          */
  int32_t K;                          /* centroids [8]                          */
  int32_t topk;                       /* refreshed clusters k [4]               */
  int32_t tau_upd;                    /* refresh trigger [3]                    */
  int32_t hist;                       /* drift history h [5]                    */
  int32_t kmeans_iters;               /* Lloyd iterations [10]                  */
  float tau_s;                        /* static confidence threshold [0.9]      */
  float tau_suf;                      /* suffix commit confidence [0.9]         */
  float alpha;                        /* drift-gate coefficient [10]            */
  uint64_t seed;                      /* K-means initialisation seed            */
  int32_t host_offload; /* 1: NVFP4 window store in pinned host memory (§4.3) */
} polestar_config;

/* Borrowed device pointers of one decoder layer, in the config dtype.
 * Matrices are row-major [out, in] (y = x W^T): wq [H*dh, d], wk/wv [Hkv*dh, d],
 * wo [d, H*dh], w_gate/w_up [F, d], w_down [d, F]; norms are gains [d]. */
typedef struct {
  const void *wq, *wk, *wv, *wo, *w_gate, *w_up, *w_down, *attn_norm, *ffn_norm;
} polestar_layer_weights;

/* Per-step results.  Device pointers are owned by the context and stay valid
 * until the next polestar_calibrate_step or polestar_release. */
typedef struct {
  const float *drift;      /* device [n_layers, batch, K]: per-cluster KL drift D
                              (Eq. 4 on proxy attention, mean over query heads);
                              0 for sequences that did not refresh this step     */
  const int32_t *topk;     /* device [n_layers, batch, topk]: selected clusters,
                              descending drift, ties to the lower id; -1 when the
                              sequence did not refresh                           */
  const uint8_t *selected; /* device [n_layers, batch, win_max]: 1 = window row in
                              a selected cluster (its update packet was computed) */
  const uint8_t *labels;   /* device [n_layers, batch, win_max]: cluster ids       */
  const float *delta;      /* device [batch, block]: last-layer drift delta_j      */
  const uint8_t *fire;     /* host [batch]: 1 = the sparse refresh ran             */
  int32_t win_len;         /* |Omega_b| of the current block (<= win_max)          */
  int32_t win_max;         /* prefix_win + suffix_win                              */
} polestar_step_out;

/* Create a context: validates cfg, allocates the K/V cache [L, batch, N, 2,
 * Hkv*dh], the window state (centroids, anchors, labels, NVFP4 codes -- in
 * pinned host memory when host_offload = 1), the proxy-attention history and
 * the step workspaces.  `layers` is a host array of n_layers entries whose
 * device pointers must stay valid for the life of the context.  stream_main
 * and stream_side are cudaStream_t values (NULL = legacy default stream; the
 * side stream may equal the main stream).  On success *out receives the
 * context; on failure *out is NULL and nothing stays allocated. */
polestar_status polestar_init(const polestar_config *cfg, const polestar_layer_weights *layers,
                              void *stream_main, void *stream_side, polestar_ctx **out);

/* One denoising step of Polestar-Cache over every layer (Algorithm 1).
 *   x0          device [batch, N, d] (config dtype), 16-byte aligned: layer-0
 *               hidden states of the current step (embeddings of the partially
 *               unmasked sequence)
 *   n_unmasked  host [batch]: tokens unmasked since the previous step (drives the
 *               tau_upd trigger of §4.1 "Update Schedule"); ignored at block entry
 *   block_index active block b, 0 <= b < gen_len / block
 *   block_entry 1 at the first step of block b: forward over the full sequence
 *               (even b) or window + block (odd b), K-means, NVFP4, proxy
 *               attention baseline; 0 for a within-block step
 *   out         may be NULL. */
polestar_status polestar_calibrate_step(polestar_ctx *ctx, const void *x0, const int32_t *n_unmasked,
                                        int32_t block_index, int32_t block_entry,
                                        polestar_step_out *out);

/* Polestar-Commit for the step just calibrated (§4.2).
 *   logits      device [batch, 2*block, vocab] fp32: rows 0..B-1 are the active
 *               block, rows B..2B-1 the suffix block (rows past the sequence end
 *               are ignored)
 *   masked      device [batch, N] uint8: 1 = position still [MASK]
 *   commit_mask device [batch, 2*block] uint8, written: 1 = commit the token
 *   conf        device [batch, 2*block] fp32 or NULL: max-softmax confidence c_j
 * Requires a preceding polestar_calibrate_step on this context. */
polestar_status polestar_commit(polestar_ctx *ctx, const float *logits, int32_t vocab,
                                const uint8_t *masked, uint8_t *commit_mask, float *conf);

/* ---- closed-loop decoding (Algorithm 1 in full; Eq. 1; App. D.1) ----
 *
 * The three calls that close the loop around polestar_calibrate_step and
 * polestar_commit, so that a whole generation runs on the device:
 *
 *   polestar_embed(x0) -> polestar_calibrate_step -> polestar_decode_logits
 *     -> polestar_commit -> polestar_decode_tokens -> (next step)
 *
 * polestar_decode_logits: logits of the 2*block rows the commit gate scores,
 * for the step just calibrated (between polestar_calibrate_step and
 * polestar_commit).  Rows 0..B-1 of each sequence are the active block's
 * last-layer outputs; rows B..2B-1 are the suffix block's update packets
 * U(t, L) for the positions the last layer refreshed this step (a sequence
 * whose sparse refresh ran), zero rows elsewhere (such rows cannot commit:
 * Algorithm 1's suffix commit reads only refreshed rows).  Each row is
 * RMS-normalised with final_norm (eps = cfg.rms_eps), rounded to the config
 * dtype, and multiplied by the LM head:
 *   lm_head     device [vocab, d] config dtype, 16-byte aligned (row-major,
 *               one row per token id)
 *   final_norm  device [d] config dtype
 *   logits      device [batch, 2*block, vocab] fp32, written (the input of
 *               polestar_commit)
 * Needs block <= 64.  POLESTAR_ERR_STATE without a calibrated, uncommitted step.
 *
 * polestar_decode_tokens: after polestar_commit, the greedy tokens of Eq. 1
 * (argmax over the vocabulary, ties to the lower id) are written into `tokens`
 * at every committed position, which leaves the mask.  Before that, the
 * progress rule: a step whose gate committed no token of the active block while
 * some are still masked commits the masked one of highest confidence (ties to
 * the lower position), so every step makes progress (the greedy fallback of
 * the decoder Polestar builds on, App. D.1).
 *   logits      device [batch, 2*block, vocab] fp32 (as given to commit)
 *   commit_mask device [batch, 2*block] uint8: polestar_commit's output, updated
 *               in place by the progress rule
 *   tokens      device [batch, N] int32, updated at committed positions
 *   masked      device [batch, N] uint8, 1 -> 0 at committed positions
 *   n_committed host [batch], written: tokens committed this step (the
 *               tokens-per-forward numerator of App. D.1)
 *   n_block_masked host [batch], written: positions of the active block still
 *               masked after this step (0 = the block is decoded)
 * Synchronises the main stream (the counts come back to the host).
 * POLESTAR_ERR_STATE unless polestar_commit ran since the last calibrate step.
 *
 * polestar_embed: layer-0 inputs of the next step, x0[s, p] = embed[tokens[s,
 * p]] where masked[s, p] = 0, else mask_emb (the [MASK] embedding).  A token
 * id outside [0, vocab) gives a zero row.
 *   embed     device [vocab, d] config dtype
 *   mask_emb  device [d] config dtype
 *   tokens    device [batch, N] int32;  masked device [batch, N] uint8
 *   x0        device [batch, N, d] config dtype, written
 * All three run on the context's main stream; buffers are the caller's. */
polestar_status polestar_decode_logits(polestar_ctx *ctx, const void *lm_head, const void *final_norm,
                                       int32_t vocab, float *logits);
polestar_status polestar_decode_tokens(polestar_ctx *ctx, const float *logits, int32_t vocab,
                                       uint8_t *commit_mask, int32_t *tokens, uint8_t *masked,
                                       int32_t *n_committed, int32_t *n_block_masked);
polestar_status polestar_embed(polestar_ctx *ctx, const void *embed, int32_t vocab, const void *mask_emb,
                               const int32_t *tokens, const uint8_t *masked, void *x0);

/* End-to-end step on HOST buffers: copies x0 (host [batch, N, d], config dtype)
 * to the device on the main stream and logits (host [batch, 2B, vocab] fp32) and
 * masked (host [batch, N] uint8) on a copy stream of the context's own, so that
 * they arrive while polestar_calibrate_step computes; then runs polestar_commit,
 * copies the commit mask back to commit_mask_host ([batch, 2B] uint8) and
 * synchronises the main stream.  The host buffers may be reused as soon as the
 * call returns.  Host buffers should be pinned for full bandwidth.  Staging
 * buffers and the copy stream are created on first use. */
polestar_status polestar_step_host(polestar_ctx *ctx, const void *x0_host, const int32_t *n_unmasked,
                                   int32_t block_index, int32_t block_entry,
                                   const float *logits_host, int32_t vocab,
                                   const uint8_t *masked_host, uint8_t *commit_mask_host);

/* ---- KV-cache staleness (App. C.2 "KV-Cache Staleness Metric") ----
 *
 * polestar_full_forward: full-sequence forward of every position of every
 * sequence through every layer from x0 (device [batch, N, d], config dtype,
 * 16-byte aligned), rewriting the context's whole K/V cache with exactly
 * recomputed keys and values -- the no-cache decoding of §3 that recomputes
 * every position at every step, and the "fully recomputed" K/V that App. C.2
 * measures a cache against.  On a context used as that reference, call it once
 * per step with the step's x0; on a calibrating context it is a full refresh.
 * Only the K/V cache changes: window state, centroids, NVFP4 store, drift
 * histories, trigger counters and the results of the last step stay as they
 * were, so calibration and commit continue normally (a call placed between
 * polestar_calibrate_step and polestar_commit does not disturb that commit).
 * Asynchronous on the main stream.
 *
 * polestar_kv_staleness: E[r] = 1 - (mean_h cos(K_r^h, Kref_r^h) +
 * mean_h cos(V_r^h, Vref_r^h)) / 2 for `rows` rows of two caches laid out
 * [rows][2][n_kv_heads * head_dim] (K then V of each row; `dtype` a
 * polestar_dtype), cosines per KV head (h), averaged over the heads.  A pair
 * of zero vectors counts as cos 1, one zero vector against a non-zero one as
 * cos 0.  kv, kv_ref: device, 16-byte aligned; E: device [rows] fp32; head_dim
 * a multiple of 8; rows <= 2^31 - 1 (else UNSUPPORTED).  Asynchronous on
 * `stream`; no context, no allocation.
 *
 * polestar_cache_staleness: the same metric between the K/V caches of two
 * contexts with the same n_layers, batch, N, n_kv_heads, head_dim and dtype:
 * E device [n_layers, batch, N] fp32, E[l, s, i] = E_i(t, l) of sequence s
 * with `ref` holding the reference (typically a context whose last call was
 * polestar_full_forward on the same x0).  Runs on ctx's main stream after
 * everything issued so far on ref's main stream. */
polestar_status polestar_full_forward(polestar_ctx *ctx, const void *x0);
polestar_status polestar_kv_staleness(const void *kv, const void *kv_ref, int64_t rows, int32_t n_kv_heads,
                                      int32_t head_dim, int32_t dtype, float *E, void *stream);
polestar_status polestar_cache_staleness(polestar_ctx *ctx, polestar_ctx *ref, float *E);

/* Free everything the context owns.  NULL is accepted; the context pointer is
 * invalid afterwards.  Synchronises the context's streams first. */
void polestar_release(polestar_ctx *ctx);

/* Message of the last failure on this context ("" if none).  With ctx == NULL,
 * the message of the last failed polestar_init on this thread. */
const char *polestar_last_error(const polestar_ctx *ctx);

/* Number of kernel launches issued on this context since init (diagnostics). */
uint64_t polestar_launch_count(const polestar_ctx *ctx);

/* ---- live per-kernel timing (CUDA events on the launching stream) ----
 * polestar_profile_begin arms up to `capacity` timed launches (event pairs are
 * recorded around each kernel launch of the classes below until the capacity
 * is used up); polestar_profile_end synchronises the main stream, fills
 * out[0 .. n_classes-1] (indexed by polestar_kernel_class) and disarms.
 * Bytes and flops are the algorithmic figures of each launch: for GEMMs the
 * weight, A-operand and output bytes and 2*M*N*K, with M the launch's row
 * bound. */
typedef enum {
  POLESTAR_KC_GEMM_STEP = 0,  /* projections of within-block steps           */
  POLESTAR_KC_GEMM_ENTRY = 1, /* projections of block-entry forwards          */
  POLESTAR_KC_ATTENTION = 2,  /* row attention + KL drift (within-block)      */
  POLESTAR_KC_CLUSTER = 3,    /* K-means/NVFP4, window patch, centroid update */
  POLESTAR_KC_SELECT = 4,     /* top-k + compaction, delta                    */
  POLESTAR_KC_COMMIT = 5,     /* confidence + commit gate                     */
  POLESTAR_KC_ROWS = 6,       /* norms, rotary/scatter, residuals, gathers    */
  POLESTAR_KC_ATTENTION_ENTRY = 7, /* the same three classes during block entry */
  POLESTAR_KC_CLUSTER_ENTRY = 8,
  POLESTAR_KC_ROWS_ENTRY = 9,
  POLESTAR_KC_COUNT = 10
} polestar_kernel_class;

typedef struct {
  uint64_t launches;   /* timed launches                     */
  double ms;           /* summed event-measured duration     */
  double bytes;        /* summed algorithmic bytes           */
  double flops;        /* summed algorithmic flops           */
  uint64_t dropped;    /* launches not timed (capacity full) */
} polestar_kernel_stats;

polestar_status polestar_profile_begin(polestar_ctx *ctx, int32_t capacity);
polestar_status polestar_profile_end(polestar_ctx *ctx, polestar_kernel_stats *out, int32_t n_classes);

/* ---- projection kernel on caller buffers (test hook) ----
 * C[M, N] (fp32, row stride ldc) = A[M, K] (row stride lda) * W[N, K]^T (row
 * stride ldw), A and W in `dtype`, all device pointers, on `stream` -- the
 * Q/K/V, O and FFN projections of the decoder layer (§2 Eq. 3) that the sparse
 * forward of §4.1 runs over gathered rows.
 * Bits 0-3 of `path` select the kernel: 0 CUDA cores; 1 the tcgen05
 * tensor-core kernels (bf16 only) with the library's own choice of kernel,
 * ring depth and K split; 2 the row-tiled tcgen05 kernel; 3 the
 * weight-stationary tcgen05 kernel (M <= 256); 7 the persistent two-SM
 * pair-tile kernel (clusters of two CTAs walk 256-row x bn-column output
 * tiles with the pair's tensor cores run as one MMA, cta_group::2; any M).
 * Bits 8-15: ring depth.  Bits 16-23: the K split over a cluster (paths 2, 3)
 * or the 64-column k-blocks per stage of path 7 (1, or 2 loaded by one 3D TMA
 * box per operand; K must then be a multiple of 64).  Bits 24-31: columns per
 * tile of paths 2 and 7 in units of 16.  Bits 4-7: the 64-column k-blocks per
 * stage of path 2.  0 = automatic.  Any other kernel number, or a combination
 * the kernel cannot run (too much shared memory, more than 8 splits), returns
 * UNSUPPORTED.
 * m_dev (device int, may be NULL) lowers the row count on the device: rows at
 * or beyond min(M, *m_dev) are left untouched.  Asynchronous. */
polestar_status polestar_debug_gemm(const void *A, int32_t lda, const void *W, int32_t ldw, float *C,
                                    int32_t ldc, int32_t M, const int32_t *m_dev, int32_t N, int32_t K,
                                    int32_t dtype, int32_t path, void *stream);

/* ---- gate/up projections with the SwiGLU activation fused (test hook) ----
 * act[m, f] = bf16(silu(g) * u), g = sum_k A[m, k] Wg[f, k], u = sum_k A[m, k]
 * Wu[f, k] (A, Wg, Wu bf16 device matrices with row strides lda, ldw; act bf16,
 * row stride ld_act >= F), the activation computed from the fp32 accumulators
 * in a tcgen05 kernel's epilogue (after the split-K reduction when K is split).
 * path 1: the library's choice (UNSUPPORTED when that is neither the row-tiled
 * nor the two-SM pair kernel); path 2: the row-tiled kernel with bits 8-15 the
 * ring depth, 16-23 the K split, 24-31 the tile width / 16 (gate and up get
 * half of it each); path 7: the two-SM pair kernel (the pair's first CTA reads
 * the gate rows, the second the up rows of the same output columns) with bits
 * 8-15 the ring depth, 16-23 the k-blocks per stage (1 or 2), 24-31 the pair
 * tile width / 16 (a multiple of 32).  m_dev as in polestar_debug_gemm.
 * Asynchronous. */
polestar_status polestar_debug_gemm_swiglu(const void *A, int32_t lda, const void *Wg, const void *Wu, int32_t ldw,
                                           void *act, int32_t ld_act, int32_t M, const int32_t *m_dev, int32_t F,
                                           int32_t K, int32_t path, void *stream);

/* ---- the projection launch the library picks (test hook) ----
 * For M rows (bf16 tensor-core path), nseg (1..3) weight segments with N[i]
 * (host array) output columns and inner size K: out[4] (host) = {kernel: 1
 * row-tiled, 2 weight-stationary, 5 two-SM pair tiles (path 7 of
 * polestar_debug_gemm); output columns per tile; K split over a cluster (for
 * kernel 5: k-blocks per stage); ring depth}.  Queries the current device's
 * occupancy; launches nothing.  CUDA error (no device) when no device is
 * visible. */
polestar_status polestar_debug_gemm_choice(int32_t M, int32_t nseg, const int32_t *N, int32_t K, int32_t *out);

/* ---- row attention + KL drift on caller buffers (test hook) ----
 * One sequence: q [R, H*dh] (rotary applied), kv [N, 2, Hkv*dh] (K then V of
 * every position), both in `dtype`; out [R, H*dh] in `dtype`.  Rows with
 * tracked[r] != 0 (host array) also read prev [R, H, N] fp32 scores and
 * prev_lse [R, H] (previous measurement), write kl [R, H] =
 * KL(softmax(new) || softmax(prev)) when `measure`, and replace prev/prev_lse by
 * the new scores when `store` (Eq. 4).  Synchronous; allocates and frees its
 * own row tables. */
polestar_status polestar_debug_attention(const void *q, const void *kv, int32_t N, int32_t H, int32_t Hkv,
                                         int32_t head_dim, int32_t R, const uint8_t *tracked, float *prev,
                                         float *prev_lse, int32_t measure, int32_t store, void *out, float *kl,
                                         int32_t dtype, void *stream);
/* The same for `batch` sequences of R rows each, in one launch (the layer
 * loop's launch shape): q [batch * R, H*dh] (sequence-major), kv [batch, N, 2,
 * Hkv*dh], out [batch * R, H*dh]; tracked (host, [R]) marks the same rows of
 * every sequence; prev [batch * R, H, N], prev_lse / kl [batch * R, H]. */
polestar_status polestar_debug_attention_batch(const void *q, const void *kv, int32_t batch, int32_t N, int32_t H,
                                               int32_t Hkv, int32_t head_dim, int32_t R, const uint8_t *tracked,
                                               float *prev, float *prev_lse, int32_t measure, int32_t store,
                                               void *out, float *kl, int32_t dtype, void *stream);

/* ---- Q/K/V projection with the rotary embedding fused (test hook) ----
 * 1 (the default): above 256 rows, where the two-SM pair kernel runs the Q/K/V
 * projection, its epilogue applies the rotary embedding and writes the bf16 Q
 * rows and K/V cache entries; 0: the projection writes fp32 and the row kernel
 * does that.  Both give the same bits.  Returns the previous setting.
 * Process-wide; not for concurrent use with running steps. */
int32_t polestar_debug_qkv_fusion(int32_t on);

/* ---- attention kernel selection (test hook) ----
 * 0: the library's choice (the tcgen05 kernel for bf16 head size 128 when
 * its work items fill every SM twice, else the pipelined mma.sync kernel); 1:
 * the mma.sync kernel; 2: the tcgen05 kernel (S and O accumulated in TMEM,
 * work items of up to 128 rows) wherever it applies (bf16, head size 128;
 * drift measured by the deferred pass).  Affects work lists built after the
 * call (context steps and polestar_debug_attention); returns the previous
 * setting, or -1 for an invalid value.  Process-wide; not for concurrent use
 * with running steps. */
int32_t polestar_debug_attention_impl(int32_t impl);

/* ---- window and trigger (host only; test hooks) ----
 * polestar_debug_window: the local window of block `block_index` (§4.1) as the
 * library computes it for a context with these sizes: span[0..1] = the block's
 * positions [start, end); pos[] (host, cap entries) = the prefix_win positions
 * before the block and the suffix_win positions after it that lie inside
 * [0, prompt_len + gen_len), in order.  Returns their number, or -1 for a
 * negative size, a generation length that is not a positive whole number of
 * blocks, a block index out of range or too small a cap.
 * polestar_debug_trigger: the tau_upd refresh trigger of §4.1 "Update
 * Schedule" for one sequence over `steps` within-block steps that start right
 * after a block entry: n_unmasked[t] (host) tokens unmasked since the previous
 * step; fire[t] (host) = 1 when the refresh runs at step t.  No device work. */
int32_t polestar_debug_window(int32_t prompt_len, int32_t gen_len, int32_t block, int32_t prefix_win,
                              int32_t suffix_win, int32_t block_index, int32_t *span, int32_t *pos, int32_t cap);
polestar_status polestar_debug_trigger(int32_t tau_upd, const int32_t *n_unmasked, int32_t steps, uint8_t *fire);

/* ---- bounded device waits (test hook) ----
 * Every mbarrier wait of the projection kernels gives up after a bound (about
 * 2 s), records a code in the context's device error word and lets its kernel
 * return; the next polestar_calibrate_step / polestar_commit on the context
 * then fails with POLESTAR_ERR_TIMEOUT (leaving the context as it was, so the
 * call can be repeated).  This hook exercises that path without a fault: on
 * the context's main stream it shortens the bound to limit_cycles SM clock
 * cycles, runs one kernel that waits on an mbarrier nobody ever arrives on (the
 * wait runs out and records code 99), restores the default bound and queues
 * the read-back of the error word.  Returns POLESTAR_OK; the timeout is
 * reported by the next call.  The bound is shared by every stream of the
 * device while the hook's kernel runs: call it with no other work in flight.
 * INVALID_ARG for ctx NULL or limit_cycles < 1. */
polestar_status polestar_debug_stalled_wait(polestar_ctx *ctx, int64_t limit_cycles);

/* ---- attention work items (host only; test hook) ----
 * The split of one sequence's attention rows into work items that the row
 * attention kernels take one per CTA group: rows [a0, a0 + na) followed by
 * [b0, b0 + nb) are cut into ceil((na + nb) / max_rows) items of near-equal size
 * (at most max_rows rows each), in order; an item that straddles the two ranges
 * holds {rowA, nA, rowB, nB}, otherwise {row, n, 0, 0}.  Writes the items to
 * out[4 * i .. 4 * i + 3] (host array of cap items) and returns their number, or
 * -1 for a negative count, max_rows < 1 or too small a cap.  No device work. */
int32_t polestar_debug_attention_items(int32_t a0, int32_t na, int32_t b0, int32_t nb, int32_t max_rows,
                                       int32_t *out, int32_t cap);

/* ---- row attention + KL drift that allocates nothing ----
 * The paper has no counterpart to this call; it exists for callers that cannot
 * let a library allocate device memory: a host application that owns every
 * device allocation through its own pool or memory cap, or a latency-critical
 * loop in which cudaMalloc/cudaFree may synchronise the device.  It computes the
 * same thing as polestar_debug_attention (bf16 only, head_dim 64 or 128), with
 * two differences: `tracked` is a DEVICE array [R] of flags (or NULL: no row
 * tracked), and all scratch (row table and work list; key-split partials meet
 * in distributed shared memory) lives in fixed file-scope device arrays of this
 * library: at most 256 rows per call; R > 256 is rejected with
 * POLESTAR_ERR_INVALID_ARG.  Every GPU that loads the library holds these
 * arrays (about 4 KB) until the library is unloaded.  The first call on a device resolves their device
 * addresses (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  Calls share the arrays, which keep the last
 * call's contents: calls that overlap on the GPU (on different streams or
 * devices' shared state) race.  Asynchronous on `stream`; no cudaMalloc,
 * cudaFree or allocating library routine is called. */
polestar_status polestar_attention_noalloc(const void *q, const void *kv, int32_t N, int32_t H, int32_t Hkv,
                                           int32_t head_dim, int32_t R, const uint8_t *tracked, float *prev,
                                           float *prev_lse, int32_t measure, int32_t store, void *out, float *kl,
                                           void *stream);

/* ---- spherical K-means + residual NVFP4 on caller buffers (test hook) ----
 * P independent problems of nw rows: Hw [P, nw, d] fp32 -> labels [P, nw]
 * uint8, z / csum / anchor [P, K, d] fp32, codes [P, nw, d/2], scales
 * [P, nw, d/16]; problem p is initialised from seed like layer p of sequence 0
 * at block `block`.  Synchronous. */
polestar_status polestar_debug_kmeans(const float *Hw, int32_t P, int32_t nw, int32_t d, int32_t K,
                                      int32_t iters, uint64_t seed, int32_t block, uint8_t *labels, float *z,
                                      float *csum, float *anchor, uint8_t *codes, uint8_t *scales, void *stream);

/* ---- storage formats of the window states (Table 11 ablation) ----
 * Encoders and decoders of the hidden-state storage formats that the paper's
 * quantization ablation compares (Table 11; NVFP4 as in App. C.3), on caller
 * buffers.  `h` / `out`: device [rows, d] fp32, 16-byte aligned; d a multiple of
 * 32.  With `anchors` (device [K, d] fp32, 16-byte aligned) and `labels`
 * (device [rows] uint8 cluster ids) a format holds the residual
 * r = fp32(h - anchors[labels[i]]) and decoding adds the anchor back
 * (App. C.3 / §4.1); with anchors NULL it holds h itself.  Layouts (row-major):
 *   FP16   codes uint16 [rows, d] binary16, nearest even; no scales.
 *   FP8    codes uint8 [rows, d]: bit 7 sign, bits 0-6 the E4M3 magnitude
 *          (nearest even, saturating at 448) of fp32(r / s); scales fp32 [rows],
 *          s = fp32(amax / 448).
 *   INT8   codes int8 [rows, d] = clamp(rint(fp32(r / s)), -127, 127); scales
 *          fp32 [rows], s = fp32(amax / 127).
 *   MXFP4  codes uint8 [rows, d/2], two E2M1 codes per byte (element 2i in the
 *          low nibble; bit 3 sign, bits 0-2 index into {0,.5,1,1.5,2,3,4,6},
 *          nearest with ties to the even index, saturating at 6) of r / 2^e;
 *          scales uint8 [rows, d/32] = e + 127 (OCP E8M0) with
 *          e = clamp(floor(log2 amax) - 2, -127, 127) per block of 32.
 *   INT2   codes uint8 [rows, d/4], element 4i+j at bits 2j..2j+1 as 2-bit two's
 *          complement of t in {-1, 0, +1}: t = sign(r) where |r| > s/2, else 0;
 *          scales fp32 [rows], s = amax.
 *   NVFP4  codes uint8 [rows, d/2] as MXFP4 but of fp32(r / s) with
 *          s = E4M3(fp32(amax / 6)) per group of 16 (scales uint8 [rows, d/16]),
 *          the library's own window-store format.
 * amax is the largest |r| of the row (FP8, INT8, INT2), block or group; a zero
 * amax stores zero codes and a zero scale.  Decoded values are
 * fp32(code value * scale) (+ anchor, fp32).
 * polestar_codec_bytes: the code and scale bytes of `rows` rows (either output
 * may be NULL); returns their sum, or -1 for an unknown format, rows < 0 or a d
 * that is not a positive multiple of 32.  encode / decode: asynchronous on
 * `stream`; INVALID_ARG for such sizes, a NULL buffer (scales may be NULL for
 * FP16), labels NULL with anchors given, or a misaligned pointer. */
typedef enum {
  POLESTAR_CODEC_FP16 = 0,
  POLESTAR_CODEC_FP8 = 1,
  POLESTAR_CODEC_INT8 = 2,
  POLESTAR_CODEC_MXFP4 = 3,
  POLESTAR_CODEC_INT2 = 4,
  POLESTAR_CODEC_NVFP4 = 5
} polestar_codec;
int64_t polestar_codec_bytes(int32_t fmt, int32_t rows, int32_t d, int64_t *code_bytes, int64_t *scale_bytes);
polestar_status polestar_codec_encode(int32_t fmt, const float *h, int32_t rows, int32_t d, const float *anchors,
                                      const uint8_t *labels, void *codes, void *scales, void *stream);
polestar_status polestar_codec_decode(int32_t fmt, const void *codes, const void *scales, int32_t rows, int32_t d,
                                      const float *anchors, const uint8_t *labels, float *out, void *stream);

/* ---- inspection (used by parity tests; synchronises the main stream) ---- */
typedef enum {
  POLESTAR_BUF_KV = 0,        /* layer l: [batch, N, 2, Hkv*dh] config dtype        */
  POLESTAR_BUF_CENTROID = 1,  /* layer l: [batch, K, d] fp32 unit proxies z_c       */
  POLESTAR_BUF_CSUM = 2,      /* layer l: [batch, K, d] fp32 member sums s_c        */
  POLESTAR_BUF_ANCHOR = 3,    /* layer l: [batch, K, d] fp32 residual anchors A_c   */
  POLESTAR_BUF_LABELS = 4,    /* layer l: [batch, win_max] uint8                    */
  POLESTAR_BUF_CODES = 5,     /* layer l: [batch, win_max, d/2] uint8 E2M1 pairs,
                                 element 2i in the low nibble                       */
  POLESTAR_BUF_SCALES = 6,    /* layer l: [batch, win_max, d/16] uint8 E4M3         */
  POLESTAR_BUF_ACT_OUT = 7,   /* [batch, block, d] fp32 last-layer output, active rows */
  POLESTAR_BUF_UPDATE = 8,    /* [batch, win_max, d] fp32 last update packet U(t,L)  */
  POLESTAR_BUF_CONF = 9,      /* [batch, 2B] fp32 confidence c                       */
  POLESTAR_BUF_DREL = 10,     /* [batch, 2B] fp32 Delta_j (drift minus history mean) */
  POLESTAR_BUF_TAUD = 11,     /* [batch, 2B] fp32 dynamic threshold tau_d            */
  POLESTAR_BUF_PROXY = 12,    /* layer l: [batch, K, H, N] fp32 last proxy scores    */
  POLESTAR_BUF_WINDOW_H = 13, /* layer l: [batch, win_max, d] fp32 block-entry inputs */
  POLESTAR_BUF_DRIFT = 14,    /* layer l: [batch, K] fp32 (same data as step_out.drift) */
  POLESTAR_BUF_TOPK = 15,     /* layer l: [batch, topk] int32                       */
  POLESTAR_BUF_SELECTED = 16, /* layer l: [batch, win_max] uint8                    */
  POLESTAR_BUF_DELTA = 17,    /* [batch, block] fp32 token drift delta_j            */
  POLESTAR_BUF_PROXY_LSE = 18,   /* layer l: [batch, K, H] fp32 log-sum-exp of the last
                                    proxy scores                                       */
  POLESTAR_BUF_ACTIVE_PREV = 19, /* [batch, block, H, N] fp32 last-layer scores of the
                                    active rows at the previous step                   */
  POLESTAR_BUF_ACTIVE_LSE = 20,  /* [batch, block, H] fp32 their log-sum-exp            */
  POLESTAR_BUF_THETA = 21,       /* [batch, block, max(hist, 1)] fp32 drift history Theta_j,
                                    oldest entry first                                 */
  POLESTAR_BUF_THETA_N = 22      /* [batch, block] int32 entries held in Theta_j        */
} polestar_buffer;

/* Copy `bytes` bytes of an internal buffer (layer `layer` where the buffer is
 * per layer) to host memory.  Fails with INVALID_ARG if bytes exceeds the
 * buffer size or the layer is out of range. */
polestar_status polestar_debug_read(polestar_ctx *ctx, int32_t which, int32_t layer, void *host_dst,
                                    size_t bytes);

/* ---- calibration state import (test hooks; snapshot parity) ----
 * The state one within-block step of Algorithm 1 reads and writes is: the K/V
 * cache of every layer, the window's cluster labels, unit centroids z_c,
 * member sums s_c and anchors A_c, the NVFP4 residual store, the proxy scores
 * and log-sum-exps of the last refresh (every layer), the last layer's
 * active-row scores and log-sum-exps, the drift histories Theta_j, and on the
 * host the active block and each sequence's count of tokens unmasked since the
 * last refresh.  Exporting it is polestar_debug_read of the buffers
 * KV, LABELS, CENTROID, CSUM, ANCHOR, CODES, SCALES, PROXY, PROXY_LSE,
 * ACTIVE_PREV, ACTIVE_LSE, THETA and THETA_N; importing it is
 * polestar_debug_write of the same buffers (same layouts, host memory,
 * synchronous; INVALID_ARG for any other buffer id, a layer out of range or
 * bytes beyond the buffer) followed by polestar_debug_enter_block, which sets
 * the host side as if block `block_index`'s entry step had just run: its local
 * window (§4.1), the trigger counts cum[batch] (host, >= 0; NULL = all 0) and
 * no pending commit, so the next call is a within-block
 * polestar_calibrate_step of that block.  INVALID_ARG for a block out of
 * range or a negative count. */
polestar_status polestar_debug_write(polestar_ctx *ctx, int32_t which, int32_t layer, const void *host_src,
                                     size_t bytes);
polestar_status polestar_debug_enter_block(polestar_ctx *ctx, int32_t block_index, const int32_t *cum);

#ifdef __cplusplus
}
#endif
#endif /* POLESTAR_H */
