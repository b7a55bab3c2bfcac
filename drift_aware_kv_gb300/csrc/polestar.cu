// Host side of the Polestar C ABI: context, buffers, and the per-step layer loop.
//
// One polestar_calibrate_step runs Algorithm 1 of "Polestar: Drift-Aware Cache
// Calibration and Token Commitment for Efficient Inference of Diffusion LLMs"
// for every sequence of the batch:
//   block entry (block-entry phase): forward over E_b (full sequence at even b, window +
//     block at odd b) writing the K/V cache and capturing the window's layer
//     inputs; spherical K-means + residual NVFP4 of every layer (one batched
//     launch); proxy-attention baseline of every layer.
//   within-block step (layer loop, §4.1 "Update Schedule"): the tau_upd trigger
//     per sequence on the host; then for every layer l, on the device: patch the
//     window with U(t, l) and re-project its K/V, incremental centroid update,
//     one QKV projection for active rows + window rows + proxies, attention with
//     the KL epilogue, top-k selection + row compaction, and the gathered O/FFN
//     projections producing the next layer's active inputs and U(t, l+1).
// polestar_commit runs the drift-aware commit gate of §4.2.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/polestar.h"
#include "gemm_tc.h"
#include "kernels.h"

using namespace polestar;

namespace {
thread_local std::string g_init_error;

size_t pad8(size_t x) { return (x + 7) & ~size_t(7); }

struct MetaLayout {
  size_t rows_off, prow_off, win_row_off, proxy_row_off, fire_seqs_off, win_pos_off, fire_off, work_off, track_off,
      total;
  int work_cap;
};

}  // namespace

struct polestar_ctx {
  polestar_config cfg{};
  std::vector<polestar_layer_weights> W;
  cudaStream_t sm = nullptr, ss = nullptr;
  int N = 0, d = 0, H = 0, Hkv = 0, dh = 0, F = 0, L = 0, b = 0, B = 0, Wmax = 0, K = 0;
  int qdim = 0, kvdim = 0, ldg = 0, entry_chunk = 1;
  size_t esz = 4;
  bool bf16 = false;
  int Rmax = 0, rows_cap = 0;
  std::string err;
  uint64_t launches = 0;

  // persistent state
  void* kv = nullptr;            // [L, b, N, 2, kvdim]
  float2* rope = nullptr;        // [N, dh/2]
  uint8_t* labels = nullptr;     // [L, b, Wmax]
  float *z = nullptr, *csum = nullptr, *anchor = nullptr;  // [L, b, K, d]
  // NVFP4 residual store.  Without host_offload: device [L, b, Wmax, d/2] and
  // [.., d/16].  With host_offload the store is pinned host memory of that shape
  // and the device holds a ring of two layers [2, b, Wmax, ..], filled ahead of
  // use and written back after each re-encode on the side stream.
  uint8_t *codes = nullptr, *scales = nullptr;
  uint8_t *codes_host = nullptr, *scales_host = nullptr;
  uint8_t *codes_host_dev = nullptr, *scales_host_dev = nullptr;  // device addresses of the host store
  bool offload = false;
  cudaEvent_t ring_in[2] = {nullptr, nullptr};    // side: layer copied into the slot
  cudaEvent_t ring_used[2] = {nullptr, nullptr};  // main: the slot's kernel is done
  cudaEvent_t ring_out[2] = {nullptr, nullptr};   // side: the slot is copied out
  float *pprev = nullptr, *pprev_lse = nullptr;            // [L, b, K, H, N], [L, b, K, H]
  float *aprev = nullptr, *aprev_lse = nullptr;            // [b, B, H, N], [b, B, H]
  // this step's scores of the tracked rows, written by the attention launch and
  // compared with the ones above by the drift pass (same layouts, one layer)
  float *pnew = nullptr, *pnew_lse = nullptr;              // [b, K, H, N], [b, K, H]
  float *anew = nullptr, *anew_lse = nullptr;              // [b, B, H, N], [b, B, H]
  float* theta = nullptr;        // [b, B, hist]
  int* theta_n = nullptr;        // [b, B]
  float* Hw = nullptr;           // [L, b, Wmax, d]
  // workspaces
  float *h_rows = nullptr, *h1 = nullptr, *gout = nullptr, *kl_rows = nullptr;
  int num_sms = 148;
  void *a_in = nullptr, *q_rows = nullptr, *attn_out = nullptr;
  void* act = nullptr;  // bf16 SwiGLU output of the fused gate/up projection [<= 128][F]
  uint8_t* write_kv = nullptr;
  float *U = nullptr, *dn = nullptr;
  // closed-loop decoding: active rows' last-layer outputs of a block entry, the
  // LM head's input rows, greedy tokens, committed counts (device + pinned host)
  float* act_last = nullptr;    // [b, B, d]
  void* dec_rows = nullptr;     // [b * 2B, d] storage type
  int* dec_ids = nullptr;       // [b * 2B]
  int* dec_counts = nullptr;    // [b, 2]: committed, still masked in the block
  int* dec_counts_h = nullptr;  // [b, 2] pinned
  int committed = 0;            // polestar_commit ran after the last calibrate step
  uint8_t *sel_a = nullptr, *sel_b = nullptr, *sel_last = nullptr;
  int *o_src = nullptr, *m_o = nullptr;
  // outputs
  float* drift = nullptr;        // [L, b, K]
  int* topk_out = nullptr;       // [L, b, topk]
  uint8_t* selected = nullptr;   // [L, b, Wmax]
  float* delta = nullptr;        // [b, B]
  float *conf = nullptr, *drel = nullptr, *taud = nullptr, *cpart = nullptr;
  uint8_t* commit_dev = nullptr;
  int csplits = 1;
  // step metadata (pinned host + device mirror)
  MetaLayout ml{};
  uint8_t* meta_h = nullptr;
  uint8_t* meta_d = nullptr;
  cudaEvent_t meta_ev = nullptr, side_ev = nullptr, main_ev = nullptr;
  // device word of timed-out waits (tensor-core GEMM, attention), copied to
  // pinned memory after every step and checked at the next call
  int* err_host = nullptr;
  cudaEvent_t err_ev = nullptr;
  // host bookkeeping
  std::vector<int> cum;
  std::vector<uint8_t> fire;
  std::vector<int> win_pos;
  int cur_block = -1, cur_entry = 0, stepped = 0, nw = 0, start = 0, end = 0;
  // e2e staging
  void* st_x0 = nullptr;
  float* st_logits = nullptr;
  size_t st_logits_cap = 0;
  uint8_t *st_masked = nullptr, *st_commit = nullptr;
  // polestar_step_host: the commit's inputs (logits, mask) come in on a copy
  // stream of the context's own while the calibration step computes
  cudaStream_t st_copy = nullptr;
  cudaEvent_t st_copy_ev = nullptr;

  std::vector<void*> dev_allocs;
  std::vector<void*> host_allocs;

  TcGemmCache tc;

  // live per-kernel timing
  // A projection whose row count lives on the device (m_dev: the compacted
  // refresh rows) is charged bytes + rows x row_bytes and rows x row_flops, the
  // rows read back (stream-ordered, into prof_rows) when the launch is recorded.
  struct ProfRec {
    int cls;
    double bytes, flops;
    double row_bytes = 0.0, row_flops = 0.0;
    int max_rows = 0;
    bool device_rows = false;
  };
  int* prof_rows = nullptr;  // pinned [prof_cap]
  bool prof_armed = false;
  int prof_cap = 0, prof_used = 0, gemm_cls = POLESTAR_KC_GEMM_STEP;
  std::vector<cudaEvent_t> prof_ev;
  std::vector<ProfRec> prof_rec;
  uint64_t prof_dropped[POLESTAR_KC_COUNT] = {};
};

namespace {

polestar_status fail(polestar_ctx* c, polestar_status st, const std::string& msg) {
  if (c)
    c->err = msg;
  else
    g_init_error = msg;
  return st;
}

#define CUDA_OR_FAIL(ctx, call)                                                                   \
  do {                                                                                            \
    cudaError_t e_ = (call);                                                                      \
    if (e_ != cudaSuccess)                                                                        \
      return fail(ctx, e_ == cudaErrorMemoryAllocation ? POLESTAR_ERR_OOM : POLESTAR_ERR_CUDA,    \
                  std::string(#call) + ": " + cudaGetErrorString(e_));                            \
  } while (0)

#define LAUNCHED(ctx)                                                                             \
  do {                                                                                            \
    ++(ctx)->launches;                                                                            \
    cudaError_t e_ = cudaGetLastError();                                                          \
    if (e_ != cudaSuccess) return fail(ctx, POLESTAR_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(e_)); \
  } while (0)

template <typename P>
polestar_status dalloc(polestar_ctx* c, P** p, size_t bytes) {
  void* q = nullptr;
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(c, POLESTAR_ERR_OOM, "cudaMalloc(" + std::to_string(bytes) + "): " + cudaGetErrorString(e));
  }
  c->dev_allocs.push_back(q);
  *p = (P*)q;
  return POLESTAR_OK;
}

template <typename P>
polestar_status halloc(polestar_ctx* c, P** p, size_t bytes) {
  void* q = nullptr;
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaHostAlloc(&q, bytes, cudaHostAllocDefault);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(c, POLESTAR_ERR_OOM, "cudaHostAlloc(" + std::to_string(bytes) + "): " + cudaGetErrorString(e));
  }
  c->host_allocs.push_back(q);
  *p = (P*)q;
  return POLESTAR_OK;
}

#define TRY(x)                             \
  do {                                     \
    polestar_status s_ = (x);              \
    if (s_ != POLESTAR_OK) return s_;      \
  } while (0)

int prof_start(polestar_ctx* c, int cls) {
  if (!c->prof_armed) return -1;
  if (c->gemm_cls == POLESTAR_KC_GEMM_ENTRY) {
    if (cls == POLESTAR_KC_ATTENTION) cls = POLESTAR_KC_ATTENTION_ENTRY;
    if (cls == POLESTAR_KC_CLUSTER) cls = POLESTAR_KC_CLUSTER_ENTRY;
    if (cls == POLESTAR_KC_ROWS) cls = POLESTAR_KC_ROWS_ENTRY;
  }
  if (c->prof_used >= c->prof_cap) {
    ++c->prof_dropped[cls];
    return -1;
  }
  const int i = c->prof_used++;
  cudaEventRecord(c->prof_ev[2 * i], c->sm);
  c->prof_rec[i] = polestar_ctx::ProfRec{cls, 0.0, 0.0};
  return i;
}

void prof_stop(polestar_ctx* c, int i, double bytes, double flops) {
  if (i < 0) return;
  cudaEventRecord(c->prof_ev[2 * i + 1], c->sm);
  c->prof_rec[i].bytes = bytes;
  c->prof_rec[i].flops = flops;
}

// A row-count-dependent launch: M rows (m_dev == nullptr) or the count at
// m_dev (at most M) when the launch runs.
void prof_stop_rows(polestar_ctx* c, int i, double fixed_bytes, double row_bytes, double row_flops, int M,
                    const int* m_dev) {
  if (i < 0) return;
  cudaEventRecord(c->prof_ev[2 * i + 1], c->sm);
  polestar_ctx::ProfRec& r = c->prof_rec[i];
  r.bytes = fixed_bytes;
  r.flops = 0.0;
  r.row_bytes = row_bytes;
  r.row_flops = row_flops;
  r.max_rows = M;
  r.device_rows = m_dev != nullptr && c->prof_rows != nullptr;
  if (r.device_rows) cudaMemcpyAsync(c->prof_rows + i, m_dev, sizeof(int), cudaMemcpyDeviceToHost, c->sm);
}

void prof_release(polestar_ctx* c) {
  for (cudaEvent_t e : c->prof_ev) cudaEventDestroy(e);
  if (c->prof_rows) cudaFreeHost(c->prof_rows);
  c->prof_rows = nullptr;
  c->prof_ev.clear();
  c->prof_rec.clear();
  c->prof_armed = false;
  c->prof_cap = c->prof_used = 0;
}

#define RUN(cls, bytes, flops, stmt)        \
  do {                                      \
    const int pi_ = prof_start(c, (cls));   \
    stmt;                                   \
    prof_stop(c, pi_, (bytes), (flops));    \
    LAUNCHED(c);                            \
  } while (0)

// A launch over M rows (or the device count at m_dev): fixed + rows x row_bytes.
#define RUN_ROWS(cls, fixed, row_bytes, M, m_dev, stmt)                 \
  do {                                                                \
    const int pi_ = prof_start(c, (cls));                             \
    stmt;                                                             \
    prof_stop_rows(c, pi_, (fixed), (row_bytes), 0.0, (M), (m_dev));  \
    LAUNCHED(c);                                                      \
  } while (0)

void free_all(polestar_ctx* c) {
  if (c->sm) cudaStreamSynchronize(c->sm);
  if (c->ss && c->ss != c->sm) cudaStreamSynchronize(c->ss);
  for (void* p : c->dev_allocs) cudaFree(p);
  for (void* p : c->host_allocs) cudaFreeHost(p);
  c->dev_allocs.clear();
  c->host_allocs.clear();
  if (c->meta_ev) cudaEventDestroy(c->meta_ev);
  if (c->err_ev) cudaEventDestroy(c->err_ev);
  c->err_ev = nullptr;
  if (c->side_ev) cudaEventDestroy(c->side_ev);
  if (c->main_ev) cudaEventDestroy(c->main_ev);
  for (int i = 0; i < 2; ++i) {
    if (c->ring_in[i]) cudaEventDestroy(c->ring_in[i]);
    if (c->ring_used[i]) cudaEventDestroy(c->ring_used[i]);
    if (c->ring_out[i]) cudaEventDestroy(c->ring_out[i]);
    c->ring_in[i] = c->ring_used[i] = c->ring_out[i] = nullptr;
  }
  c->meta_ev = c->side_ev = c->main_ev = nullptr;
  if (c->st_copy) {
    cudaStreamSynchronize(c->st_copy);
    cudaStreamDestroy(c->st_copy);
  }
  if (c->st_copy_ev) cudaEventDestroy(c->st_copy_ev);
  c->st_copy = nullptr;
  c->st_copy_ev = nullptr;
  tc_gemm_cache_clear(&c->tc);
  prof_release(c);
}

std::string validate(const polestar_config* c) {
  if (c->n_layers < 1) return "n_layers must be >= 1";
  if (c->dtype != POLESTAR_FP32 && c->dtype != POLESTAR_BF16) return "dtype must be 0 (fp32) or 1 (bf16)";
  if (c->head_dim != 64 && c->head_dim != 128) return "head_dim must be 64 or 128";
  if (c->n_heads < 1 || c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads) return "n_heads must be a multiple of n_kv_heads";
  if (c->d_model < 16 || c->d_model % 16) return "d_model must be a positive multiple of 16";
  if (c->d_model > 4096) return "d_model above 4096 is not supported by the clustering kernel";
  if (c->ffn_dim < 8 || c->ffn_dim % 8) return "ffn_dim must be a positive multiple of 8";
  if (c->n_heads * c->head_dim > 8192) return "n_heads * head_dim above 8192 is not supported";
  if (c->batch < 1 || c->batch > 32) return "batch must be in [1, 32]";
  if (c->block < 8 || c->block % 8) return "block must be a positive multiple of 8";
  if (c->gen_len < c->block || c->gen_len % c->block) return "gen_len must be a positive multiple of block";
  if (c->prompt_len < 0) return "prompt_len must be >= 0";
  if (c->prefix_win < 0 || c->suffix_win < 0 || c->prefix_win + c->suffix_win < 1) return "bad window sizes";
  if (c->prefix_win + c->suffix_win > 128) return "window above 128 rows is not supported";
  if (c->K < 1 || c->K > 8) return "K must be in [1, 8]";
  if (c->topk < 1 || c->topk > c->K) return "topk must be in [1, K]";
  if (c->tau_upd < 0 || c->hist < 0 || c->hist > 64 || c->kmeans_iters < 1) return "bad schedule parameters";
  if (!(c->rms_eps >= 0.f) || !(c->rope_base > 0.f)) return "bad rms_eps / rope_base";
  if (polestar::kmeans_cluster_size(c->d_model, c->prefix_win + c->suffix_win, c->K) < 0)
    return "window x d_model too large for the clustering kernel";
  return "";
}

MetaLayout meta_layout(int rows_cap, int b, int K, int Wmax, int N) {
  MetaLayout m{};
  // attention items (at most ATT_ITEM_ROWS rows of one sequence): block-entry
  // rows, within-block rows (active block + window + proxies), proxy baselines
  m.work_cap = b * (N / ATT_ITEM_ROWS + 2) + b * ((Wmax + K) / ATT_ITEM_ROWS + 3) + 2 * b + 64;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t r = o;
    o = (o + bytes + 15) & ~size_t(15);
    return r;
  };
  m.rows_off = take(sizeof(int4) * rows_cap);
  m.prow_off = take(sizeof(int4) * pad8((size_t)b * K));
  m.win_row_off = take(sizeof(int) * b);
  m.proxy_row_off = take(sizeof(int) * b);
  m.fire_seqs_off = take(sizeof(int) * b);
  m.win_pos_off = take(sizeof(int) * Wmax);
  m.fire_off = take(b);
  m.work_off = take(sizeof(int4) * m.work_cap);
  m.track_off = take(sizeof(int4) * ((size_t)b * K + (size_t)rows_cap));  // rows_cap >= b * block
  m.total = o;
  return m;
}

template <typename T>
T* meta_h(polestar_ctx* c, size_t off) { return (T*)(c->meta_h + off); }
template <typename T>
T* meta_d(polestar_ctx* c, size_t off) { return (T*)(c->meta_d + off); }

// Local window of block blk (§4.1): the block is [start, end); the window holds
// the `prefix` positions before it and the `suffix` positions after it that lie
// inside [0, N), in position order.
void window_of(int prompt_len, int N, int B, int prefix, int suffix, int blk, int* start, int* end,
               std::vector<int>& pos) {
  *start = prompt_len + blk * B;
  *end = *start + B;
  pos.clear();
  for (int p = *start - prefix; p < *start; ++p)
    if (p >= 0) pos.push_back(p);
  for (int p = *end; p < *end + suffix; ++p)
    if (p < N) pos.push_back(p);
}

// tau_upd trigger of one sequence (§4.1 "Update Schedule"): the tokens unmasked
// since the last refresh accumulate, this step's included; the refresh fires
// when they exceed tau_upd, and the count starts again.
bool trigger_step(int& cum, int n_unmasked, int tau_upd) {
  cum += n_unmasked;
  const bool fire = cum > tau_upd;
  if (fire) cum = 0;
  return fire;
}

void compute_window(polestar_ctx* c, int blk) {
  window_of(c->cfg.prompt_len, c->N, c->B, c->cfg.prefix_win, c->cfg.suffix_win, blk, &c->start, &c->end,
            c->win_pos);
  c->nw = (int)c->win_pos.size();
}

// ---- GEMM dispatch: tcgen05 tensor cores for bf16, CUDA cores for fp32 ----
// Several projections of the same rows (Q/K/V, gate/up): one tensor-core
// launch for bf16, one CUDA-core launch per matrix for fp32.
template <typename T>
polestar_status gemm(polestar_ctx* c, const void* A, int lda, const void* W, int ldw, float* C, int ldc, int M,
                     const int* m_dev, int N, int K);

template <typename T>
polestar_status gemm_multi(polestar_ctx* c, const void* A, int lda, int nseg, const void* const* W, const int* N,
                           float* const* C, int ldc, int M, const int* m_dev, int K) {
  if (M <= 0) return POLESTAR_OK;
  if (sizeof(T) == 2 && tc_gemm_supported(K, lda, K)) {
    double wbytes = 0.0, row_bytes = 0.0, row_flops = 0.0;
    int ldw[3];
    for (int i = 0; i < nseg; ++i) {
      ldw[i] = K;
      wbytes += (double)N[i] * K * sizeof(T);
      row_bytes += (double)K * sizeof(T) + (double)N[i] * 4.0;
      row_flops += 2.0 * N[i] * K;
    }
    const int pi = prof_start(c, c->gemm_cls);
    cudaError_t e = tc_gemm_bf16_multi(&c->tc, A, lda, nseg, W, ldw, N, C, ldc, M, m_dev, K, c->sm);
    prof_stop_rows(c, pi, wbytes, row_bytes, row_flops, M, m_dev);
    ++c->launches;
    if (e != cudaSuccess) return fail(c, POLESTAR_ERR_CUDA, std::string("tcgen05 gemm: ") + cudaGetErrorString(e));
    return POLESTAR_OK;
  }
  for (int i = 0; i < nseg; ++i) TRY(gemm<T>(c, A, lda, W[i], K, C[i], ldc, M, m_dev, N[i], K));
  return POLESTAR_OK;
}

template <typename T>
polestar_status gemm(polestar_ctx* c, const void* A, int lda, const void* W, int ldw, float* C, int ldc, int M,
                     const int* m_dev, int N, int K) {
  if (M <= 0) return POLESTAR_OK;
  const double wbytes = (double)N * K * sizeof(T);
  const double row_bytes = (double)K * sizeof(T) + (double)N * 4.0;
  const double row_flops = 2.0 * N * K;
  if (sizeof(T) == 2 && tc_gemm_supported(K, lda, ldw)) {
    const int pi = prof_start(c, c->gemm_cls);
    cudaError_t e = tc_gemm_bf16(&c->tc, A, lda, W, ldw, C, ldc, M, m_dev, N, K, c->sm);
    prof_stop_rows(c, pi, wbytes, row_bytes, row_flops, M, m_dev);
    ++c->launches;
    if (e != cudaSuccess) return fail(c, POLESTAR_ERR_CUDA, std::string("tcgen05 gemm: ") + cudaGetErrorString(e));
    return POLESTAR_OK;
  }
  const int pi = prof_start(c, c->gemm_cls);
  launch_gemm_simt<T>(A, lda, W, ldw, C, ldc, M, m_dev, N, K, c->sm);
  prof_stop_rows(c, pi, wbytes, row_bytes, row_flops, M, m_dev);
  LAUNCHED(c);
  return POLESTAR_OK;
}

// Q/K/V projection of R rows (A = a_in, rows table `rows`) with the rotary
// embedding and the scatter of Q rows and K/V cache entries: fused into the
// two-SM pair kernel's epilogue when that kernel runs (more than 256 rows,
// bf16), else the projection into gout followed by the row kernel.  Both give
// the same bits (the same accumulators, the same rotation arithmetic).
bool g_qkv_fusion = true;

template <typename T>
polestar_status qkv_rope(polestar_ctx* c, const polestar_layer_weights& w, const int4* rows, const uint8_t* write_kv,
                         int R, void* kv_layer, size_t kv_seq) {
  const int d = c->d;
  const void* Ws[3] = {w.wq, w.wk, w.wv};
  const int Ns[3] = {c->qdim, c->kvdim, c->kvdim};
  int ch[4] = {0, 0, 0, 0};
  if (sizeof(T) == 2 && g_qkv_fusion && R > 256 && tc_gemm_supported(d, d, d) && c->qdim % 256 == 0 &&
      c->kvdim % 256 == 0 && 256 % c->dh == 0 && tc_gemm_choice(&c->tc, R, 3, Ns, d, ch) == cudaSuccess &&
      ch[0] == 5) {
    TcQkvRope q;
    q.rows = rows;
    q.write_kv = write_kv;
    q.rope = c->rope;
    q.q_out = c->q_rows;
    q.kv_layer = kv_layer;
    q.kv_seq_stride = kv_seq;
    q.kvdim = c->kvdim;
    q.dh = c->dh;
    const double wbytes = (double)(c->qdim + 2 * c->kvdim) * d * sizeof(T);
    const double row_bytes = (double)d * sizeof(T) + (double)(c->qdim + 2 * c->kvdim) * sizeof(T);
    const double row_flops = 2.0 * (c->qdim + 2 * c->kvdim) * d;
    const int pi = prof_start(c, c->gemm_cls);
    const cudaError_t e = tc_gemm_bf16_qkv_rope(&c->tc, c->a_in, d, Ws, Ns, R, d, q, c->sm);
    prof_stop_rows(c, pi, wbytes, row_bytes, row_flops, R, nullptr);
    ++c->launches;
    if (e != cudaSuccess) return fail(c, POLESTAR_ERR_CUDA, std::string("tcgen05 Q/K/V + rotary: ") + cudaGetErrorString(e));
    return POLESTAR_OK;
  }
  float* Cs[3] = {c->gout, c->gout + c->qdim, c->gout + c->qdim + c->kvdim};
  TRY(gemm_multi<T>(c, c->a_in, d, 3, Ws, Ns, Cs, c->ldg, R, nullptr, d));
  // fp32 Q/K/V read, bf16 Q written (the K/V rows written depend on the rows' kinds: not counted)
  RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)(c->qdim + 2 * c->kvdim) * 4.0 + (double)c->qdim * c->esz, R, nullptr,
           (launch_rope_scatter<T>(c->gout, c->ldg, rows, write_kv, R, c->H, c->Hkv, c->dh, c->rope, c->q_rows,
                                   kv_layer, kv_seq, c->kvdim, c->sm)));
  return POLESTAR_OK;
}

// Gate/up projections + SwiGLU: one fused tcgen05 launch writing the bf16
// activation into *act_out for at most 128 rows when the library's kernel
// choice is the row-tiled kernel (else the two projections into gout and the
// activation kernel into a_in).  With more rows the fused tile's two half-width
// weight boxes per stage made the projection slower than the launch it saves
// (measured at LLaDA-8B batch 8 and Dream-7B batch 4).
template <typename T>
polestar_status gate_up_swiglu(polestar_ctx* c, const polestar_layer_weights& w, int R, const int* m_dev,
                               const void** act_out) {
  const int d = c->d, F = c->F;
  const int Ns[2] = {F, F};
  int ch[4] = {0, 0, 0, 0};
  if (sizeof(T) == 2 && c->act && R > 0 && tc_gemm_supported(d, d, d) &&
      tc_gemm_choice(&c->tc, R, 2, Ns, d, ch) == cudaSuccess && ((R <= 128 && ch[0] == 1) || ch[0] == 5)) {
    const int pi = prof_start(c, c->gemm_cls);
    const cudaError_t e = tc_gemm_bf16_swiglu(&c->tc, c->a_in, d, w.w_gate, w.w_up, d, F, c->act, F, R, m_dev, d, c->sm);
    prof_stop_rows(c, pi, (double)2 * F * d * sizeof(T), (double)d * sizeof(T) + (double)F * 2.0, 4.0 * F * d, R,
                   m_dev);
    ++c->launches;
    if (e != cudaSuccess) return fail(c, POLESTAR_ERR_CUDA, std::string("tcgen05 gemm + SwiGLU: ") + cudaGetErrorString(e));
    *act_out = c->act;
    return POLESTAR_OK;
  }
  const void* Ws[2] = {w.w_gate, w.w_up};
  float* Cs[2] = {c->gout, c->gout + F};
  TRY(gemm_multi<T>(c, c->a_in, d, 2, Ws, Ns, Cs, c->ldg, R, m_dev, d));
  RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)F * (8.0 + sizeof(T)), R, m_dev,
           (launch_swiglu<T>(c->gout, c->ldg, m_dev, R, F, c->a_in, c->sm)));
  *act_out = c->a_in;
  return POLESTAR_OK;
}

// A wait inside a kernel that ran out of time (the kernels record its code in
// the device error word and return): reported as POLESTAR_ERR_TIMEOUT by the
// first call after the step that hit it.
polestar_status check_timeouts(polestar_ctx* c) {
  if (!c->err_ev || cudaEventQuery(c->err_ev) != cudaSuccess) {
    cudaGetLastError();  // not ready (or never recorded): nothing to report yet
    return POLESTAR_OK;
  }
  const int code = *c->err_host;
  if (code == 0) return POLESTAR_OK;
  *c->err_host = 0;
  cudaMemsetAsync(c->tc.err, 0, sizeof(int), c->sm);
  tc_gemm_reset_after_timeout(&c->tc, c->sm);
  return fail(c, POLESTAR_ERR_TIMEOUT, "a device wait timed out (code " + std::to_string(code) +
                                           "); the step's results are not valid");
}

polestar_status record_timeouts(polestar_ctx* c) {
  CUDA_OR_FAIL(c, cudaMemcpyAsync(c->err_host, c->tc.err, sizeof(int), cudaMemcpyDeviceToHost, c->sm));
  CUDA_OR_FAIL(c, cudaEventRecord(c->err_ev, c->sm));
  return POLESTAR_OK;
}

// ------------------------------------------------------------------ NVFP4 store offload
// With host_offload the residual store lives in pinned host memory.  The block
// entry's encoder writes it directly (device mapping of the pinned buffer, over
// NVLink-C2C on Grace-Blackwell); within a block, layer l is fetched into device
// ring slot l & 1 one layer ahead on the side stream and written back after its
// patch.  Every main-stream use of a slot is followed by ring_writeback (side
// stream, after the use), and the fetch of a later layer into that slot is
// queued behind it on the side stream, so a slot is never refilled before its
// previous contents reached the host.
size_t code_layer_bytes(const polestar_ctx* c) { return (size_t)c->b * c->Wmax * (c->d / 2); }
size_t scale_layer_bytes(const polestar_ctx* c) { return (size_t)c->b * c->Wmax * (c->d / 16); }
uint8_t* layer_codes(polestar_ctx* c, int l) {
  return c->codes + (size_t)(c->offload ? (l & 1) : l) * code_layer_bytes(c);
}
uint8_t* layer_scales(polestar_ctx* c, int l) {
  return c->scales + (size_t)(c->offload ? (l & 1) : l) * scale_layer_bytes(c);
}

// side stream: host store layer l -> its ring slot; main waits before use
polestar_status ring_fetch(polestar_ctx* c, int l) {
  const size_t cb = code_layer_bytes(c), sb = scale_layer_bytes(c);
  CUDA_OR_FAIL(c, cudaMemcpyAsync(layer_codes(c, l), c->codes_host + (size_t)l * cb, cb, cudaMemcpyHostToDevice, c->ss));
  CUDA_OR_FAIL(c, cudaMemcpyAsync(layer_scales(c, l), c->scales_host + (size_t)l * sb, sb, cudaMemcpyHostToDevice, c->ss));
  CUDA_OR_FAIL(c, cudaEventRecord(c->ring_in[l & 1], c->ss));
  CUDA_OR_FAIL(c, cudaStreamWaitEvent(c->sm, c->ring_in[l & 1], 0));
  return POLESTAR_OK;
}

// after the main-stream kernel that wrote slot l & 1: slot -> host store layer l
polestar_status ring_writeback(polestar_ctx* c, int l) {
  const size_t cb = code_layer_bytes(c), sb = scale_layer_bytes(c);
  CUDA_OR_FAIL(c, cudaEventRecord(c->ring_used[l & 1], c->sm));
  CUDA_OR_FAIL(c, cudaStreamWaitEvent(c->ss, c->ring_used[l & 1], 0));
  CUDA_OR_FAIL(c, cudaMemcpyAsync(c->codes_host + (size_t)l * cb, layer_codes(c, l), cb, cudaMemcpyDeviceToHost, c->ss));
  CUDA_OR_FAIL(c, cudaMemcpyAsync(c->scales_host + (size_t)l * sb, layer_scales(c, l), sb, cudaMemcpyDeviceToHost, c->ss));
  CUDA_OR_FAIL(c, cudaEventRecord(c->ring_out[l & 1], c->ss));
  return POLESTAR_OK;
}

// ------------------------------------------------------------------ block entry
// fwd_only: the full-sequence forward alone (every position, every layer),
// rewriting the K/V cache and nothing else -- no window capture, no active-row
// score history, no K-means, proxies or trigger reset (polestar_full_forward).
template <typename T>
polestar_status block_entry(polestar_ctx* c, const void* x0, int blk, bool fwd_only = false) {
  const int L = c->L, b = c->b, N = c->N, d = c->d;
  const bool full = fwd_only || (blk % 2 == 0);
  // rows of one sequence (E_b), padded to 8
  std::vector<int> E;
  if (full) {
    for (int p = 0; p < N; ++p) E.push_back(p);
  } else {
    std::vector<char> in(N, 0);
    for (int p : c->win_pos) in[p] = 1;
    for (int p = c->start; p < c->end; ++p) in[p] = 1;
    for (int p = 0; p < N; ++p)
      if (in[p]) E.push_back(p);
  }
  c->gemm_cls = POLESTAR_KC_GEMM_ENTRY;
  const int per_seq = (int)pad8(E.size());
  const int chunk = std::max(1, std::min(b, c->Rmax / per_seq));
  // host metadata: rows of all sequences, proxy rows, window positions
  int4* rows_h = meta_h<int4>(c, c->ml.rows_off);
  std::vector<int> widx_of(N, -1);
  for (int i = 0; i < c->nw; ++i) widx_of[c->win_pos[i]] = i;
  for (int s = 0; s < b; ++s) {
    for (int i = 0; i < per_seq; ++i) {
      int4 m = make_int4(s, 0, ROW_NONE, 0);
      if (i < (int)E.size()) {
        const int p = E[i];
        m.y = p;
        if (fwd_only) {
          m.z = ROW_OTHER;
        } else if (p >= c->start && p < c->end) {
          m.z = ROW_ACTIVE;
          m.w = p - c->start;
        } else if (widx_of[p] >= 0) {
          m.z = ROW_WINDOW;
          m.w = widx_of[p];
        } else {
          m.z = ROW_OTHER;
        }
      }
      rows_h[(size_t)s * per_seq + i] = m;
    }
  }
  int4* prow_h = meta_h<int4>(c, c->ml.prow_off);
  for (int s = 0; s < b; ++s)
    for (int k = 0; k < c->K; ++k) prow_h[s * c->K + k] = make_int4(s, 0, ROW_PROXY, k);
  for (size_t i = (size_t)b * c->K; i < pad8((size_t)b * c->K); ++i) prow_h[i] = make_int4(b - 1, 0, ROW_NONE, 0);
  int* wp = meta_h<int>(c, c->ml.win_pos_off);
  for (int i = 0; i < c->nw; ++i) wp[i] = c->win_pos[i];
  // attention work lists: per chunk (row offsets relative to the chunk), then proxies
  int4* work_h = meta_h<int4>(c, c->ml.work_off);
  int nwk = 0;
  std::vector<int> chunk_work_off, chunk_work_n;
  const bool bf16 = c->cfg.dtype == POLESTAR_BF16;
  const int entry_rows =
      attention_item_rows(bf16, c->dh, (long long)std::min(chunk, b) * ((E.size() + ATT_TC_ROWS - 1) / ATT_TC_ROWS),
                          c->H, false);
  for (int s0 = 0; s0 < b; s0 += chunk) {
    const int ns = std::min(chunk, b - s0);
    chunk_work_off.push_back(nwk);
    for (int i = 0; i < ns; ++i) nwk = attention_items(work_h, nwk, i * per_seq, (int)E.size(), 0, 0, entry_rows);
    chunk_work_n.push_back(nwk - chunk_work_off.back());
  }
  const int proxy_work_off = nwk;
  const int proxy_rows =
      attention_item_rows(bf16, c->dh, (long long)b * ((c->K + ATT_TC_ROWS - 1) / ATT_TC_ROWS), c->H, false);
  for (int s = 0; s < b; ++s) nwk = attention_items(work_h, nwk, s * c->K, c->K, 0, 0, proxy_rows);
  const int proxy_work_n = nwk - proxy_work_off;
  if (nwk > c->ml.work_cap) return fail(c, POLESTAR_ERR_UNSUPPORTED, "attention work list overflow");
  CUDA_OR_FAIL(c, cudaMemcpyAsync(c->meta_d, c->meta_h, c->ml.total, cudaMemcpyHostToDevice, c->sm));
  CUDA_OR_FAIL(c, cudaEventRecord(c->meta_ev, c->sm));
  const int4* work_d = meta_d<int4>(c, c->ml.work_off);

  const size_t kv_layer = (size_t)b * N * 2 * c->kvdim;
  const size_t kv_seq = (size_t)N * 2 * c->kvdim;
  T* kv = (T*)c->kv;
  const float eps = c->cfg.rms_eps;
  const int4* rows_all = meta_d<int4>(c, c->ml.rows_off);

  for (int s0 = 0, ci = 0; s0 < b; s0 += chunk, ++ci) {
    const int ns = std::min(chunk, b - s0);
    const int R = ns * per_seq;
    const int4* rows = rows_all + (size_t)s0 * per_seq;
    RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)d * (c->esz + 4), R, nullptr,
             (launch_gather_input<T>(x0, rows, R, N, d, c->h_rows, c->sm)));
    for (int l = 0; l < L; ++l) {
      const polestar_layer_weights& w = c->W[l];
      if (!fwd_only)
        RUN(POLESTAR_KC_ROWS, (double)ns * c->nw * d * 8.0, 0.0,
            (launch_capture_window(c->h_rows, rows, R, d, c->Wmax, c->Hw + (size_t)l * b * c->Wmax * d,
                                   (size_t)c->Wmax * d, c->sm)));
      RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)d * (4 + c->esz), R, nullptr,
               (launch_rmsnorm<T>(c->h_rows, nullptr, nullptr, rows, nullptr, c->K, w.attn_norm, R, d, eps, c->a_in,
                                  c->sm)));
      TRY(qkv_rope<T>(c, w, rows, nullptr, R, kv + (size_t)l * kv_layer, kv_seq));
      AttnArgs aa{};
      aa.q = c->q_rows;
      aa.ldq = c->qdim;
      aa.rows = rows;
      aa.R = R;
      aa.kv_layer = kv + (size_t)l * kv_layer;
      aa.kv_seq_stride = kv_seq;
      aa.kvdim = c->kvdim;
      aa.N = N;
      aa.H = c->H;
      aa.Hkv = c->Hkv;
      aa.dh = c->dh;
      aa.K = c->K;
      aa.B = c->B;
      aa.scale = 1.f / sqrtf((float)c->dh);
      aa.out = c->attn_out;
      aa.ldo = c->qdim;
      aa.other_live = 1;
      aa.work = work_d + chunk_work_off[ci];
      aa.n_work = chunk_work_n[ci];
      aa.item_rows = entry_rows;
      const bool track = (l == L - 1) && !fwd_only;
      if (track) {
        aa.active_prev = c->aprev;
        aa.active_prev_lse = c->aprev_lse;
        aa.store = 1;
      }
      const double attn_bytes = (double)ns * N * 2 * c->kvdim * c->esz +
                                (track ? (double)ns * c->B * c->H * N * 4.0 : 0.0);
      aa.batch = b;
      aa.err = tc_error_word(&c->tc);
      RUN(POLESTAR_KC_ATTENTION, attn_bytes, 4.0 * R * N * c->qdim, CUDA_OR_FAIL(c, (launch_row_attention<T>(aa, c->sm))));
      TRY(gemm<T>(c, c->attn_out, c->qdim, w.wo, c->qdim, c->gout, c->ldg, R, nullptr, d, c->qdim));
      RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)d * (12 + c->esz), R, nullptr,
               (launch_residual_rmsnorm<T>(c->h_rows, nullptr, nullptr, R, c->gout, c->ldg, w.ffn_norm, d, eps,
                                           c->h1, c->a_in, c->sm)));
      const void* act = nullptr;
      TRY(gate_up_swiglu<T>(c, w, R, nullptr, &act));
      TRY(gemm<T>(c, act, c->F, w.w_down, c->F, c->gout, c->ldg, R, nullptr, d, c->F));
      RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)d * 12.0, R, nullptr,
               (launch_residual_scatter<T>(c->h1, c->gout, c->ldg, nullptr, nullptr, R, rows, d, c->Wmax, c->h_rows,
                                           nullptr, c->sm)));
    }
    // the active rows' last-layer outputs: the rows the commit gate scores
    if (!fwd_only)
      RUN(POLESTAR_KC_ROWS, (double)ns * c->B * d * 8.0, 0.0,
          (launch_capture_active(c->h_rows, rows, R, d, c->B, c->act_last, c->sm)));
  }
  if (fwd_only) return POLESTAR_OK;
  // spherical K-means + residual NVFP4 for every (layer, sequence)
  KmeansArgs ka{};
  ka.Hw = c->Hw;
  ka.L = L;
  ka.batch = b;
  ka.Wmax = c->Wmax;
  ka.nw = c->nw;
  ka.d = d;
  ka.K = c->K;
  ka.iters = c->cfg.kmeans_iters;
  ka.seed = c->cfg.seed;
  ka.block = blk;
  ka.labels = c->labels;
  ka.z = c->z;
  ka.csum = c->csum;
  ka.anchor = c->anchor;
  // window rows read once, labels / codes / scales written, z, member sums and
  // anchors written (the iterations' re-reads of the rows are not counted)
  const double km_bytes = (double)L * b *
                          ((double)c->nw * d * (4.0 + 0.5 + 1.0 / 16) + (double)c->nw + 3.0 * c->K * d * 4.0);
  if (!c->offload) {
    ka.layer0 = 0;
    ka.codes = c->codes;
    ka.scales = c->scales;
    RUN(POLESTAR_KC_CLUSTER, km_bytes, 0.0, (launch_kmeans_encode(ka, c->sm)));
  } else {
    // every layer at once, the encoder storing straight into the pinned host
    // store through its device mapping; the previous step's write-backs to
    // that store (side stream) finish first
    CUDA_OR_FAIL(c, cudaEventRecord(c->side_ev, c->ss));
    CUDA_OR_FAIL(c, cudaStreamWaitEvent(c->sm, c->side_ev, 0));
    ka.layer0 = 0;
    ka.codes = c->codes_host_dev;
    ka.scales = c->scales_host_dev;
    RUN(POLESTAR_KC_CLUSTER, km_bytes, 0.0, (launch_kmeans_encode(ka, c->sm)));
  }
  // proxy-attention baseline P(t_b, l) of every layer
  const int Rp = (int)pad8((size_t)b * c->K);
  const int4* prow = meta_d<int4>(c, c->ml.prow_off);
  for (int l = 0; l < L; ++l) {
    const polestar_layer_weights& w = c->W[l];
    RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)d * (4 + c->esz), b * c->K, nullptr,
             (launch_rmsnorm<T>(nullptr, nullptr, nullptr, prow, c->z + (size_t)l * b * c->K * d, c->K, w.attn_norm,
                                Rp, d, eps, c->a_in, c->sm)));
    TRY(gemm<T>(c, c->a_in, d, w.wq, d, c->gout, c->ldg, Rp, nullptr, c->qdim, d));
    RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)c->qdim * (4 + c->esz), b * c->K, nullptr,
             (launch_rope_scatter<T>(c->gout, c->ldg, prow, nullptr, Rp, c->H, c->Hkv, c->dh, c->rope, c->q_rows,
                                     nullptr, 0, c->kvdim, c->sm)));
    AttnArgs aa{};
    aa.q = c->q_rows;
    aa.ldq = c->qdim;
    aa.rows = prow;
    aa.R = Rp;
    aa.kv_layer = kv + (size_t)l * kv_layer;
    aa.kv_seq_stride = kv_seq;
    aa.kvdim = c->kvdim;
    aa.N = N;
    aa.H = c->H;
    aa.Hkv = c->Hkv;
    aa.dh = c->dh;
    aa.K = c->K;
    aa.B = c->B;
    aa.scale = 1.f / sqrtf((float)c->dh);
    aa.out = c->attn_out;
    aa.ldo = c->qdim;
    aa.proxy_prev = c->pprev + (size_t)l * b * c->K * c->H * N;
    aa.proxy_prev_lse = c->pprev_lse + (size_t)l * b * c->K * c->H;
    aa.store = 1;
    aa.work = work_d + proxy_work_off;
    aa.n_work = proxy_work_n;
    aa.item_rows = proxy_rows;
    const double attn_bytes = (double)b * N * 2 * c->kvdim * c->esz + (double)b * c->K * c->H * N * 4.0;
    aa.batch = b;
    aa.err = tc_error_word(&c->tc);
    RUN(POLESTAR_KC_ATTENTION, attn_bytes, 4.0 * Rp * N * c->qdim, CUDA_OR_FAIL(c, (launch_row_attention<T>(aa, c->sm))));
  }
  std::fill(c->cum.begin(), c->cum.end(), 0);
  std::fill(c->fire.begin(), c->fire.end(), 0);
  c->sel_last = nullptr;
  return POLESTAR_OK;
}

// ------------------------------------------------------------- within-block step
template <typename T>
polestar_status within_step(polestar_ctx* c, const void* x0, const int32_t* n_unmasked) {
  const int L = c->L, b = c->b, N = c->N, d = c->d, B = c->B;
  // update schedule (§4.1): refresh when the tokens decoded since the last
  // refresh exceed tau_upd
  std::vector<int> fire_seqs;
  for (int s = 0; s < b; ++s) {
    c->fire[s] = trigger_step(c->cum[s], n_unmasked ? n_unmasked[s] : 0, c->cfg.tau_upd);
    if (c->fire[s]) fire_seqs.push_back(s);
  }
  const int n_fire = (int)fire_seqs.size();
  c->gemm_cls = POLESTAR_KC_GEMM_STEP;
  // row space: active rows of every sequence, then per refreshing sequence its
  // window rows and its K proxy rows (padded to 8)
  int4* rows_h = meta_h<int4>(c, c->ml.rows_off);
  int* win_row = meta_h<int>(c, c->ml.win_row_off);
  int* proxy_row = meta_h<int>(c, c->ml.proxy_row_off);
  int* fseq = meta_h<int>(c, c->ml.fire_seqs_off);
  int* wp = meta_h<int>(c, c->ml.win_pos_off);
  uint8_t* fire_h = meta_h<uint8_t>(c, c->ml.fire_off);
  int R = 0;
  for (int s = 0; s < b; ++s)
    for (int j = 0; j < B; ++j) rows_h[R++] = make_int4(s, c->start + j, ROW_ACTIVE, j);
  for (int s = 0; s < b; ++s) {
    win_row[s] = -1;
    proxy_row[s] = -1;
    fire_h[s] = c->fire[s];
  }
  for (int f = 0; f < n_fire; ++f) {
    const int s = fire_seqs[f];
    fseq[f] = s;
    win_row[s] = R;
    for (int j = 0; j < c->nw; ++j) rows_h[R++] = make_int4(s, c->win_pos[j], ROW_WINDOW, j);
    proxy_row[s] = R;
    for (int k = 0; k < c->K; ++k) rows_h[R++] = make_int4(s, 0, ROW_PROXY, k);
    while (R % 8) rows_h[R++] = make_int4(s, 0, ROW_NONE, 0);
  }
  {
    // rows whose drift the deferred pass measures: the refreshing sequences'
    // proxies (every layer), then the active rows (last layer)
    int4* track = meta_h<int4>(c, c->ml.track_off);
    int n = 0;
    for (int f = 0; f < n_fire; ++f)
      for (int k = 0; k < c->K; ++k) track[n++] = make_int4(proxy_row[fire_seqs[f]] + k, fire_seqs[f], ROW_PROXY, k);
    for (int s = 0; s < b; ++s)
      for (int j = 0; j < B; ++j) track[n++] = make_int4(s * B + j, s, ROW_ACTIVE, j);
  }
  for (int i = 0; i < c->nw; ++i) wp[i] = c->win_pos[i];
  int4* work_h = meta_h<int4>(c, c->ml.work_off);
  int nwk = 0;
  // one sequence's active rows and (when it refreshes) its window + proxy rows
  long long items128 = 0;
  for (int s = 0; s < b; ++s) items128 += (B + (win_row[s] >= 0 ? c->nw + c->K : 0) + ATT_TC_ROWS - 1) / ATT_TC_ROWS;
  const int step_rows = attention_item_rows(c->cfg.dtype == POLESTAR_BF16, c->dh, items128, c->H, true, true);
  for (int s = 0; s < b; ++s)
    nwk = attention_items(work_h, nwk, s * B, B, win_row[s] >= 0 ? win_row[s] : 0, win_row[s] >= 0 ? c->nw + c->K : 0,
                          step_rows);
  if (nwk > c->ml.work_cap) return fail(c, POLESTAR_ERR_UNSUPPORTED, "attention work list overflow");
  CUDA_OR_FAIL(c, cudaMemcpyAsync(c->meta_d, c->meta_h, c->ml.total, cudaMemcpyHostToDevice, c->sm));
  CUDA_OR_FAIL(c, cudaEventRecord(c->meta_ev, c->sm));
  const int4* rows = meta_d<int4>(c, c->ml.rows_off);
  const int* fire_d = meta_d<int>(c, c->ml.fire_seqs_off);
  const int* win_row_d = meta_d<int>(c, c->ml.win_row_off);
  const int* proxy_row_d = meta_d<int>(c, c->ml.proxy_row_off);

  const size_t kv_layer = (size_t)b * N * 2 * c->kvdim;
  const size_t kv_seq = (size_t)N * 2 * c->kvdim;
  T* kv = (T*)c->kv;
  const float eps = c->cfg.rms_eps;
  const int n_active = b * B;

  RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)d * (2 * c->esz + 4), n_active, nullptr,
           (launch_gather_input<T>(x0, rows, n_active, N, d, c->h_rows, c->sm, c->W[0].attn_norm, eps, c->a_in)));
  uint8_t* sel_prev = c->sel_a;
  uint8_t* sel_cur = c->sel_b;
  if (n_fire > 0) {
    RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)d * (c->esz + 4), n_fire * c->nw, nullptr,
             (launch_gather_window<T>(x0, meta_d<int>(c, c->ml.win_pos_off), c->nw, fire_d, n_fire, N, d, c->Wmax,
                                      c->U, sel_prev, c->sm)));
  }
  if (n_fire > 0 && c->offload) {
    // fetches read the host store only after everything queued on the main
    // stream so far (the block entry's encoder writes it directly)
    CUDA_OR_FAIL(c, cudaEventRecord(c->main_ev, c->sm));
    CUDA_OR_FAIL(c, cudaStreamWaitEvent(c->ss, c->main_ev, 0));
    TRY(ring_fetch(c, 0));
  }
  for (int l = 0; l < L; ++l) {
    const polestar_layer_weights& w = c->W[l];
    float* zl = c->z + (size_t)l * b * c->K * d;
    if (n_fire > 0) {
      // next layer's residual codes come in while this layer runs
      if (c->offload && l + 1 < L) {
        const size_t cb = code_layer_bytes(c), sb = scale_layer_bytes(c);
        CUDA_OR_FAIL(c, cudaMemcpyAsync(layer_codes(c, l + 1), c->codes_host + (size_t)(l + 1) * cb, cb,
                                        cudaMemcpyHostToDevice, c->ss));
        CUDA_OR_FAIL(c, cudaMemcpyAsync(layer_scales(c, l + 1), c->scales_host + (size_t)(l + 1) * sb, sb,
                                        cudaMemcpyHostToDevice, c->ss));
        CUDA_OR_FAIL(c, cudaEventRecord(c->ring_in[(l + 1) & 1], c->ss));
      }
      if (c->offload && l > 0) CUDA_OR_FAIL(c, cudaStreamWaitEvent(c->sm, c->ring_in[l & 1], 0));
      PatchArgs pa{};
      pa.fire_seqs = fire_d;
      pa.n_fire = n_fire;
      pa.nw = c->nw;
      pa.Wmax = c->Wmax;
      pa.d = d;
      pa.K = c->K;
      pa.labels = c->labels + (size_t)l * b * c->Wmax;
      pa.anchor = c->anchor + (size_t)l * b * c->K * d;
      pa.codes = layer_codes(c, l);
      pa.scales = layer_scales(c, l);
      pa.U = c->U;
      pa.sel_prev = sel_prev;
      pa.win_row = win_row_d;
      pa.h_rows = c->h_rows;
      pa.write_kv = c->write_kv;
      pa.dn = c->dn;
      pa.csum = c->csum + (size_t)l * b * c->K * d;
      pa.z = zl;
      pa.gain = w.attn_norm;
      pa.eps = eps;
      pa.a_out = c->a_in;
      pa.proxy_row = proxy_row_d;
      // lower bound: every window row's codes read, its layer input and
      // projection input written, the anchors read once; a patched row also
      // reads its packet and writes its direction change and new codes
      RUN_ROWS(POLESTAR_KC_CLUSTER, (double)n_fire * c->K * d * 4.0, (double)d * (0.5 + 1.0 / 16 + 4 + c->esz),
               n_fire * c->nw, nullptr, (launch_window_patch<T>(pa, c->sm)));
      if (c->offload) TRY(ring_writeback(c, l));
      // member sums read and written, z and the proxy rows' input written (the
      // selected rows' direction changes it reads are data-dependent: not counted)
      RUN(POLESTAR_KC_CLUSTER, (double)n_fire * c->K * d * (12.0 + c->esz), 0.0,
          (launch_centroid_update<T>(pa, c->sm)));
    }
    // the projections' input rows were normalised by their producers: active
    // rows by the previous layer's final residual (or the input gather), window
    // rows by the patch, proxy rows by the centroid update
    TRY(qkv_rope<T>(c, w, rows, c->write_kv, R, kv + (size_t)l * kv_layer, kv_seq));
    AttnArgs aa{};
    aa.q = c->q_rows;
    aa.ldq = c->qdim;
    aa.rows = rows;
    aa.R = R;
    aa.kv_layer = kv + (size_t)l * kv_layer;
    aa.kv_seq_stride = kv_seq;
    aa.kvdim = c->kvdim;
    aa.N = N;
    aa.H = c->H;
    aa.Hkv = c->Hkv;
    aa.dh = c->dh;
    aa.K = c->K;
    aa.B = B;
    aa.scale = 1.f / sqrtf((float)c->dh);
    aa.out = c->attn_out;
    aa.ldo = c->qdim;
    aa.other_live = 1;
    aa.proxy_prev = c->pprev + (size_t)l * b * c->K * c->H * N;
    aa.proxy_prev_lse = c->pprev_lse + (size_t)l * b * c->K * c->H;
    if (l == L - 1) {
      aa.active_prev = c->aprev;
      aa.active_prev_lse = c->aprev_lse;
    }
    // drift deferred to the pass below: the attention writes the tracked rows'
    // new scores, the drift pass compares them with the stored ones and
    // replaces those
    aa.measure = 1;
    aa.store = 1;
    aa.proxy_new = c->pnew;
    aa.proxy_new_lse = c->pnew_lse;
    aa.active_new = c->anew;
    aa.active_new_lse = c->anew_lse;
    aa.kl_out = c->kl_rows;
    aa.work = meta_d<int4>(c, c->ml.work_off);
    aa.n_work = nwk;
    aa.item_rows = step_rows;
    const double tracked_keys = (double)n_fire * c->K * c->H * N + (l == L - 1 ? (double)b * B * c->H * N : 0.0);
    const double attn_bytes = (double)b * N * 2 * c->kvdim * c->esz + tracked_keys * 4.0;
    aa.batch = b;
    aa.err = tc_error_word(&c->tc);
    RUN(POLESTAR_KC_ATTENTION, attn_bytes, 4.0 * R * N * c->qdim, CUDA_OR_FAIL(c, (launch_row_attention<T>(aa, c->sm))));
    {
      DriftArgs da{};
      da.track = meta_d<int4>(c, c->ml.track_off);
      da.n_track = n_fire * c->K + (l == L - 1 ? b * B : 0);
      da.H = c->H;
      da.N = N;
      da.K = c->K;
      da.B = B;
      da.proxy_prev = aa.proxy_prev;
      da.proxy_prev_lse = aa.proxy_prev_lse;
      da.active_prev = c->aprev;
      da.active_prev_lse = c->aprev_lse;
      da.proxy_new = c->pnew;
      da.proxy_new_lse = c->pnew_lse;
      da.active_new = c->anew;
      da.active_new_lse = c->anew_lse;
      da.kl_out = c->kl_rows;
      da.store = 1;
      RUN(POLESTAR_KC_ATTENTION, tracked_keys * 12.0, 0.0, (launch_drift(da, c->sm)));
    }
    SelectArgs sa{};
    sa.batch = b;
    sa.Wmax = c->Wmax;
    sa.nw = c->nw;
    sa.K = c->K;
    sa.topk = c->cfg.topk;
    sa.H = c->H;
    sa.B = B;
    sa.kl_rows = c->kl_rows;
    sa.proxy_row = proxy_row_d;
    sa.win_row = win_row_d;
    sa.labels = c->labels + (size_t)l * b * c->Wmax;
    sa.drift = c->drift + (size_t)l * b * c->K;
    sa.topk_out = c->topk_out + (size_t)l * b * c->cfg.topk;
    sa.selected = c->selected + (size_t)l * b * c->Wmax;
    sa.sel_cur = sel_cur;
    sa.o_src = c->o_src;
    sa.m_o = c->m_o;
    sa.n_active = n_active;
    RUN(POLESTAR_KC_SELECT,
        (double)n_fire * c->K * c->H * 4.0 + (double)b * c->Wmax * 3.0 + (double)(n_active + n_fire * c->nw) * 4.0, 0.0,
        (launch_select(sa, c->sm)));
    if (l == L - 1) {
      RUN(POLESTAR_KC_SELECT, (double)b * B * c->H * 4.0, 0.0,
          (launch_delta_finalize(c->kl_rows, b, B, c->H, c->delta, c->sm)));
    }
    // gathered O/FFN over active rows + selected window rows
    const int Rc = n_active + n_fire * c->nw;
    RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)c->qdim * 2 * c->esz, Rc, c->m_o,
             (launch_gather_T<T>(c->attn_out, c->o_src, c->m_o, Rc, c->qdim, c->a_in, c->sm)));
    TRY(gemm<T>(c, c->a_in, c->qdim, w.wo, c->qdim, c->gout, c->ldg, Rc, c->m_o, d, c->qdim));
    RUN_ROWS(POLESTAR_KC_ROWS, 0.0, (double)d * (12 + c->esz), Rc, c->m_o,
             (launch_residual_rmsnorm<T>(c->h_rows, c->o_src, c->m_o, Rc, c->gout, c->ldg, w.ffn_norm, d, eps, c->h1,
                                         c->a_in, c->sm)));
    const void* act = nullptr;
    TRY(gate_up_swiglu<T>(c, w, Rc, c->m_o, &act));
    TRY(gemm<T>(c, act, c->F, w.w_down, c->F, c->gout, c->ldg, Rc, c->m_o, d, c->F));
    // every row: two fp32 rows read, one written; the active rows also write
    // the next layer's projection input
    RUN_ROWS(POLESTAR_KC_ROWS, l + 1 < L ? (double)n_active * d * c->esz : 0.0, (double)d * 12.0, Rc, c->m_o,
             (launch_residual_scatter<T>(c->h1, c->gout, c->ldg, c->o_src, c->m_o, Rc, rows, d, c->Wmax, c->h_rows,
                                         c->U, c->sm, l + 1 < L ? c->W[l + 1].attn_norm : nullptr, eps, c->a_in)));
    std::swap(sel_prev, sel_cur);
  }
  c->sel_last = sel_prev;  // selection of the last layer
  return POLESTAR_OK;
}

template <typename T>
polestar_status step_impl(polestar_ctx* c, const void* x0, const int32_t* n_unmasked, int blk, int entry) {
  if (entry) return block_entry<T>(c, x0, blk);
  return within_step<T>(c, x0, n_unmasked);
}

}  // namespace

// ============================================================================ ABI

extern "C" polestar_status polestar_init(const polestar_config* cfg, const polestar_layer_weights* layers,
                                         void* stream_main, void* stream_side, polestar_ctx** out) {
  if (!out) return fail(nullptr, POLESTAR_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cfg || !layers) return fail(nullptr, POLESTAR_ERR_INVALID_ARG, "cfg or layers is NULL");
  const std::string v = validate(cfg);
  if (!v.empty()) return fail(nullptr, POLESTAR_ERR_INVALID_ARG, v);
  for (int l = 0; l < cfg->n_layers; ++l) {
    const polestar_layer_weights& w = layers[l];
    if (!w.wq || !w.wk || !w.wv || !w.wo || !w.w_gate || !w.w_up || !w.w_down || !w.attn_norm || !w.ffn_norm)
      return fail(nullptr, POLESTAR_ERR_INVALID_ARG, "layer " + std::to_string(l) + " has a NULL weight pointer");
  }
  polestar_ctx* c = new (std::nothrow) polestar_ctx();
  if (!c) return fail(nullptr, POLESTAR_ERR_OOM, "context allocation failed");
  c->cfg = *cfg;
  c->W.assign(layers, layers + cfg->n_layers);
  c->sm = (cudaStream_t)stream_main;
  c->ss = stream_side ? (cudaStream_t)stream_side : c->sm;
  c->L = cfg->n_layers;
  c->d = cfg->d_model;
  c->H = cfg->n_heads;
  c->Hkv = cfg->n_kv_heads;
  c->dh = cfg->head_dim;
  c->F = cfg->ffn_dim;
  c->b = cfg->batch;
  c->B = cfg->block;
  c->N = cfg->prompt_len + cfg->gen_len;
  c->Wmax = cfg->prefix_win + cfg->suffix_win;
  c->K = cfg->K;
  c->qdim = c->H * c->dh;
  c->kvdim = c->Hkv * c->dh;
  c->bf16 = cfg->dtype == POLESTAR_BF16;
  c->esz = c->bf16 ? 2 : 4;
  c->ldg = std::max(std::max(c->qdim + 2 * c->kvdim, 2 * c->F), c->d);
  c->ldg = (c->ldg + 3) & ~3;
  c->cum.assign(c->b, 0);
  c->fire.assign(c->b, 0);

  auto run = [&]() -> polestar_status {
    const int L = c->L, b = c->b, N = c->N, d = c->d, Wmax = c->Wmax, K = c->K, H = c->H, B = c->B;
    const int within_rows = b * B + b * (int)pad8(Wmax + K);
    const int entry_rows = std::max((int)pad8(N), std::min(b * (int)pad8(N), 16384));
    c->Rmax = std::max(within_rows, entry_rows);
    c->rows_cap = std::max(within_rows, b * (int)pad8(N));
    CUDA_OR_FAIL(c, cudaEventCreateWithFlags(&c->meta_ev, cudaEventDisableTiming));
    CUDA_OR_FAIL(c, cudaEventCreateWithFlags(&c->side_ev, cudaEventDisableTiming));
    CUDA_OR_FAIL(c, cudaEventCreateWithFlags(&c->main_ev, cudaEventDisableTiming));
    CUDA_OR_FAIL(c, cudaEventCreateWithFlags(&c->err_ev, cudaEventDisableTiming));
    if (!tc_error_word(&c->tc)) return fail(c, POLESTAR_ERR_OOM, "device error word");
    TRY(halloc(c, &c->err_host, sizeof(int)));
    *c->err_host = 0;
    TRY(dalloc(c, &c->kv, (size_t)L * b * N * 2 * c->kvdim * c->esz));
    CUDA_OR_FAIL(c, cudaMemsetAsync(c->kv, 0, (size_t)L * b * N * 2 * c->kvdim * c->esz, c->sm));
    TRY(dalloc(c, &c->rope, sizeof(float2) * (size_t)N * (c->dh / 2)));
    {
      std::vector<float2> tab((size_t)N * (c->dh / 2));
      for (int p = 0; p < N; ++p)
        for (int i = 0; i < c->dh / 2; ++i) {
          const double th = std::pow((double)cfg->rope_base, -2.0 * i / (double)c->dh);
          tab[(size_t)p * (c->dh / 2) + i] = make_float2((float)std::cos(p * th), (float)std::sin(p * th));
        }
      CUDA_OR_FAIL(c, cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice));
    }
    TRY(dalloc(c, &c->labels, (size_t)L * b * Wmax));
    CUDA_OR_FAIL(c, cudaMemset(c->labels, 0, (size_t)L * b * Wmax));
    TRY(dalloc(c, &c->z, sizeof(float) * (size_t)L * b * K * d));
    TRY(dalloc(c, &c->csum, sizeof(float) * (size_t)L * b * K * d));
    TRY(dalloc(c, &c->anchor, sizeof(float) * (size_t)L * b * K * d));
    c->offload = cfg->host_offload != 0;
    const int code_layers = c->offload ? 2 : L;
    TRY(dalloc(c, &c->codes, (size_t)code_layers * b * Wmax * (d / 2)));
    TRY(dalloc(c, &c->scales, (size_t)code_layers * b * Wmax * (d / 16)));
    if (c->offload) {
      for (int i = 0; i < 2; ++i) {
        CUDA_OR_FAIL(c, cudaEventCreateWithFlags(&c->ring_in[i], cudaEventDisableTiming));
        CUDA_OR_FAIL(c, cudaEventCreateWithFlags(&c->ring_used[i], cudaEventDisableTiming));
        CUDA_OR_FAIL(c, cudaEventCreateWithFlags(&c->ring_out[i], cudaEventDisableTiming));
      }
    }
    TRY(dalloc(c, &c->pprev, sizeof(float) * (size_t)L * b * K * H * N));
    TRY(dalloc(c, &c->pprev_lse, sizeof(float) * (size_t)L * b * K * H));
    TRY(dalloc(c, &c->aprev, sizeof(float) * (size_t)b * B * H * N));
    TRY(dalloc(c, &c->aprev_lse, sizeof(float) * (size_t)b * B * H));
    TRY(dalloc(c, &c->pnew, sizeof(float) * (size_t)b * K * H * N));
    TRY(dalloc(c, &c->pnew_lse, sizeof(float) * (size_t)b * K * H));
    TRY(dalloc(c, &c->anew, sizeof(float) * (size_t)b * B * H * N));
    TRY(dalloc(c, &c->anew_lse, sizeof(float) * (size_t)b * B * H));
    TRY(dalloc(c, &c->theta, sizeof(float) * (size_t)b * B * std::max(1, cfg->hist)));
    TRY(dalloc(c, &c->theta_n, sizeof(int) * (size_t)b * B));
    CUDA_OR_FAIL(c, cudaMemset(c->theta_n, 0, sizeof(int) * (size_t)b * B));
    TRY(dalloc(c, &c->Hw, sizeof(float) * (size_t)L * b * Wmax * d));
    const int R = c->Rmax;
    TRY(dalloc(c, &c->h_rows, sizeof(float) * (size_t)R * d));
    TRY(dalloc(c, &c->h1, sizeof(float) * (size_t)R * d));
    TRY(dalloc(c, &c->gout, sizeof(float) * (size_t)R * c->ldg));
    TRY(dalloc(c, &c->kl_rows, sizeof(float) * (size_t)R * H));
    {
      int dev = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
    }
    TRY(dalloc(c, &c->a_in, c->esz * (size_t)R * std::max(std::max(d, c->F), c->qdim)));
    // SwiGLU activation written by the fused gate/up epilogue (row-tiled kernel
    // up to 128 rows, two-SM pair kernel above 256)
    if (c->bf16) TRY(dalloc(c, &c->act, 2 * (size_t)R * c->F));
    TRY(dalloc(c, &c->q_rows, c->esz * (size_t)R * c->qdim));
    TRY(dalloc(c, &c->attn_out, c->esz * (size_t)R * c->qdim));
    TRY(dalloc(c, &c->write_kv, (size_t)R));
    TRY(dalloc(c, &c->U, sizeof(float) * (size_t)b * Wmax * d));
    TRY(dalloc(c, &c->act_last, sizeof(float) * (size_t)b * B * d));
    TRY(dalloc(c, &c->dec_rows, c->esz * (size_t)b * 2 * B * d));
    TRY(dalloc(c, &c->dec_ids, sizeof(int) * (size_t)b * 2 * B));
    TRY(dalloc(c, &c->dec_counts, sizeof(int) * 2 * (size_t)b));
    TRY(halloc(c, &c->dec_counts_h, sizeof(int) * 2 * (size_t)b));
    TRY(dalloc(c, &c->dn, sizeof(float) * (size_t)b * Wmax * d));
    TRY(dalloc(c, &c->sel_a, (size_t)b * Wmax));
    TRY(dalloc(c, &c->sel_b, (size_t)b * Wmax));
    CUDA_OR_FAIL(c, cudaMemset(c->sel_a, 0, (size_t)b * Wmax));
    CUDA_OR_FAIL(c, cudaMemset(c->sel_b, 0, (size_t)b * Wmax));
    TRY(dalloc(c, &c->o_src, sizeof(int) * (size_t)R));
    TRY(dalloc(c, &c->m_o, sizeof(int)));
    TRY(dalloc(c, &c->drift, sizeof(float) * (size_t)L * b * K));
    TRY(dalloc(c, &c->topk_out, sizeof(int) * (size_t)L * b * cfg->topk));
    TRY(dalloc(c, &c->selected, (size_t)L * b * Wmax));
    TRY(dalloc(c, &c->delta, sizeof(float) * (size_t)b * B));
    CUDA_OR_FAIL(c, cudaMemset(c->drift, 0, sizeof(float) * (size_t)L * b * K));
    CUDA_OR_FAIL(c, cudaMemset(c->topk_out, 0xFF, sizeof(int) * (size_t)L * b * cfg->topk));
    CUDA_OR_FAIL(c, cudaMemset(c->selected, 0, (size_t)L * b * Wmax));
    CUDA_OR_FAIL(c, cudaMemset(c->delta, 0, sizeof(float) * (size_t)b * B));
    TRY(dalloc(c, &c->conf, sizeof(float) * (size_t)b * 2 * B));
    TRY(dalloc(c, &c->drel, sizeof(float) * (size_t)b * 2 * B));
    TRY(dalloc(c, &c->taud, sizeof(float) * (size_t)b * 2 * B));
    TRY(dalloc(c, &c->commit_dev, (size_t)b * 2 * B));
    c->csplits = std::max(1, std::min(32, (2 * 152 + b * 2 * B - 1) / (b * 2 * B)));
    TRY(dalloc(c, &c->cpart, sizeof(float) * 2 * (size_t)b * 2 * B * c->csplits));
    c->ml = meta_layout(c->rows_cap, b, K, Wmax, N);
    TRY(halloc(c, &c->meta_h, c->ml.total));
    TRY(dalloc(c, &c->meta_d, c->ml.total));
    if (cfg->host_offload) {
      TRY(halloc(c, &c->codes_host, (size_t)L * b * Wmax * (d / 2)));
      TRY(halloc(c, &c->scales_host, (size_t)L * b * Wmax * (d / 16)));
      CUDA_OR_FAIL(c, cudaHostGetDevicePointer((void**)&c->codes_host_dev, c->codes_host, 0));
      CUDA_OR_FAIL(c, cudaHostGetDevicePointer((void**)&c->scales_host_dev, c->scales_host, 0));
    }
    CUDA_OR_FAIL(c, cudaDeviceSynchronize());
    return POLESTAR_OK;
  };
  const polestar_status st = run();
  if (st != POLESTAR_OK) {
    g_init_error = c->err;
    free_all(c);
    delete c;
    return st;
  }
  *out = c;
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_calibrate_step(polestar_ctx* c, const void* x0, const int32_t* n_unmasked,
                                                   int32_t block_index, int32_t block_entry,
                                                   polestar_step_out* out) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!x0) return fail(c, POLESTAR_ERR_INVALID_ARG, "x0 is NULL");
  if ((uintptr_t)x0 & 15) return fail(c, POLESTAR_ERR_INVALID_ARG, "x0 must be 16-byte aligned");
  const int n_blocks = c->cfg.gen_len / c->B;
  if (block_index < 0 || block_index >= n_blocks)
    return fail(c, POLESTAR_ERR_INVALID_ARG, "block_index out of range");
  if (!block_entry && c->cur_block != block_index)
    return fail(c, POLESTAR_ERR_STATE, "within-block step without the block's entry step");
  if (!block_entry && !n_unmasked) return fail(c, POLESTAR_ERR_INVALID_ARG, "n_unmasked is NULL");
  if (!block_entry)
    for (int s = 0; s < c->b; ++s)
      if (n_unmasked[s] < 0) return fail(c, POLESTAR_ERR_INVALID_ARG, "negative n_unmasked");
  // the host metadata buffer may still be in flight from the previous step
  CUDA_OR_FAIL(c, cudaEventSynchronize(c->meta_ev));
  TRY(check_timeouts(c));
  compute_window(c, block_index);
  polestar_status st = c->bf16 ? step_impl<__nv_bfloat16>(c, x0, n_unmasked, block_index, block_entry)
                               : step_impl<float>(c, x0, n_unmasked, block_index, block_entry);
  if (st != POLESTAR_OK) {
    c->stepped = 0;
    return st;
  }
  TRY(record_timeouts(c));
  c->cur_block = block_index;
  c->cur_entry = block_entry ? 1 : 0;
  c->stepped = 1;
  c->committed = 0;
  if (out) {
    out->drift = c->drift;
    out->topk = c->topk_out;
    out->selected = c->selected;
    out->labels = c->labels;
    out->delta = c->delta;
    out->fire = c->fire.data();
    out->win_len = c->nw;
    out->win_max = c->Wmax;
  }
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_commit(polestar_ctx* c, const float* logits, int32_t vocab,
                                           const uint8_t* masked, uint8_t* commit_mask, float* conf) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!logits || !masked || !commit_mask) return fail(c, POLESTAR_ERR_INVALID_ARG, "NULL buffer");
  if (vocab < 1) return fail(c, POLESTAR_ERR_INVALID_ARG, "vocab must be >= 1");
  if (!c->stepped) return fail(c, POLESTAR_ERR_STATE, "polestar_commit before polestar_calibrate_step");
  CommitArgs a{};
  a.logits = logits;
  a.V = vocab;
  a.batch = c->b;
  a.B = c->B;
  a.N = c->N;
  a.start = c->start;
  a.hist = c->cfg.hist;
  a.Wmax = c->Wmax;
  a.nw = c->nw;
  a.block_entry = c->cur_entry;
  a.tau_s = c->cfg.tau_s;
  a.tau_suf = c->cfg.tau_suf;
  a.alpha = c->cfg.alpha;
  a.masked = masked;
  a.delta = c->delta;
  a.theta = c->theta;
  a.theta_n = c->theta_n;
  a.fire = meta_d<uint8_t>(c, c->ml.fire_off);
  a.sel_last = c->sel_last ? c->sel_last : c->sel_a;
  a.win_pos = meta_d<int>(c, c->ml.win_pos_off);
  a.part = c->cpart;
  a.splits = c->csplits;
  a.commit = commit_mask;
  a.conf = c->conf;
  a.conf_user = conf;
  a.drel = c->drel;
  a.taud = c->taud;
  const int pi = prof_start(c, POLESTAR_KC_COMMIT);
  launch_commit(a, c->sm);
  prof_stop(c, pi, (double)c->b * 2 * c->B * vocab * 4.0, 0.0);
  c->launches += 2;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(c, POLESTAR_ERR_CUDA, std::string("commit launch: ") + cudaGetErrorString(e));
  c->stepped = 0;
  c->committed = 1;
  return POLESTAR_OK;
}

// ------------------------------------------------------------------ closed-loop decoding
namespace {
template <typename T>
polestar_status decode_logits_impl(polestar_ctx* c, const void* lm_head, const void* final_norm, int vocab,
                                   float* logits) {
  const int b = c->b, B = c->B, d = c->d;
  DecodeRowsArgs a{};
  a.act = c->cur_entry ? c->act_last : c->h_rows;
  a.U = c->U;
  a.sel = c->cur_entry ? nullptr : c->sel_last;
  a.fire = meta_d<uint8_t>(c, c->ml.fire_off);
  for (int i = 0; i < 64; ++i) a.suffix_widx[i] = -1;
  for (int w = 0; w < c->nw; ++w) {
    const int i = c->win_pos[w] - (c->start + B);
    if (i >= 0 && i < B) a.suffix_widx[i] = w;
  }
  a.batch = b;
  a.B = B;
  a.d = d;
  a.Wmax = c->Wmax;
  a.N = c->N;
  a.start = c->start;
  a.gain = final_norm;
  a.eps = c->cfg.rms_eps;
  a.out = c->dec_rows;
  RUN(POLESTAR_KC_ROWS, (double)b * 2 * B * d * (4 + c->esz), 0.0, (launch_decode_rows<T>(a, c->sm)));
  TRY(gemm<T>(c, c->dec_rows, d, lm_head, d, logits, vocab, b * 2 * B, nullptr, vocab, d));
  return POLESTAR_OK;
}
}  // namespace

extern "C" polestar_status polestar_decode_logits(polestar_ctx* c, const void* lm_head, const void* final_norm,
                                                  int32_t vocab, float* logits) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!lm_head || !final_norm || !logits) return fail(c, POLESTAR_ERR_INVALID_ARG, "NULL buffer");
  if (vocab < 1) return fail(c, POLESTAR_ERR_INVALID_ARG, "vocab must be >= 1");
  if (c->B > 64) return fail(c, POLESTAR_ERR_UNSUPPORTED, "block size above 64");
  if (!c->stepped) return fail(c, POLESTAR_ERR_STATE, "polestar_decode_logits needs a calibrate step not yet committed");
  c->gemm_cls = c->cur_entry ? POLESTAR_KC_GEMM_ENTRY : POLESTAR_KC_GEMM_STEP;
  return c->bf16 ? decode_logits_impl<__nv_bfloat16>(c, lm_head, final_norm, vocab, logits)
                 : decode_logits_impl<float>(c, lm_head, final_norm, vocab, logits);
}

extern "C" polestar_status polestar_decode_tokens(polestar_ctx* c, const float* logits, int32_t vocab,
                                                  uint8_t* commit_mask, int32_t* tokens, uint8_t* masked,
                                                  int32_t* n_committed, int32_t* n_block_masked) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!logits || !commit_mask || !tokens || !masked || !n_committed || !n_block_masked)
    return fail(c, POLESTAR_ERR_INVALID_ARG, "NULL buffer");
  if (vocab < 1) return fail(c, POLESTAR_ERR_INVALID_ARG, "vocab must be >= 1");
  if (!c->committed) return fail(c, POLESTAR_ERR_STATE, "polestar_decode_tokens needs a preceding polestar_commit");
  const int b = c->b, B = c->B;
  RUN(POLESTAR_KC_COMMIT, (double)b * 2 * B * vocab * 4.0, 0.0,
      (launch_argmax(logits, vocab, b * 2 * B, c->dec_ids, c->sm)));
  ApplyArgs a{};
  a.commit = commit_mask;
  a.conf = c->conf;
  a.ids = c->dec_ids;
  a.tokens = tokens;
  a.masked = masked;
  a.counts = c->dec_counts;
  a.batch = b;
  a.B = B;
  a.N = c->N;
  a.start = c->start;
  RUN(POLESTAR_KC_COMMIT, 0.0, 0.0, (launch_apply_commits(a, c->sm)));
  CUDA_OR_FAIL(c, cudaMemcpyAsync(c->dec_counts_h, c->dec_counts, sizeof(int) * 2 * b, cudaMemcpyDeviceToHost,
                                  c->sm));
  CUDA_OR_FAIL(c, cudaStreamSynchronize(c->sm));
  for (int s = 0; s < b; ++s) {
    n_committed[s] = c->dec_counts_h[2 * s];
    n_block_masked[s] = c->dec_counts_h[2 * s + 1];
  }
  c->committed = 0;
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_embed(polestar_ctx* c, const void* embed, int32_t vocab, const void* mask_emb,
                                          const int32_t* tokens, const uint8_t* masked, void* x0) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!embed || !mask_emb || !tokens || !masked || !x0) return fail(c, POLESTAR_ERR_INVALID_ARG, "NULL buffer");
  if (vocab < 1) return fail(c, POLESTAR_ERR_INVALID_ARG, "vocab must be >= 1");
  const int rows = c->b * c->N;
  const double eb = (double)rows * c->d * 2.0 * c->esz;  // one table row read, one input row written
  if (c->bf16)
    RUN(POLESTAR_KC_ROWS, eb, 0.0,
        (launch_embed<__nv_bfloat16>(embed, mask_emb, tokens, masked, vocab, rows, c->d, x0, c->sm)));
  else
    RUN(POLESTAR_KC_ROWS, eb, 0.0, (launch_embed<float>(embed, mask_emb, tokens, masked, vocab, rows, c->d, x0, c->sm)));
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_step_host(polestar_ctx* c, const void* x0_host, const int32_t* n_unmasked,
                                              int32_t block_index, int32_t block_entry, const float* logits_host,
                                              int32_t vocab, const uint8_t* masked_host,
                                              uint8_t* commit_mask_host) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!x0_host || !logits_host || !masked_host || !commit_mask_host)
    return fail(c, POLESTAR_ERR_INVALID_ARG, "NULL host buffer");
  if (vocab < 1) return fail(c, POLESTAR_ERR_INVALID_ARG, "vocab must be >= 1");
  const size_t x0_bytes = (size_t)c->b * c->N * c->d * c->esz;
  const size_t lg_bytes = (size_t)c->b * 2 * c->B * vocab * sizeof(float);
  if (!c->st_x0) {
    TRY(dalloc(c, &c->st_x0, x0_bytes));
    TRY(dalloc(c, &c->st_masked, (size_t)c->b * c->N));
    TRY(dalloc(c, &c->st_commit, (size_t)c->b * 2 * c->B));
  }
  if (lg_bytes > c->st_logits_cap) {
    TRY(dalloc(c, &c->st_logits, lg_bytes));
    c->st_logits_cap = lg_bytes;
  }
  if (!c->st_copy) {
    CUDA_OR_FAIL(c, cudaStreamCreateWithFlags(&c->st_copy, cudaStreamNonBlocking));
    CUDA_OR_FAIL(c, cudaEventCreateWithFlags(&c->st_copy_ev, cudaEventDisableTiming));
  }
  // the calibration step needs x0 first; the logits and mask only feed the
  // commit, so they are copied on the copy stream while the step computes
  // (the previous call's commit finished reading the staging buffers before
  // that call returned)
  CUDA_OR_FAIL(c, cudaMemcpyAsync(c->st_x0, x0_host, x0_bytes, cudaMemcpyHostToDevice, c->sm));
  CUDA_OR_FAIL(c, cudaMemcpyAsync(c->st_logits, logits_host, lg_bytes, cudaMemcpyHostToDevice, c->st_copy));
  CUDA_OR_FAIL(c, cudaMemcpyAsync(c->st_masked, masked_host, (size_t)c->b * c->N, cudaMemcpyHostToDevice,
                                  c->st_copy));
  CUDA_OR_FAIL(c, cudaEventRecord(c->st_copy_ev, c->st_copy));
  const polestar_status cs = polestar_calibrate_step(c, c->st_x0, n_unmasked, block_index, block_entry, nullptr);
  CUDA_OR_FAIL(c, cudaStreamWaitEvent(c->sm, c->st_copy_ev, 0));
  if (cs != POLESTAR_OK) {
    cudaStreamSynchronize(c->st_copy);
    return cs;
  }
  TRY(polestar_commit(c, c->st_logits, vocab, c->st_masked, c->st_commit, nullptr));
  CUDA_OR_FAIL(c, cudaMemcpyAsync(commit_mask_host, c->st_commit, (size_t)c->b * 2 * c->B, cudaMemcpyDeviceToHost,
                                  c->sm));
  CUDA_OR_FAIL(c, cudaStreamSynchronize(c->sm));
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_full_forward(polestar_ctx* c, const void* x0) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!x0) return fail(c, POLESTAR_ERR_INVALID_ARG, "x0 is NULL");
  if ((uintptr_t)x0 & 15) return fail(c, POLESTAR_ERR_INVALID_ARG, "x0 must be 16-byte aligned");
  // the host metadata buffer may still be in flight from the previous call
  CUDA_OR_FAIL(c, cudaEventSynchronize(c->meta_ev));
  TRY(check_timeouts(c));
  TRY(c->bf16 ? block_entry<__nv_bfloat16>(c, x0, 0, true) : block_entry<float>(c, x0, 0, true));
  TRY(record_timeouts(c));
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_kv_staleness(const void* kv, const void* kv_ref, int64_t rows, int32_t n_kv_heads,
                                                 int32_t head_dim, int32_t dtype, float* E, void* stream) {
  if (rows < 0 || n_kv_heads < 1 || head_dim < 8 || head_dim % 8) return POLESTAR_ERR_INVALID_ARG;
  if (dtype != POLESTAR_FP32 && dtype != POLESTAR_BF16) return POLESTAR_ERR_INVALID_ARG;
  if (rows == 0) return POLESTAR_OK;
  if (!kv || !kv_ref || !E) return POLESTAR_ERR_INVALID_ARG;
  if (((uintptr_t)kv | (uintptr_t)kv_ref) & 15) return POLESTAR_ERR_INVALID_ARG;
  if (rows > 0x7FFFFFFFLL) return POLESTAR_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  const cudaError_t e = dtype == POLESTAR_BF16
                            ? launch_kv_staleness<__nv_bfloat16>(kv, kv_ref, rows, n_kv_heads, head_dim, E, st)
                            : launch_kv_staleness<float>(kv, kv_ref, rows, n_kv_heads, head_dim, E, st);
  return e == cudaSuccess ? POLESTAR_OK : POLESTAR_ERR_CUDA;
}

extern "C" polestar_status polestar_cache_staleness(polestar_ctx* c, polestar_ctx* ref, float* E) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!ref || !E) return fail(c, POLESTAR_ERR_INVALID_ARG, "NULL reference context or output");
  if (ref == c) return fail(c, POLESTAR_ERR_INVALID_ARG, "the reference must be another context");
  if (ref->L != c->L || ref->b != c->b || ref->N != c->N || ref->Hkv != c->Hkv || ref->dh != c->dh ||
      ref->bf16 != c->bf16)
    return fail(c, POLESTAR_ERR_INVALID_ARG, "reference context has another cache shape or dtype");
  // the reference's cache is complete once its main stream reaches this point
  CUDA_OR_FAIL(c, cudaEventRecord(ref->main_ev, ref->sm));
  CUDA_OR_FAIL(c, cudaStreamWaitEvent(c->sm, ref->main_ev, 0));
  const long long rows = (long long)c->L * c->b * c->N;
  const int pi = prof_start(c, POLESTAR_KC_ROWS);
  const cudaError_t e = c->bf16 ? launch_kv_staleness<__nv_bfloat16>(c->kv, ref->kv, rows, c->Hkv, c->dh, E, c->sm)
                                : launch_kv_staleness<float>(c->kv, ref->kv, rows, c->Hkv, c->dh, E, c->sm);
  prof_stop(c, pi, (double)rows * 4 * c->kvdim * c->esz + (double)rows * 4.0, 0.0);
  if (e != cudaSuccess) return fail(c, POLESTAR_ERR_CUDA, std::string("staleness launch: ") + cudaGetErrorString(e));
  c->launches += 1;
  return POLESTAR_OK;
}

extern "C" void polestar_release(polestar_ctx* c) {
  if (!c) return;
  free_all(c);
  delete c;
}

extern "C" const char* polestar_last_error(const polestar_ctx* c) {
  return c ? c->err.c_str() : g_init_error.c_str();
}

extern "C" uint64_t polestar_launch_count(const polestar_ctx* c) { return c ? c->launches : 0; }

extern "C" polestar_status polestar_debug_read(polestar_ctx* c, int32_t which, int32_t layer, void* host_dst,
                                               size_t bytes) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!host_dst) return fail(c, POLESTAR_ERR_INVALID_ARG, "host_dst is NULL");
  const size_t L = c->L, b = c->b, N = c->N, d = c->d, Wmax = c->Wmax, K = c->K, H = c->H, B = c->B;
  const void* base = nullptr;
  size_t per = 0;
  bool layered = true;
  switch (which) {
    case POLESTAR_BUF_KV: base = c->kv; per = b * N * 2 * c->kvdim * c->esz; break;
    case POLESTAR_BUF_CENTROID: base = c->z; per = b * K * d * 4; break;
    case POLESTAR_BUF_CSUM: base = c->csum; per = b * K * d * 4; break;
    case POLESTAR_BUF_ANCHOR: base = c->anchor; per = b * K * d * 4; break;
    case POLESTAR_BUF_LABELS: base = c->labels; per = b * Wmax; break;
    case POLESTAR_BUF_CODES:
    case POLESTAR_BUF_SCALES: {
      const bool cd = which == POLESTAR_BUF_CODES;
      const size_t pl = cd ? code_layer_bytes(c) : scale_layer_bytes(c);
      if (layer < 0 || (size_t)layer >= L) return fail(c, POLESTAR_ERR_INVALID_ARG, "layer out of range");
      if (bytes > pl) return fail(c, POLESTAR_ERR_INVALID_ARG, "bytes exceeds the buffer size");
      if (c->offload) {  // the host store is authoritative
        CUDA_OR_FAIL(c, cudaStreamSynchronize(c->sm));
        CUDA_OR_FAIL(c, cudaStreamSynchronize(c->ss));
        std::memcpy(host_dst, (cd ? c->codes_host : c->scales_host) + (size_t)layer * pl, bytes);
        return POLESTAR_OK;
      }
      base = cd ? c->codes : c->scales;
      per = pl;
      break;
    }
    case POLESTAR_BUF_ACT_OUT: base = c->h_rows; per = b * B * d * 4; layered = false; break;
    case POLESTAR_BUF_UPDATE: base = c->U; per = b * Wmax * d * 4; layered = false; break;
    case POLESTAR_BUF_CONF: base = c->conf; per = b * 2 * B * 4; layered = false; break;
    case POLESTAR_BUF_DREL: base = c->drel; per = b * 2 * B * 4; layered = false; break;
    case POLESTAR_BUF_TAUD: base = c->taud; per = b * 2 * B * 4; layered = false; break;
    case POLESTAR_BUF_PROXY: base = c->pprev; per = b * K * H * N * 4; break;
    case POLESTAR_BUF_WINDOW_H: base = c->Hw; per = b * Wmax * d * 4; break;
    case POLESTAR_BUF_DRIFT: base = c->drift; per = b * K * 4; break;
    case POLESTAR_BUF_TOPK: base = c->topk_out; per = b * c->cfg.topk * 4; break;
    case POLESTAR_BUF_SELECTED: base = c->selected; per = b * Wmax; break;
    case POLESTAR_BUF_DELTA: base = c->delta; per = b * B * 4; layered = false; break;
    case POLESTAR_BUF_PROXY_LSE: base = c->pprev_lse; per = b * K * H * 4; break;
    case POLESTAR_BUF_ACTIVE_PREV: base = c->aprev; per = b * B * H * N * 4; layered = false; break;
    case POLESTAR_BUF_ACTIVE_LSE: base = c->aprev_lse; per = b * B * H * 4; layered = false; break;
    case POLESTAR_BUF_THETA: base = c->theta; per = b * B * std::max(1, c->cfg.hist) * 4; layered = false; break;
    case POLESTAR_BUF_THETA_N: base = c->theta_n; per = b * B * 4; layered = false; break;
    default: return fail(c, POLESTAR_ERR_INVALID_ARG, "unknown buffer id");
  }
  if (layered && (layer < 0 || (size_t)layer >= L)) return fail(c, POLESTAR_ERR_INVALID_ARG, "layer out of range");
  if (bytes > per) return fail(c, POLESTAR_ERR_INVALID_ARG, "bytes exceeds the buffer size");
  const char* src = (const char*)base + (layered ? (size_t)layer * per : 0);
  CUDA_OR_FAIL(c, cudaStreamSynchronize(c->sm));
  CUDA_OR_FAIL(c, cudaMemcpy(host_dst, src, bytes, cudaMemcpyDeviceToHost));
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_debug_write(polestar_ctx* c, int32_t which, int32_t layer, const void* host_src,
                                                size_t bytes) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!host_src) return fail(c, POLESTAR_ERR_INVALID_ARG, "host_src is NULL");
  const size_t L = c->L, b = c->b, N = c->N, d = c->d, Wmax = c->Wmax, K = c->K, H = c->H, B = c->B;
  void* base = nullptr;
  size_t per = 0;
  bool layered = true;
  switch (which) {
    case POLESTAR_BUF_KV: base = c->kv; per = b * N * 2 * c->kvdim * c->esz; break;
    case POLESTAR_BUF_CENTROID: base = c->z; per = b * K * d * 4; break;
    case POLESTAR_BUF_CSUM: base = c->csum; per = b * K * d * 4; break;
    case POLESTAR_BUF_ANCHOR: base = c->anchor; per = b * K * d * 4; break;
    case POLESTAR_BUF_LABELS: base = c->labels; per = b * Wmax; break;
    case POLESTAR_BUF_CODES:
    case POLESTAR_BUF_SCALES: {
      const bool cd = which == POLESTAR_BUF_CODES;
      const size_t pl = cd ? code_layer_bytes(c) : scale_layer_bytes(c);
      if (layer < 0 || (size_t)layer >= L) return fail(c, POLESTAR_ERR_INVALID_ARG, "layer out of range");
      if (bytes > pl) return fail(c, POLESTAR_ERR_INVALID_ARG, "bytes exceeds the buffer size");
      CUDA_OR_FAIL(c, cudaStreamSynchronize(c->sm));
      if (c->offload) {  // the host store is authoritative; the device ring refills from it
        CUDA_OR_FAIL(c, cudaStreamSynchronize(c->ss));
        std::memcpy((cd ? c->codes_host : c->scales_host) + (size_t)layer * pl, host_src, bytes);
        return POLESTAR_OK;
      }
      CUDA_OR_FAIL(c, cudaMemcpy((cd ? c->codes : c->scales) + (size_t)layer * pl, host_src, bytes,
                                 cudaMemcpyHostToDevice));
      return POLESTAR_OK;
    }
    case POLESTAR_BUF_PROXY: base = c->pprev; per = b * K * H * N * 4; break;
    case POLESTAR_BUF_PROXY_LSE: base = c->pprev_lse; per = b * K * H * 4; break;
    case POLESTAR_BUF_WINDOW_H: base = c->Hw; per = b * Wmax * d * 4; break;
    case POLESTAR_BUF_ACTIVE_PREV: base = c->aprev; per = b * B * H * N * 4; layered = false; break;
    case POLESTAR_BUF_ACTIVE_LSE: base = c->aprev_lse; per = b * B * H * 4; layered = false; break;
    case POLESTAR_BUF_THETA: base = c->theta; per = b * B * std::max(1, c->cfg.hist) * 4; layered = false; break;
    case POLESTAR_BUF_THETA_N: base = c->theta_n; per = b * B * 4; layered = false; break;
    default: return fail(c, POLESTAR_ERR_INVALID_ARG, "buffer is not part of the calibration state");
  }
  if (layered && (layer < 0 || (size_t)layer >= L)) return fail(c, POLESTAR_ERR_INVALID_ARG, "layer out of range");
  if (bytes > per) return fail(c, POLESTAR_ERR_INVALID_ARG, "bytes exceeds the buffer size");
  char* dst = (char*)base + (layered ? (size_t)layer * per : 0);
  CUDA_OR_FAIL(c, cudaStreamSynchronize(c->sm));
  CUDA_OR_FAIL(c, cudaMemcpy(dst, host_src, bytes, cudaMemcpyHostToDevice));
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_debug_enter_block(polestar_ctx* c, int32_t block_index, const int32_t* cum) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (block_index < 0 || block_index >= c->cfg.gen_len / c->B)
    return fail(c, POLESTAR_ERR_INVALID_ARG, "block_index out of range");
  for (int s = 0; cum && s < c->b; ++s)
    if (cum[s] < 0) return fail(c, POLESTAR_ERR_INVALID_ARG, "negative count");
  CUDA_OR_FAIL(c, cudaStreamSynchronize(c->sm));
  compute_window(c, block_index);
  for (int s = 0; s < c->b; ++s) {
    c->cum[s] = cum ? cum[s] : 0;
    c->fire[s] = 0;
  }
  c->sel_last = nullptr;
  c->cur_block = block_index;
  c->cur_entry = 1;
  c->stepped = 0;
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_profile_begin(polestar_ctx* c, int32_t capacity) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (capacity < 1) return fail(c, POLESTAR_ERR_INVALID_ARG, "capacity must be >= 1");
  CUDA_OR_FAIL(c, cudaStreamSynchronize(c->sm));
  prof_release(c);
  c->prof_ev.resize(2 * (size_t)capacity);
  for (size_t i = 0; i < c->prof_ev.size(); ++i) {
    cudaError_t e = cudaEventCreate(&c->prof_ev[i]);
    if (e != cudaSuccess) {
      c->prof_ev.resize(i);
      prof_release(c);
      return fail(c, POLESTAR_ERR_CUDA, std::string("cudaEventCreate: ") + cudaGetErrorString(e));
    }
  }
  c->prof_rec.assign(capacity, polestar_ctx::ProfRec{0, 0.0, 0.0});
  {
    cudaError_t e = cudaHostAlloc(&c->prof_rows, sizeof(int) * (size_t)capacity, cudaHostAllocDefault);
    if (e != cudaSuccess) {
      c->prof_rows = nullptr;
      prof_release(c);
      return fail(c, POLESTAR_ERR_OOM, std::string("cudaHostAlloc: ") + cudaGetErrorString(e));
    }
  }
  c->prof_cap = capacity;
  c->prof_used = 0;
  for (auto& d : c->prof_dropped) d = 0;
  c->prof_armed = true;
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_profile_end(polestar_ctx* c, polestar_kernel_stats* out, int32_t n_classes) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (!c->prof_armed) return fail(c, POLESTAR_ERR_STATE, "profiling is not armed");
  if (!out || n_classes < 1) return fail(c, POLESTAR_ERR_INVALID_ARG, "bad output array");
  CUDA_OR_FAIL(c, cudaStreamSynchronize(c->sm));
  for (int k = 0; k < n_classes; ++k) out[k] = polestar_kernel_stats{0, 0.0, 0.0, 0.0, 0};
  for (int i = 0; i < c->prof_used; ++i) {
    const auto& r = c->prof_rec[i];
    if (r.cls >= n_classes) continue;
    float ms = 0.f;
    CUDA_OR_FAIL(c, cudaEventElapsedTime(&ms, c->prof_ev[2 * i], c->prof_ev[2 * i + 1]));
    out[r.cls].launches += 1;
    out[r.cls].ms += ms;
    const double rows = r.device_rows ? (double)std::min(std::max(c->prof_rows[i], 0), r.max_rows) : (double)r.max_rows;
    out[r.cls].bytes += r.bytes + rows * r.row_bytes;
    out[r.cls].flops += r.flops + rows * r.row_flops;
  }
  for (int k = 0; k < n_classes && k < POLESTAR_KC_COUNT; ++k) out[k].dropped = c->prof_dropped[k];
  prof_release(c);
  return POLESTAR_OK;
}

extern "C" polestar_status polestar_debug_gemm(const void* A, int32_t lda, const void* W, int32_t ldw, float* C,
                                               int32_t ldc, int32_t M, const int32_t* m_dev, int32_t N, int32_t K,
                                               int32_t dtype, int32_t path, void* stream) {
  static TcGemmCache cache;
  if (!A || !W || !C || M < 0 || N < 1 || K < 1) return POLESTAR_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const int kind = path & 0xF;
  if (kind == 1 || kind == 2 || kind == 3 || kind == 7) {
    if (dtype != POLESTAR_BF16 || !tc_gemm_supported(K, lda, ldw)) return POLESTAR_ERR_UNSUPPORTED;
    TcGemmChoice force;
    force.kernel = kind == 7 ? 5 : kind - 1;
    force.kpack = (path >> 4) & 0xF;
    force.stages = (path >> 8) & 0xFF;
    force.splits = (path >> 16) & 0xFF;
    force.bn = ((path >> 24) & 0xFF) * 16;
    const cudaError_t e = tc_gemm_bf16(&cache, A, lda, W, ldw, C, ldc, M, m_dev, N, K, st, &force);
    if (e == cudaErrorInvalidValue) return POLESTAR_ERR_UNSUPPORTED;
    return e == cudaSuccess ? POLESTAR_OK : POLESTAR_ERR_CUDA;
  }
  if (kind != 0) return POLESTAR_ERR_UNSUPPORTED;
  if (dtype == POLESTAR_BF16)
    launch_gemm_simt<__nv_bfloat16>(A, lda, W, ldw, C, ldc, M, m_dev, N, K, st);
  else
    launch_gemm_simt<float>(A, lda, W, ldw, C, ldc, M, m_dev, N, K, st);
  return cudaGetLastError() == cudaSuccess ? POLESTAR_OK : POLESTAR_ERR_CUDA;
}

extern "C" polestar_status polestar_debug_gemm_swiglu(const void* A, int32_t lda, const void* Wg, const void* Wu,
                                                      int32_t ldw, void* act, int32_t ld_act, int32_t M,
                                                      const int32_t* m_dev, int32_t F, int32_t K, int32_t path,
                                                      void* stream) {
  static TcGemmCache cache;
  if (!A || !Wg || !Wu || !act || M < 0 || F < 1 || K < 1 || ld_act < F) return POLESTAR_ERR_INVALID_ARG;
  const int kind = path & 0xF;
  if (kind != 1 && kind != 2 && kind != 7) return POLESTAR_ERR_UNSUPPORTED;
  if (!tc_gemm_supported(K, lda, ldw)) return POLESTAR_ERR_UNSUPPORTED;
  TcGemmChoice force;
  force.kernel = kind == 2 ? 1 : (kind == 7 ? 5 : 0);
  force.stages = (path >> 8) & 0xFF;
  force.splits = (path >> 16) & 0xFF;
  force.bn = ((path >> 24) & 0xFF) * 16;
  const cudaError_t e = tc_gemm_bf16_swiglu(&cache, A, lda, Wg, Wu, ldw, F, act, ld_act, M, m_dev, K,
                                            (cudaStream_t)stream, kind != 1 ? &force : nullptr);
  if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) return POLESTAR_ERR_UNSUPPORTED;
  return e == cudaSuccess ? POLESTAR_OK : POLESTAR_ERR_CUDA;
}

extern "C" polestar_status polestar_debug_gemm_choice(int32_t M, int32_t nseg, const int32_t* N, int32_t K,
                                                      int32_t* out) {
  static TcGemmCache cache;
  if (!N || !out || M < 1 || nseg < 1 || nseg > 3 || K < 1) return POLESTAR_ERR_INVALID_ARG;
  return tc_gemm_choice(&cache, M, nseg, N, K, out) == cudaSuccess ? POLESTAR_OK : POLESTAR_ERR_CUDA;
}

namespace {
polestar_status debug_attention(const void* q, const void* kv, int batch, int N, int H, int Hkv, int head_dim, int R,
                                const uint8_t* tracked, float* prev, float* prev_lse, int measure, int store,
                                void* out, float* kl, int dtype, cudaStream_t st) {
  if (!q || !kv || !out || batch < 1 || R < 1 || N < 1 || H < 1 || Hkv < 1 || H % Hkv) return POLESTAR_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return POLESTAR_ERR_UNSUPPORTED;
  bool any_tracked = false;
  for (int r = 0; tracked && r < R; ++r) any_tracked |= tracked[r] != 0;
  if (any_tracked && (!prev || !prev_lse || (measure && !kl))) return POLESTAR_ERR_INVALID_ARG;
  const size_t rows_total = (size_t)batch * R;
  std::vector<int4> rows(rows_total), work;
  for (int s = 0; s < batch; ++s)
    for (int r = 0; r < R; ++r)
      rows[(size_t)s * R + r] = make_int4(s, 0, (tracked && tracked[r]) ? ROW_ACTIVE : ROW_OTHER, r);
  const int item_rows = attention_item_rows(dtype == POLESTAR_BF16, head_dim,
                                            (long long)batch * ((R + ATT_TC_ROWS - 1) / ATT_TC_ROWS), H,
                                            any_tracked && measure, true);
  work.resize((size_t)batch * ((R + item_rows - 1) / item_rows));
  int nw = 0;
  for (int s = 0; s < batch; ++s) nw = attention_items(work.data(), nw, s * R, R, 0, 0, item_rows);
  work.resize(nw);
  int4* d_rows = nullptr;
  int4* d_work = nullptr;
  if (cudaMalloc(&d_rows, sizeof(int4) * rows_total) != cudaSuccess) return POLESTAR_ERR_OOM;
  if (cudaMalloc(&d_work, sizeof(int4) * work.size()) != cudaSuccess) {
    cudaFree(d_rows);
    return POLESTAR_ERR_OOM;
  }
  cudaMemcpy(d_rows, rows.data(), sizeof(int4) * rows_total, cudaMemcpyHostToDevice);
  cudaMemcpy(d_work, work.data(), sizeof(int4) * work.size(), cudaMemcpyHostToDevice);
  // drift measured as in the layer loop: the attention writes the tracked rows'
  // new scores, the drift pass compares them with prev and replaces those
  const bool defer = any_tracked && measure;
  std::vector<int4> track;
  if (defer)
    for (int s = 0; s < batch; ++s)
      for (int r = 0; r < R; ++r)
        if (tracked[r]) track.push_back(make_int4(s * R + r, s, ROW_ACTIVE, r));
  float* d_new = nullptr;
  float* d_new_lse = nullptr;
  int4* d_track = nullptr;
  auto release = [&]() {
    cudaFree(d_rows);
    cudaFree(d_work);
    if (d_new) cudaFree(d_new);
    if (d_new_lse) cudaFree(d_new_lse);
    if (d_track) cudaFree(d_track);
  };
  if (defer) {
    if (cudaMalloc(&d_new, sizeof(float) * rows_total * H * N) != cudaSuccess ||
        cudaMalloc(&d_new_lse, sizeof(float) * rows_total * H) != cudaSuccess ||
        cudaMalloc(&d_track, sizeof(int4) * track.size()) != cudaSuccess) {
      release();
      return POLESTAR_ERR_OOM;
    }
    cudaMemcpy(d_track, track.data(), sizeof(int4) * track.size(), cudaMemcpyHostToDevice);
  }
  AttnArgs a{};
  a.q = q;
  a.ldq = H * head_dim;
  a.rows = d_rows;
  a.R = (int)rows_total;
  a.kv_layer = kv;
  a.kv_seq_stride = (size_t)N * 2 * Hkv * head_dim;
  a.kvdim = Hkv * head_dim;
  a.N = N;
  a.H = H;
  a.Hkv = Hkv;
  a.dh = head_dim;
  a.K = 1;
  a.B = R;
  a.scale = 1.f / sqrtf((float)head_dim);
  a.out = out;
  a.ldo = H * head_dim;
  a.other_live = 1;
  a.active_prev = any_tracked ? prev : nullptr;
  a.active_prev_lse = any_tracked ? prev_lse : nullptr;
  a.measure = measure;
  a.store = store;
  a.kl_out = kl;
  a.work = d_work;
  a.n_work = (int)work.size();
  a.item_rows = item_rows;
  a.batch = batch;
  if (defer) {
    a.active_new = d_new;
    a.active_new_lse = d_new_lse;
  }
  cudaError_t e = dtype == POLESTAR_BF16 ? launch_row_attention<__nv_bfloat16>(a, st) : launch_row_attention<float>(a, st);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess && defer) {
    DriftArgs da{};
    da.track = d_track;
    da.n_track = (int)track.size();
    da.H = H;
    da.N = N;
    da.K = 1;
    da.B = R;
    da.active_prev = prev;
    da.active_prev_lse = prev_lse;
    da.active_new = d_new;
    da.active_new_lse = d_new_lse;
    da.kl_out = kl;
    da.store = store;
    launch_drift(da, st);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  release();
  return e == cudaSuccess ? POLESTAR_OK : POLESTAR_ERR_CUDA;
}
}  // namespace

extern "C" polestar_status polestar_debug_attention(const void* q, const void* kv, int32_t N, int32_t H,
                                                    int32_t Hkv, int32_t head_dim, int32_t R,
                                                    const uint8_t* tracked, float* prev, float* prev_lse,
                                                    int32_t measure, int32_t store, void* out, float* kl,
                                                    int32_t dtype, void* stream) {
  return debug_attention(q, kv, 1, N, H, Hkv, head_dim, R, tracked, prev, prev_lse, measure, store, out, kl, dtype,
                         (cudaStream_t)stream);
}

extern "C" polestar_status polestar_debug_attention_batch(const void* q, const void* kv, int32_t batch, int32_t N,
                                                          int32_t H, int32_t Hkv, int32_t head_dim, int32_t R,
                                                          const uint8_t* tracked, float* prev, float* prev_lse,
                                                          int32_t measure, int32_t store, void* out, float* kl,
                                                          int32_t dtype, void* stream) {
  return debug_attention(q, kv, batch, N, H, Hkv, head_dim, R, tracked, prev, prev_lse, measure, store, out, kl, dtype,
                         (cudaStream_t)stream);
}

extern "C" int32_t polestar_debug_window(int32_t prompt_len, int32_t gen_len, int32_t block, int32_t prefix_win,
                                        int32_t suffix_win, int32_t block_index, int32_t* span, int32_t* pos,
                                        int32_t cap) {
  if (prompt_len < 0 || gen_len < 1 || block < 1 || gen_len % block || prefix_win < 0 || suffix_win < 0 ||
      block_index < 0 || block_index >= gen_len / block || !span || cap < 0 || (cap > 0 && !pos))
    return -1;
  std::vector<int> w;
  int start = 0, end = 0;
  window_of(prompt_len, prompt_len + gen_len, block, prefix_win, suffix_win, block_index, &start, &end, w);
  if ((int)w.size() > cap) return -1;
  span[0] = start;
  span[1] = end;
  for (size_t i = 0; i < w.size(); ++i) pos[i] = w[i];
  return (int32_t)w.size();
}

extern "C" polestar_status polestar_debug_stalled_wait(polestar_ctx* c, int64_t limit_cycles) {
  if (!c) return POLESTAR_ERR_INVALID_ARG;
  if (limit_cycles < 1) return fail(c, POLESTAR_ERR_INVALID_ARG, "limit_cycles must be positive");
  int* err = tc_error_word(&c->tc);
  if (!err) return fail(c, POLESTAR_ERR_OOM, "device error word");
  const cudaError_t e = tc_debug_stalled_wait(err, 99, (long long)limit_cycles, c->sm);
  if (e != cudaSuccess) return fail(c, POLESTAR_ERR_CUDA, std::string("stalled wait: ") + cudaGetErrorString(e));
  return record_timeouts(c);
}

extern "C" polestar_status polestar_debug_trigger(int32_t tau_upd, const int32_t* n_unmasked, int32_t steps,
                                                  uint8_t* fire) {
  if (steps < 0 || (steps > 0 && (!n_unmasked || !fire))) return POLESTAR_ERR_INVALID_ARG;
  int cum = 0;
  for (int t = 0; t < steps; ++t) {
    if (n_unmasked[t] < 0) return POLESTAR_ERR_INVALID_ARG;
    fire[t] = trigger_step(cum, n_unmasked[t], tau_upd) ? 1 : 0;
  }
  return POLESTAR_OK;
}

extern "C" int32_t polestar_debug_attention_items(int32_t a0, int32_t na, int32_t b0, int32_t nb, int32_t max_rows,
                                                 int32_t* out, int32_t cap) {
  if (na < 0 || nb < 0 || max_rows < 1 || cap < 0 || (cap > 0 && !out)) return -1;
  const int tot = na + nb;
  const int k = tot > 0 ? (tot + max_rows - 1) / max_rows : 0;
  if (k > cap) return -1;
  std::vector<int4> w((size_t)k + 1);
  const int n = attention_items(w.data(), 0, a0, na, b0, nb, max_rows);
  for (int i = 0; i < n; ++i) {
    out[4 * i + 0] = w[i].x;
    out[4 * i + 1] = w[i].y;
    out[4 * i + 2] = w[i].z;
    out[4 * i + 3] = w[i].w;
  }
  return n;
}

extern "C" int32_t polestar_debug_qkv_fusion(int32_t on) {
  const int32_t old = g_qkv_fusion ? 1 : 0;
  g_qkv_fusion = on != 0;
  return old;
}

extern "C" int32_t polestar_debug_attention_impl(int32_t impl) {
  if (impl < 0 || impl > 2) return -1;
  return attention_set_impl(impl);
}

extern "C" polestar_status polestar_debug_kmeans(const float* Hw, int32_t P, int32_t nw, int32_t d, int32_t K,
                                                 int32_t iters, uint64_t seed, int32_t block, uint8_t* labels,
                                                 float* z, float* csum, float* anchor, uint8_t* codes,
                                                 uint8_t* scales, void* stream) {
  if (!Hw || !labels || !z || !csum || !anchor || !codes || !scales || P < 1 || iters < 1)
    return POLESTAR_ERR_INVALID_ARG;
  if (nw < 1 || nw > 128 || K < 1 || K > 8 || K > nw || d < 16 || d % 16 || d > 4096 ||
      kmeans_cluster_size(d, nw, K) < 0)
    return POLESTAR_ERR_UNSUPPORTED;
  KmeansArgs a{};
  a.Hw = Hw;
  a.L = P;
  a.batch = 1;
  a.Wmax = nw;
  a.nw = nw;
  a.d = d;
  a.K = K;
  a.iters = iters;
  a.seed = seed;
  a.block = block;
  a.labels = labels;
  a.z = z;
  a.csum = csum;
  a.anchor = anchor;
  a.codes = codes;
  a.scales = scales;
  cudaStream_t st = (cudaStream_t)stream;
  launch_kmeans_encode(a, st);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? POLESTAR_OK : POLESTAR_ERR_CUDA;
}
