// Internal launch interface of the Polestar kernels (not part of the C ABI).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "common.cuh"

namespace polestar {

// Launch with programmatic dependent launch enabled (see pdl_enter()).
template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- row kernels (k_rows.cu) ----
// gain != nullptr also writes a[r] = T(RMSNorm(h[r]) * gain)
template <typename T>
void launch_gather_input(const void* x0, const int4* rows, int R, int N, int d, float* h, cudaStream_t st,
                         const void* gain = nullptr, float eps = 0.f, void* a = nullptr);
template <typename T>
void launch_gather_window(const void* x0, const int* win_pos, int nw, const int* fire_seqs, int n_fire, int N,
                          int d, int Wmax, float* U, uint8_t* sel, cudaStream_t st);
template <typename T>
void launch_rmsnorm(const float* h, const int* src, const int* m_dev, const int4* rows, const float* z, int K,
                    const void* gain, int R, int d, float eps, void* a, cudaStream_t st);
template <typename T>
void launch_rope_scatter(const float* qkv, int ldq, const int4* rows, const uint8_t* write_kv, int R, int H,
                         int Hkv, int dh, const float2* tab, void* qout, void* kv_layer, size_t kv_seq_stride,
                         int kvdim, cudaStream_t st);
template <typename T>
void launch_residual_rmsnorm(const float* h, const int* src, const int* m_dev, int R, const float* y, int ldy,
                             const void* gain, int d, float eps, float* h1, void* a, cudaStream_t st);
template <typename T>
void launch_swiglu(const float* gu, int ldg, const int* m_dev, int R, int F, void* act, cudaStream_t st);
// gain != nullptr: rows written to h also get an[row] = T(RMSNorm(out) * gain)
template <typename T>
void launch_residual_scatter(const float* h1, const float* y, int ldy, const int* src, const int* m_dev, int R,
                             const int4* rows, int d, int Wmax, float* h, float* U, cudaStream_t st,
                             const void* gain = nullptr, float eps = 0.f, void* an = nullptr);
template <typename T>
void launch_gather_T(const void* src, const int* idx, const int* m_dev, int R, int w, void* dst,
                     cudaStream_t st);
// ---- closed-loop decoding (k_decode.cu) ----
struct DecodeRowsArgs {
  const float* act;        // [batch, B, d] last-layer outputs of the active rows
  const float* U;          // [batch, Wmax, d] update packets U(t, L)
  const uint8_t* sel;      // [batch, Wmax] rows the last layer refreshed (null: none)
  const uint8_t* fire;     // [batch] sequences whose window the step refreshed
  int suffix_widx[64];     // window index of position start + B + i, or -1
  int batch, B, d, Wmax, N, start;
  const void* gain;        // [d] final norm gain (storage type)
  float eps;
  void* out;               // [batch * 2B, d] storage type: the LM head's input rows
};
struct ApplyArgs {
  uint8_t* commit;         // [batch, 2B] commit mask, progress rule applied in place
  const float* conf;       // [batch, 2B]
  const int* ids;          // [batch, 2B] greedy tokens
  int* tokens;             // [batch, N]
  uint8_t* masked;         // [batch, N]
  int* counts;             // [batch, 2]: tokens committed this step, current-block tokens still masked
  int batch, B, N, start;
};
template <typename T>
void launch_decode_rows(const DecodeRowsArgs& a, cudaStream_t st);
void launch_argmax(const float* logits, int V, int R, int* ids, cudaStream_t st);
void launch_apply_commits(const ApplyArgs& a, cudaStream_t st);
template <typename T>
void launch_embed(const void* embed, const void* mask_emb, const int* tokens, const uint8_t* masked, int vocab,
                  int rows, int d, void* x0, cudaStream_t st);
void launch_capture_active(const float* h, const int4* rows, int R, int d, int B, float* act, cudaStream_t st);

void launch_capture_window(const float* h, const int4* rows, int R, int d, int Wmax, float* Hw_layer,
                           size_t seq_stride, cudaStream_t st);

// ---- attention + KL (k_attention.cu) ----
struct AttnArgs {
  const void* q;           // [R, ldq] storage type, rotary applied
  int ldq;
  const int4* rows;        // [R] {seq, pos, kind, aux}
  int R;
  const void* kv_layer;    // layer base of the K/V cache; seq stride below
  size_t kv_seq_stride;    // elements between sequences
  int kvdim;               // Hkv * dh
  int N, H, Hkv, dh, K, B;
  float scale;             // 1/sqrt(dh)
  void* out;               // [R, ldo] storage type (not written for proxy rows)
  int ldo;
  int other_live;
  // drift tracking (nullptr = off)
  float* proxy_prev;       // [batch, K, H, N] scores of this layer's proxies
  float* proxy_prev_lse;   // [batch, K, H]
  float* active_prev;      // [batch, B, H, N] scores of the active rows (last layer)
  float* active_prev_lse;  // [batch, B, H]
  int measure;             // 1: write KL(new || prev) to kl_out[r, h]
  int store;               // 1: replace prev by the new scores
  float* kl_out;           // [R, H]
  // deferred drift (all four set, with measure): a tracked row's new scores and
  // log-sum-exp go to these buffers (the layout of the *_prev ones) and the
  // kernel neither reads *_prev nor computes KL; launch_drift then does both
  float* proxy_new;        // [batch, K, H, N]
  float* proxy_new_lse;    // [batch, K, H]
  float* active_new;       // [batch, B, H, N]
  float* active_new_lse;   // [batch, B, H]
  // bf16 tensor-core path: work list of items {rowA, nA, rowB, nB}, each the
  // rows [rowA, rowA + nA) and [rowB, rowB + nB) of ONE sequence, at most
  // ATT_ITEM_ROWS in all (nullptr: CUDA-core path by rows)
  const int4* work;
  int n_work;
  int batch;               // sequences in the K/V view of kv_layer
  // set by the launcher: key ranges per (item, head) (a thread-block cluster
  // whose partials meet in distributed shared memory) and K/V ring depth
  int splits;
  int stages;
  int* err;                // device word for the code of a timed-out wait (may be null)
  int item_rows;           // rows per work item the list was built with (ATT_ITEM_ROWS or ATT_TC_ROWS)
};
constexpr int ATT_ITEM_ROWS = 48;  // pipelined mma.sync kernel: 3 compute warps x 16 rows
constexpr int ATT_TC_ROWS = 128;   // tcgen05 kernel: one TMEM lane per row
// Work items for the rows [a0, a0 + na) ++ [b0, b0 + nb) of one sequence,
// appended at w[n..]; returns the new count (items of near-equal size, at most
// max_rows rows each).
int attention_items(int4* w, int n, int a0, int na, int b0, int nb, int max_rows = ATT_ITEM_ROWS);
// Rows per work item for a bf16/fp32 launch with head size dh whose items, at
// ATT_TC_ROWS rows, would number about `items128` (all sequences) over H
// heads, `measures` when some rows compute KL drift and `deferred` when that
// drift goes to the deferred drift pass: ATT_TC_ROWS when the tcgen05 kernel
// runs it (bf16, head size 128, no in-kernel drift, and either selected
// through attention_set_impl or enough items to fill every SM twice), else
// ATT_ITEM_ROWS.
int attention_item_rows(bool bf16, int dh, long long items128, int H, bool measures, bool deferred = false);

// ---- KL drift of tracked rows from their new and previous scores (k_drift.cu) ----
// Eq. 4 for each tracked (row, head): KL(softmax(new) || softmax(prev)) from the
// scores an attention launch wrote in deferred mode; with store, the new scores
// and log-sum-exps then replace the previous ones.
struct DriftArgs {
  const int4* track;       // [n_track] {step row r (kl_out row), seq, kind (ROW_PROXY / ROW_ACTIVE), idx}
  int n_track;
  int H, N, K, B;
  float* proxy_prev;       // [batch, K, H, N] / [batch, K, H]
  float* proxy_prev_lse;
  float* active_prev;      // [batch, B, H, N] / [batch, B, H]
  float* active_prev_lse;
  const float* proxy_new;  // same layouts: this step's scores
  const float* proxy_new_lse;
  const float* active_new;
  const float* active_new_lse;
  float* kl_out;           // [rows, H]
  int store;
};
void launch_drift(const DriftArgs& a, cudaStream_t st);
// Test hook: 0 = library's choice, 1 = pipelined mma.sync kernel only, 2 =
// tcgen05 kernel wherever it applies; returns the previous setting.
int attention_set_impl(int impl);
cudaError_t launch_attention_tc(const AttnArgs& a, int batch, cudaStream_t st);
// Key splits and ring depth of the pipelined bf16 kernel for a grid of n_work
// items x H heads.
int attention_pipe_config(int n_work, int H, int N, int dh, int num_sms, int* stages);
cudaError_t launch_attention_pipe(const AttnArgs& a, int batch, cudaStream_t st);
template <typename T>
cudaError_t launch_row_attention(const AttnArgs& a, cudaStream_t st);

// ---- K-means + NVFP4 (k_cluster.cu) ----
struct KmeansArgs {
  const float* Hw;         // [L, batch, Wmax, d] block-entry layer inputs of window rows
  int L, batch, Wmax, nw, d, K, iters;
  int layer0;              // first layer of this launch (it covers layers layer0 .. layer0 + L - 1)
  uint64_t seed;
  int block;
  uint8_t* labels;         // [L, batch, Wmax]
  float* z;                // [L, batch, K, d]
  float* csum;             // [L, batch, K, d]
  float* anchor;           // [L, batch, K, d]
  uint8_t* codes;          // [L, batch, Wmax, d/2] of this launch's layers (from layer0)
  uint8_t* scales;         // [L, batch, Wmax, d/16]
};
void launch_kmeans_encode(const KmeansArgs& a, cudaStream_t st);
// Thread-block cluster size of the K-means kernel for this shape (-1: unsupported).
int kmeans_cluster_size(int d, int nw, int K);

// Within-block patch of layer l's window cache (Algorithm 1, Dequantize + Patch steps):
// decode every window row of each firing sequence, replace the rows of the
// previous layer's selection by their update packet, re-encode those rows,
// and write the patched hidden states into the step's row space.
struct PatchArgs {
  const int* fire_seqs;    // [n_fire]
  int n_fire, nw, Wmax, d, K;
  const uint8_t* labels;   // layer base [batch, Wmax]
  const float* anchor;     // layer base [batch, K, d]
  uint8_t* codes;          // layer base [batch, Wmax, d/2]
  uint8_t* scales;         // layer base [batch, Wmax, d/16]
  const float* U;          // [batch, Wmax, d]
  const uint8_t* sel_prev; // [batch, Wmax]
  const int* win_row;      // [batch] first row of the sequence's window rows in the step row space (-1: none)
  float* h_rows;           // [R, d]
  uint8_t* write_kv;       // [R]
  float* dn;               // [batch, Wmax, d]: normalise(new) - normalise(old) for patched rows
  float* csum;             // layer base [batch, K, d]
  float* z;                // layer base [batch, K, d]
  // fused projection input: a_out[row] = T(RMSNorm(row) * gain) for every
  // patched window row and every proxy row (proxy rows start at proxy_row[s])
  const void* gain;
  float eps;
  void* a_out;
  const int* proxy_row;
};
template <typename T>
void launch_window_patch(const PatchArgs& a, cudaStream_t st);
template <typename T>
void launch_centroid_update(const PatchArgs& a, cudaStream_t st);

// ---- selection (k_select.cu) ----
struct SelectArgs {
  int batch, Wmax, nw, K, topk, H, B;
  const float* kl_rows;    // [R, H]
  const int* proxy_row;    // [batch] first proxy row of the sequence (-1: not refreshing)
  const int* win_row;      // [batch] first window row (-1)
  const uint8_t* labels;   // layer base [batch, Wmax]
  float* drift;            // layer base [batch, K]
  int* topk_out;           // layer base [batch, topk]
  uint8_t* selected;       // layer base [batch, Wmax]
  uint8_t* sel_cur;        // [batch, Wmax]
  int* o_src;              // [R] compact row list (active rows then selected window rows)
  int* m_o;                // [1]
  int n_active;            // batch * B
};
void launch_select(const SelectArgs& a, cudaStream_t st);
void launch_delta_finalize(const float* kl_rows, int batch, int B, int H, float* delta, cudaStream_t st);

// ---- commit (k_commit.cu) ----
struct CommitArgs {
  const float* logits;     // [batch, 2B, V]
  int V, batch, B, N, start, hist, Wmax, nw, block_entry;
  float tau_s, tau_suf, alpha;
  const uint8_t* masked;   // [batch, N]
  const float* delta;      // [batch, B]
  float* theta;            // [batch, B, hist]
  int* theta_n;            // [batch, B]
  const uint8_t* fire;     // device [batch]
  const uint8_t* sel_last; // [batch, Wmax] last-layer selection
  const int* win_pos;      // [nw]
  float* part;             // [batch*2B, splits, 2]
  int splits;
  uint8_t* commit;         // [batch, 2B]
  float* conf;             // [batch, 2B]
  float* conf_user;        // optional copy
  float* drel;             // [batch, 2B]
  float* taud;             // [batch, 2B]
};
void launch_commit(const CommitArgs& a, cudaStream_t st);

// ---- KV-cache staleness (k_staleness.cu) ----
// E[r] = 1 - (mean_h cos(K_r^h, Kref_r^h) + mean_h cos(V_r^h, Vref_r^h)) / 2 over
// rows laid out [rows][2][Hkv * dh] (K then V); dh a multiple of 8, both
// buffers 16-byte aligned.
template <typename T>
cudaError_t launch_kv_staleness(const void* kv, const void* ref, long long rows, int Hkv, int dh, float* E,
                                cudaStream_t st);

// ---- GEMM: C[M, N] (fp32, ldc) = A[M, K] (T, lda) * W[N, K]^T (T, ldw) ----
// m_dev (nullable): device row count; rows >= min(M, *m_dev) are not computed.
template <typename T>
void launch_gemm_simt(const void* A, int lda, const void* W, int ldw, float* C, int ldc, int M, const int* m_dev,
                      int N, int K, cudaStream_t st);

}  // namespace polestar
