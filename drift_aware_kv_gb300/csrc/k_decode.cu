// Closed-loop decoding around the calibrated layer loop ("Polestar: Drift-Aware
// Cache Calibration and Token Commitment for Efficient Inference of Diffusion
// LLMs", Algorithm 1 in full, Eq. 1 greedy reconstruction, App. D.1 accounting):
//   * the rows the commit gate scores -- the active block's last-layer outputs
//     and the suffix block's refreshed update packets U(t, L) -- normalised
//     with the final RMSNorm into the LM head's input rows;
//   * the greedy token of each row (Eq. 1: argmax over the vocabulary, ties to
//     the lower id);
//   * the progress rule (a step that commits no current-block token while some
//     remain masked commits the masked one of highest confidence) and the
//     token / mask update of the committed positions;
//   * the layer-0 inputs of the next step: the embedding of every decoded
//     token, the mask embedding elsewhere.
// All are small, memory-bound kernels: one CTA per row, vector loads.
#include "kernels.h"

namespace polestar {

constexpr int DEC_THREADS = 256;

template <typename T>
__global__ void __launch_bounds__(DEC_THREADS) decode_rows_kernel(DecodeRowsArgs a) {
  __shared__ float red[32];
  pdl_enter();
  const int r = blockIdx.x;
  const int s = r / (2 * a.B), j = r % (2 * a.B);
  const float* src = nullptr;
  if (j < a.B) {
    src = a.act + ((size_t)s * a.B + j) * a.d;
  } else if (a.sel && a.fire[s] && a.start + j < a.N) {
    const int w = a.suffix_widx[j - a.B];
    if (w >= 0 && a.sel[(size_t)s * a.Wmax + w]) src = a.U + ((size_t)s * a.Wmax + w) * a.d;
  }
  if (a.start + j >= a.N) src = nullptr;
  T* dst = (T*)a.out + (size_t)r * a.d;
  float ss = 0.f;
  if (src)
    for (int k = threadIdx.x; k < a.d; k += DEC_THREADS) ss += src[k] * src[k];
  const float tot = block_sum(ss, red);
  const float inv = src ? rsqrtf(tot / (float)a.d + a.eps) : 0.f;
  for (int k = threadIdx.x; k < a.d; k += DEC_THREADS) {
    const float g = to_f<T>(((const T*)a.gain)[k]);
    dst[k] = from_f<T>(src ? src[k] * inv * g : 0.f);
  }
}

// Greedy token of each row: the first maximum over the vocabulary.
__global__ void __launch_bounds__(DEC_THREADS) argmax_kernel(const float* __restrict__ logits, int V, int* __restrict__ ids) {
  __shared__ float sv[DEC_THREADS / 32];
  __shared__ int si[DEC_THREADS / 32];
  pdl_enter();
  const float* row = logits + (size_t)blockIdx.x * V;
  float best = -INFINITY;
  int bi = 0x7FFFFFFF;
  for (int v = threadIdx.x; v < V; v += DEC_THREADS) {
    const float x = row[v];
    if (x > best) {  // strictly greater: within a thread the first maximum stays
      best = x;
      bi = v;
    }
  }
  // warp then block reduction, ties to the lower id
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ob > best || (ob == best && oi < bi)) {
      best = ob;
      bi = oi;
    }
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) {
    sv[wid] = best;
    si[wid] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = sv[0];
    int i = si[0];
    for (int w = 1; w < DEC_THREADS / 32; ++w)
      if (sv[w] > b || (sv[w] == b && si[w] < i)) {
        b = sv[w];
        i = si[w];
      }
    ids[blockIdx.x] = i;
  }
}

// One warp per sequence: the progress rule on the current block, then the
// committed positions take their greedy tokens and leave the mask.
__global__ void apply_commits_kernel(ApplyArgs a) {
  pdl_enter();
  const int s = blockIdx.x, lane = threadIdx.x;
  uint8_t* cm = a.commit + (size_t)s * 2 * a.B;
  const float* conf = a.conf + (size_t)s * 2 * a.B;
  // current block: does any masked token commit?  otherwise the most confident
  bool any = false;
  float bc = -INFINITY;
  int bj = -1;
  for (int j0 = 0; j0 < a.B; j0 += 32) {
    const int j = j0 + lane;
    const int p = a.start + j;
    const bool m = j < a.B && p < a.N && a.masked[(size_t)s * a.N + p];
    any |= m && cm[j];
    float c = m ? conf[j] : -INFINITY;
    int jj = m ? j : 0x7FFFFFFF;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float oc = __shfl_xor_sync(0xffffffffu, c, o);
      const int oj = __shfl_xor_sync(0xffffffffu, jj, o);
      if (oc > c || (oc == c && oj < jj)) {
        c = oc;
        jj = oj;
      }
    }
    if (c > bc || (c == bc && jj < bj)) {
      bc = c;
      bj = jj;
    }
  }
  any = __any_sync(0xffffffffu, any);
  __syncwarp();
  if (!any && bj >= 0 && bj < a.B && lane == 0) cm[bj] = 1;
  __syncwarp();
  int cnt = 0;
  for (int j0 = 0; j0 < 2 * a.B; j0 += 32) {
    const int j = j0 + lane;
    const int p = a.start + j;
    if (j < 2 * a.B && p < a.N && cm[j] && a.masked[(size_t)s * a.N + p]) {
      a.tokens[(size_t)s * a.N + p] = a.ids[(size_t)s * 2 * a.B + j];
      a.masked[(size_t)s * a.N + p] = 0;
      ++cnt;
    }
  }
  __syncwarp();
  // masked positions of the current block left after this step
  int left = 0;
  for (int j0 = 0; j0 < a.B; j0 += 32) {
    const int j = j0 + lane;
    const int p = a.start + j;
    if (j < a.B && p < a.N && a.masked[(size_t)s * a.N + p]) ++left;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    left += __shfl_xor_sync(0xffffffffu, left, o);
  }
  if (lane == 0) {
    a.counts[2 * s] = cnt;
    a.counts[2 * s + 1] = left;
  }
}

// Layer-0 inputs: the embedding row of each decoded token, the mask embedding
// at masked positions.
// A token id outside [0, vocab) gives a zero row.
template <typename T>
__global__ void __launch_bounds__(DEC_THREADS) embed_kernel(const T* __restrict__ embed, const T* __restrict__ mask_emb,
                                                            const int* __restrict__ tokens,
                                                            const uint8_t* __restrict__ masked, int vocab, int d,
                                                            T* __restrict__ x0) {
  pdl_enter();
  const size_t r = blockIdx.x;
  const int tok = tokens[r];
  const bool ok = masked[r] || (tok >= 0 && tok < vocab);
  const T* src = masked[r] ? mask_emb : embed + (size_t)(ok ? tok : 0) * d;
  T* dst = x0 + r * d;
  for (int k = threadIdx.x; k < d; k += DEC_THREADS) dst[k] = ok ? src[k] : from_f<T>(0.f);
}

// Block entry: the active rows' last-layer outputs, act[seq, j] = h[r] for the
// rows of kind ROW_ACTIVE.
__global__ void __launch_bounds__(DEC_THREADS) capture_active_kernel(const float* __restrict__ h,
                                                                      const int4* __restrict__ rows, int R, int d, int B,
                                                                      float* __restrict__ act) {
  pdl_enter();
  const int r = blockIdx.x;
  if (r >= R) return;
  const int4 m = rows[r];
  if (m.z != ROW_ACTIVE) return;
  const float* s = h + (size_t)r * d;
  float* dst = act + ((size_t)m.x * B + m.w) * d;
  for (int k = threadIdx.x; k < d; k += DEC_THREADS) dst[k] = s[k];
}

template <typename T>
void launch_decode_rows(const DecodeRowsArgs& a, cudaStream_t st) {
  launch_pdl(decode_rows_kernel<T>, dim3(a.batch * 2 * a.B), dim3(DEC_THREADS), 0, st, a);
}
void launch_argmax(const float* logits, int V, int R, int* ids, cudaStream_t st) {
  launch_pdl(argmax_kernel, dim3(R), dim3(DEC_THREADS), 0, st, logits, V, ids);
}
void launch_apply_commits(const ApplyArgs& a, cudaStream_t st) {
  launch_pdl(apply_commits_kernel, dim3(a.batch), dim3(32), 0, st, a);
}
template <typename T>
void launch_embed(const void* embed, const void* mask_emb, const int* tokens, const uint8_t* masked, int vocab,
                  int rows, int d, void* x0, cudaStream_t st) {
  launch_pdl(embed_kernel<T>, dim3(rows), dim3(DEC_THREADS), 0, st, (const T*)embed, (const T*)mask_emb, tokens, masked,
             vocab, d, (T*)x0);
}
void launch_capture_active(const float* h, const int4* rows, int R, int d, int B, float* act, cudaStream_t st) {
  launch_pdl(capture_active_kernel, dim3(R), dim3(DEC_THREADS), 0, st, h, rows, R, d, B, act);
}

template void launch_decode_rows<float>(const DecodeRowsArgs&, cudaStream_t);
template void launch_decode_rows<__nv_bfloat16>(const DecodeRowsArgs&, cudaStream_t);
template void launch_embed<float>(const void*, const void*, const int*, const uint8_t*, int, int, int, void*,
                                  cudaStream_t);
template void launch_embed<__nv_bfloat16>(const void*, const void*, const int*, const uint8_t*, int, int, int, void*,
                                          cudaStream_t);

}  // namespace polestar
