// Row-wise kernels of the decoder layer: input gather, RMSNorm (A-operand
// producer), rotary embedding + K/V cache scatter, residual adds, SwiGLU.
// Model pieces follow the LLaDA / Dream decoder layer the Polestar paper runs
// (§2, Eq. 3: bidirectional attention over cached and fresh K/V).
#include "kernels.h"

namespace polestar {

// h[r, :] = x0[seq_r, pos_r, :] (storage type -> fp32), rows of kind NONE zeroed;
// with `gain` also a[r] = T(RMSNorm(h[r]) * gain) (the first projection's input).
template <typename T>
__global__ void gather_input_kernel(const T* __restrict__ x0, const int4* __restrict__ rows, int R,
                                    int N, int d, float* __restrict__ h, const T* __restrict__ gain, float eps,
                                    T* __restrict__ a) {
  pdl_enter();
  __shared__ float red[32];
  const int r = blockIdx.x;
  if (r >= R) return;
  const int4 m = rows[r];
  float* dst = h + (size_t)r * d;
  if (m.z == ROW_NONE || m.z == ROW_PROXY) {
    for (int i = threadIdx.x; i < d; i += blockDim.x) dst[i] = 0.f;
    return;
  }
  const T* src = x0 + ((size_t)m.x * N + m.y) * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float v = to_f<T>(src[i]);
    dst[i] = v;
    ss += v * v;
  }
  if (!gain) return;
  ss = block_sum(ss, red);
  const float inv = 1.f / sqrtf(ss / (float)d + eps);
  T* ao = a + (size_t)r * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) ao[i] = from_f<T>(dst[i] * inv * to_f<T>(gain[i]));
}

// Gather window rows of firing sequences from x0 into the update-packet buffer
// U[seq, widx, :] (layer-0 packet = current inputs).
template <typename T>
__global__ void gather_window_kernel(const T* __restrict__ x0, const int* __restrict__ win_pos, int nw,
                                     const int* __restrict__ fire_seqs, int N, int d, int Wmax,
                                     float* __restrict__ U, uint8_t* __restrict__ sel) {
  pdl_enter();
  const int j = blockIdx.x, f = blockIdx.y;
  const int s = fire_seqs[f];
  const T* src = x0 + ((size_t)s * N + win_pos[j]) * d;
  float* dst = U + ((size_t)s * Wmax + j) * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) dst[i] = to_f<T>(src[i]);
  if (threadIdx.x == 0) sel[s * Wmax + j] = 1;
}

// RMSNorm of row sources into the GEMM A operand: a[r] = T(x / sqrt(mean x^2 + eps) * g).
// Source of row r: h[r] (active/window/other), z[seq, c] (proxy; K x d per seq),
// or h[src[r]] when `src` is given (compacted rows).
template <typename T>
__global__ void rmsnorm_kernel(const float* __restrict__ h, const int* __restrict__ src,
                               const int* __restrict__ m_dev, const int4* __restrict__ rows,
                               const float* __restrict__ z, int K, const T* __restrict__ gain, int R,
                               int d, float eps, T* __restrict__ a) {
  pdl_enter();
  __shared__ float red[32];
  const int r = blockIdx.x;
  const int Rm = m_dev ? min(R, *m_dev) : R;
  if (r >= Rm) return;
  const float* x;
  T* out = a + (size_t)r * d;
  if (rows) {
    const int4 m = rows[r];
    if (m.z == ROW_NONE) {
      for (int i = threadIdx.x; i < d; i += blockDim.x) out[i] = from_f<T>(0.f);
      return;
    }
    x = (m.z == ROW_PROXY) ? z + ((size_t)m.x * K + m.w) * d : h + (size_t)r * d;
  } else {
    x = h + (size_t)(src ? src[r] : r) * d;
  }
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) ss += x[i] * x[i];
  ss = block_sum(ss, red);
  const float inv = 1.f / sqrtf(ss / (float)d + eps);
  for (int i = threadIdx.x; i < d; i += blockDim.x) out[i] = from_f<T>(x[i] * inv * to_f<T>(gain[i]));
}

// Rotary embedding (rotate-half, absolute positions) and K/V scatter.
// qkv: [R, ldq] fp32 GEMM output with Q at [0, qdim), K at [qdim, qdim+kvdim),
// V at [qdim+kvdim, qdim+2kvdim).  Q of proxy rows is stored without rotation.
// K/V of a row go to the cache when its kind is ACTIVE/OTHER, or WINDOW with
// write_kv[r] set (a patched row; every window row when write_kv is null);
// proxy rows' K/V are discarded.
template <typename T>
__global__ void rope_scatter_kernel(const float* __restrict__ qkv, int ldq, const int4* __restrict__ rows,
                                    const uint8_t* __restrict__ write_kv, int R, int H, int Hkv, int dh,
                                    const float2* __restrict__ rope_tab, T* __restrict__ qout,
                                    T* __restrict__ kv_layer, size_t kv_seq_stride, int kvdim) {
  pdl_enter();
  const int r = blockIdx.x;
  if (r >= R) return;
  const int4 m = rows[r];
  if (m.z == ROW_NONE) return;
  const int half = dh / 2, qdim = H * dh;
  const float* src = qkv + (size_t)r * ldq;
  const float2* tab = rope_tab + (size_t)m.y * half;
  const bool rot = (m.z != ROW_PROXY);
  T* qo = qout + (size_t)r * qdim;
  for (int i = threadIdx.x; i < H * half; i += blockDim.x) {
    const int hh = i / half, k = i % half;
    const float x1 = src[hh * dh + k], x2 = src[hh * dh + k + half];
    float y1 = x1, y2 = x2;
    if (rot) {
      const float2 cs = tab[k];
      y1 = x1 * cs.x - x2 * cs.y;
      y2 = x2 * cs.x + x1 * cs.y;
    }
    qo[hh * dh + k] = from_f<T>(y1);
    qo[hh * dh + k + half] = from_f<T>(y2);
  }
  const bool wkv = (m.z == ROW_ACTIVE || m.z == ROW_OTHER) || (m.z == ROW_WINDOW && (!write_kv || write_kv[r]));
  if (!wkv) return;
  T* kdst = kv_layer + (size_t)m.x * kv_seq_stride + (size_t)m.y * 2 * kvdim;
  T* vdst = kdst + kvdim;
  const float* ks = src + qdim;
  const float* vs = src + qdim + kvdim;
  for (int i = threadIdx.x; i < Hkv * half; i += blockDim.x) {
    const int hh = i / half, k = i % half;
    const float2 cs = tab[k];
    const float x1 = ks[hh * dh + k], x2 = ks[hh * dh + k + half];
    kdst[hh * dh + k] = from_f<T>(x1 * cs.x - x2 * cs.y);
    kdst[hh * dh + k + half] = from_f<T>(x2 * cs.x + x1 * cs.y);
  }
  for (int i = threadIdx.x; i < kvdim; i += blockDim.x) vdst[i] = from_f<T>(vs[i]);
}

// h1[i] = h[src_i] + y[i];  a[i] = T(RMSNorm(h1[i]) * g).  (attention residual +
// FFN pre-norm).  With src == nullptr the row is i itself and h1 may alias h.
template <typename T>
__global__ void residual_rmsnorm_kernel(const float* h, const int* __restrict__ src,
                                        const int* __restrict__ m_dev, int R, const float* __restrict__ y,
                                        int ldy, const T* __restrict__ gain, int d, float eps,
                                        float* h1, T* __restrict__ a) {
  pdl_enter();
  __shared__ float red[32];
  const int i = blockIdx.x;
  const int Rm = m_dev ? min(R, *m_dev) : R;
  if (i >= Rm) return;
  const float* x = h + (size_t)(src ? src[i] : i) * d;
  const float* yy = y + (size_t)i * ldy;
  float* o = h1 + (size_t)i * d;
  float ss = 0.f;
  for (int k = threadIdx.x; k < d; k += blockDim.x) {
    const float v = x[k] + yy[k];
    o[k] = v;
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float inv = 1.f / sqrtf(ss / (float)d + eps);
  T* ao = a + (size_t)i * d;
  for (int k = threadIdx.x; k < d; k += blockDim.x) ao[k] = from_f<T>(o[k] * inv * to_f<T>(gain[k]));
}

// act[i, f] = T(silu(g) * u) with g = gu[i, f], u = gu[i, F + f].
template <typename T>
__global__ void swiglu_kernel(const float* __restrict__ gu, int ldg, const int* __restrict__ m_dev, int R,
                              int F, T* __restrict__ act) {
  pdl_enter();
  const int i = blockIdx.y;
  const int Rm = m_dev ? min(R, *m_dev) : R;
  if (i >= Rm) return;
  const float* g = gu + (size_t)i * ldg;
  for (int f = blockIdx.x * blockDim.x + threadIdx.x; f < F; f += gridDim.x * blockDim.x) {
    const float gv = g[f];
    const float sg = gv / (1.f + expf(-gv));
    act[(size_t)i * F + f] = from_f<T>(sg * g[F + f]);
  }
}

// Final FFN residual: out = h1[i] + y[i]; written to h[src_i] when that row is an
// active/other row (input of the next layer), or to the update packet
// U[seq, widx] when it is a window row (U(t, l+1), the update packet of §4.1).
// With `gain` (the next layer's attention-norm gain), rows written to h also
// get a[src_i] = T(RMSNorm(out) * gain), the next projection's input.
template <typename T>
__global__ void residual_scatter_kernel(const float* __restrict__ h1, const float* __restrict__ y, int ldy,
                                        const int* __restrict__ src, const int* __restrict__ m_dev, int R,
                                        const int4* __restrict__ rows, int d, int Wmax, float* h,
                                        float* __restrict__ U, const T* __restrict__ gain, float eps,
                                        T* __restrict__ an) {
  pdl_enter();
  __shared__ float red[32];
  const int i = blockIdx.x;
  const int Rm = m_dev ? min(R, *m_dev) : R;
  if (i >= Rm) return;
  const int r = src ? src[i] : i;
  const int4 m = rows[r];
  const bool to_u = (m.z == ROW_WINDOW && U);
  float* dst = to_u ? U + ((size_t)m.x * Wmax + m.w) * d : h + (size_t)r * d;
  const float* a = h1 + (size_t)i * d;
  const float* b = y + (size_t)i * ldy;
  float ss = 0.f;
  for (int k = threadIdx.x; k < d; k += blockDim.x) {
    const float v = a[k] + b[k];
    dst[k] = v;
    ss += v * v;
  }
  if (!gain || to_u) return;  // uniform per block
  ss = block_sum(ss, red);
  const float inv = 1.f / sqrtf(ss / (float)d + eps);
  T* ao = an + (size_t)r * d;
  for (int k = threadIdx.x; k < d; k += blockDim.x) ao[k] = from_f<T>(dst[k] * inv * to_f<T>(gain[k]));
}

// dst[i, :] = src[idx[i], :] (storage type rows)
template <typename T>
__global__ void gather_T_kernel(const T* __restrict__ src, const int* __restrict__ idx,
                                const int* __restrict__ m_dev, int R, int w, T* __restrict__ dst) {
  pdl_enter();
  const int i = blockIdx.x;
  const int Rm = m_dev ? min(R, *m_dev) : R;
  if (i >= Rm) return;
  const T* s = src + (size_t)idx[i] * w;
  T* o = dst + (size_t)i * w;
  for (int k = threadIdx.x; k < w; k += blockDim.x) o[k] = s[k];
}

// Block-entry capture of the layer inputs of window rows: Hw[seq, widx, :] = h[r].
__global__ void capture_window_kernel(const float* __restrict__ h, const int4* __restrict__ rows, int R,
                                      int d, int Wmax, float* __restrict__ Hw_layer, size_t seq_stride) {
  pdl_enter();
  const int r = blockIdx.x;
  if (r >= R) return;
  const int4 m = rows[r];
  if (m.z != ROW_WINDOW) return;
  float* dst = Hw_layer + (size_t)m.x * seq_stride + (size_t)m.w * d;
  const float* s = h + (size_t)r * d;
  for (int k = threadIdx.x; k < d; k += blockDim.x) dst[k] = s[k];
}

// ------------------------------------------------------------------ launchers
template <typename T>
void launch_gather_input(const void* x0, const int4* rows, int R, int N, int d, float* h, cudaStream_t st,
                         const void* gain, float eps, void* a) {
  launch_pdl(gather_input_kernel<T>, dim3(R), dim3(256), 0, st, (const T*)x0, rows, R, N, d, h, (const T*)gain,
             eps, (T*)a);
}
template <typename T>
void launch_gather_window(const void* x0, const int* win_pos, int nw, const int* fire_seqs, int n_fire,
                          int N, int d, int Wmax, float* U, uint8_t* sel, cudaStream_t st) {
  launch_pdl(gather_window_kernel<T>, dim3(nw, n_fire), dim3(256), 0, st, (const T*)x0, win_pos, nw, fire_seqs, N, d,
                                   Wmax, U, sel);
}
template <typename T>
void launch_rmsnorm(const float* h, const int* src, const int* m_dev, const int4* rows, const float* z,
                    int K, const void* gain, int R, int d, float eps, void* a, cudaStream_t st) {
  launch_pdl(rmsnorm_kernel<T>, dim3(R), dim3(256), 0, st, h, src, m_dev, rows, z, K, (const T*)gain, R, d, eps, (T*)a);
}
template <typename T>
void launch_rope_scatter(const float* qkv, int ldq, const int4* rows, const uint8_t* write_kv, int R, int H,
                         int Hkv, int dh, const float2* tab, void* qout, void* kv_layer, size_t kv_seq_stride,
                         int kvdim, cudaStream_t st) {
  launch_pdl(rope_scatter_kernel<T>, dim3(R), dim3(256), 0, st, qkv, ldq, rows, write_kv, R, H, Hkv, dh, tab, (T*)qout,
                                            (T*)kv_layer, kv_seq_stride, kvdim);
}
template <typename T>
void launch_residual_rmsnorm(const float* h, const int* src, const int* m_dev, int R, const float* y, int ldy,
                             const void* gain, int d, float eps, float* h1, void* a, cudaStream_t st) {
  launch_pdl(residual_rmsnorm_kernel<T>, dim3(R), dim3(256), 0, st, h, src, m_dev, R, y, ldy, (const T*)gain, d, eps, h1, (T*)a);
}
template <typename T>
void launch_swiglu(const float* gu, int ldg, const int* m_dev, int R, int F, void* act, cudaStream_t st) {
  dim3 grid((F + 1023) / 1024, R);
  launch_pdl(swiglu_kernel<T>, dim3(grid), dim3(256), 0, st, gu, ldg, m_dev, R, F, (T*)act);
}
template <typename T>
void launch_residual_scatter(const float* h1, const float* y, int ldy, const int* src, const int* m_dev, int R,
                             const int4* rows, int d, int Wmax, float* h, float* U, cudaStream_t st,
                             const void* gain, float eps, void* an) {
  launch_pdl(residual_scatter_kernel<T>, dim3(R), dim3(256), 0, st, h1, y, ldy, src, m_dev, R, rows, d, Wmax, h, U,
             (const T*)gain, eps, (T*)an);
}
template <typename T>
void launch_gather_T(const void* src, const int* idx, const int* m_dev, int R, int w, void* dst,
                     cudaStream_t st) {
  launch_pdl(gather_T_kernel<T>, dim3(R), dim3(256), 0, st, (const T*)src, idx, m_dev, R, w, (T*)dst);
}
void launch_capture_window(const float* h, const int4* rows, int R, int d, int Wmax, float* Hw_layer,
                           size_t seq_stride, cudaStream_t st) {
  launch_pdl(capture_window_kernel, dim3(R), dim3(256), 0, st, h, rows, R, d, Wmax, Hw_layer, seq_stride);
}

#define INST(T)                                                                                          \
  template void launch_gather_input<T>(const void*, const int4*, int, int, int, float*, cudaStream_t,     \
                                       const void*, float, void*);                                       \
  template void launch_residual_scatter<T>(const float*, const float*, int, const int*, const int*, int,  \
                                           const int4*, int, int, float*, float*, cudaStream_t,          \
                                           const void*, float, void*);                                   \
  template void launch_gather_window<T>(const void*, const int*, int, const int*, int, int, int, int,    \
                                        float*, uint8_t*, cudaStream_t);                                 \
  template void launch_rmsnorm<T>(const float*, const int*, const int*, const int4*, const float*, int,  \
                                  const void*, int, int, float, void*, cudaStream_t);                    \
  template void launch_rope_scatter<T>(const float*, int, const int4*, const uint8_t*, int, int, int, int, \
                                       const float2*, void*, void*, size_t, int, cudaStream_t);          \
  template void launch_residual_rmsnorm<T>(const float*, const int*, const int*, int, const float*, int, \
                                           const void*, int, float, float*, void*, cudaStream_t);        \
  template void launch_swiglu<T>(const float*, int, const int*, int, int, void*, cudaStream_t);          \
  template void launch_gather_T<T>(const void*, const int*, const int*, int, int, void*, cudaStream_t);
INST(float)
INST(__nv_bfloat16)
#undef INST

}  // namespace polestar
