// Row-wise kernels of the decoder layer: input gather, RMSNorm (A-operand
// producer), rotary embedding + K/V cache scatter, residual adds, SwiGLU.
// Model pieces follow the LLaDA / Dream decoder layer the Polestar paper runs
// (§2, Eq. 3: bidirectional attention over cached and fresh K/V).
//
// Layout of the work: one CTA of ROW_THREADS threads per row; thread t owns the
// 4-element groups t, t + ROW_THREADS, ... of the row (at most ROW_V4 of them,
// so rows up to ROW_THREADS * ROW_V4 * 4 = 8192 elements).  Every thread first
// issues all of its vector loads, then computes from registers, so a row costs
// about one memory round trip instead of one per loop iteration.
#include "kernels.h"

namespace polestar {

namespace {

constexpr int ROW_THREADS = 512;
constexpr int ROW_V4 = 4;

__device__ __forceinline__ float4 ld4(const float* p) { return *(const float4*)p; }
__device__ __forceinline__ void st4(float* p, float4 v) { *(float4*)p = v; }

template <typename T>
__device__ __forceinline__ float4 ld4t(const T* p);
template <>
__device__ __forceinline__ float4 ld4t<float>(const float* p) {
  return *(const float4*)p;
}
template <>
__device__ __forceinline__ float4 ld4t<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *(const uint2*)p;
  const __nv_bfloat162 a = *(const __nv_bfloat162*)&u.x, b = *(const __nv_bfloat162*)&u.y;
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}

template <typename T>
__device__ __forceinline__ void st4t(T* p, float4 v);
template <>
__device__ __forceinline__ void st4t<float>(float* p, float4 v) {
  *(float4*)p = v;
}
template <>
__device__ __forceinline__ void st4t<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *(const uint32_t*)&a;
  u.y = *(const uint32_t*)&b;
  *(uint2*)p = u;
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }
__device__ __forceinline__ float dot4(float4 a) { return a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w; }
__device__ __forceinline__ float4 scale4(float4 a, float s, float4 g) {
  return make_float4(a.x * s * g.x, a.y * s * g.y, a.z * s * g.z, a.w * s * g.w);
}

// element offset of the thread's j-th 4-group
__device__ __forceinline__ int grp(int j) { return (j * ROW_THREADS + threadIdx.x) * 4; }

}  // namespace

// h[r, :] = x0[seq_r, pos_r, :] (storage type -> fp32), rows of kind NONE zeroed;
// with `gain` also a[r] = T(RMSNorm(h[r]) * gain) (the first projection's input).
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS)
    gather_input_kernel(const T* __restrict__ x0, const int4* __restrict__ rows, int R, int N, int d,
                        float* __restrict__ h, const T* __restrict__ gain, float eps, T* __restrict__ a) {
  pdl_enter();
  __shared__ float red[32];
  const int r = blockIdx.x;
  if (r >= R) return;
  const int4 m = rows[r];
  float* dst = h + (size_t)r * d;
  if (m.z == ROW_NONE || m.z == ROW_PROXY) {
#pragma unroll
    for (int j = 0; j < ROW_V4; ++j)
      if (grp(j) < d) st4(dst + grp(j), make_float4(0.f, 0.f, 0.f, 0.f));
    return;
  }
  const T* src = x0 + ((size_t)m.x * N + m.y) * d;
  float4 v[ROW_V4];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j) v[j] = grp(j) < d ? ld4t<T>(src + grp(j)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j)
    if (grp(j) < d) {
      st4(dst + grp(j), v[j]);
      ss += dot4(v[j]);
    }
  if (!gain) return;
  ss = block_sum(ss, red);
  const float inv = 1.f / sqrtf(ss / (float)d + eps);
  T* ao = a + (size_t)r * d;
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j)
    if (grp(j) < d) st4t<T>(ao + grp(j), scale4(v[j], inv, ld4t<T>(gain + grp(j))));
}

// Gather window rows of firing sequences from x0 into the update-packet buffer
// U[seq, widx, :] (layer-0 packet = current inputs).
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS)
    gather_window_kernel(const T* __restrict__ x0, const int* __restrict__ win_pos, int nw,
                         const int* __restrict__ fire_seqs, int N, int d, int Wmax, float* __restrict__ U,
                         uint8_t* __restrict__ sel) {
  pdl_enter();
  const int j = blockIdx.x, f = blockIdx.y;
  const int s = fire_seqs[f];
  const T* src = x0 + ((size_t)s * N + win_pos[j]) * d;
  float* dst = U + ((size_t)s * Wmax + j) * d;
  float4 v[ROW_V4];
#pragma unroll
  for (int q = 0; q < ROW_V4; ++q) v[q] = grp(q) < d ? ld4t<T>(src + grp(q)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int q = 0; q < ROW_V4; ++q)
    if (grp(q) < d) st4(dst + grp(q), v[q]);
  if (threadIdx.x == 0) sel[s * Wmax + j] = 1;
}

// RMSNorm of row sources into the GEMM A operand: a[r] = T(x / sqrt(mean x^2 + eps) * g).
// Source of row r: h[r] (active/window/other), z[seq, c] (proxy; K x d per seq),
// or h[src[r]] when `src` is given (compacted rows).
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS)
    rmsnorm_kernel(const float* __restrict__ h, const int* __restrict__ src, const int* __restrict__ m_dev,
                   const int4* __restrict__ rows, const float* __restrict__ z, int K, const T* __restrict__ gain,
                   int R, int d, float eps, T* __restrict__ a) {
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
#pragma unroll
      for (int j = 0; j < ROW_V4; ++j)
        if (grp(j) < d) st4t<T>(out + grp(j), make_float4(0.f, 0.f, 0.f, 0.f));
      return;
    }
    x = (m.z == ROW_PROXY) ? z + ((size_t)m.x * K + m.w) * d : h + (size_t)r * d;
  } else {
    x = h + (size_t)(src ? src[r] : r) * d;
  }
  float4 v[ROW_V4];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j) v[j] = grp(j) < d ? ld4(x + grp(j)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j) ss += dot4(v[j]);
  ss = block_sum(ss, red);
  const float inv = 1.f / sqrtf(ss / (float)d + eps);
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j)
    if (grp(j) < d) st4t<T>(out + grp(j), scale4(v[j], inv, ld4t<T>(gain + grp(j))));
}

// Rotary embedding (rotate-half, absolute positions) and K/V scatter.
// qkv: [R, ldq] fp32 GEMM output with Q at [0, qdim), K at [qdim, qdim+kvdim),
// V at [qdim+kvdim, qdim+2kvdim).  Q of proxy rows is stored without rotation.
// K/V of a row go to the cache when its kind is ACTIVE/OTHER, or WINDOW with
// write_kv[r] set (a patched row; every window row when write_kv is null);
// proxy rows' K/V are discarded.  Thread work item: 4 consecutive rotary pairs
// (k .. k+3 with partners k+half .. k+half+3) of one head.
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS)
    rope_scatter_kernel(const float* __restrict__ qkv, int ldq, const int4* __restrict__ rows,
                        const uint8_t* __restrict__ write_kv, int R, int H, int Hkv, int dh,
                        const float2* __restrict__ rope_tab, T* __restrict__ qout, T* __restrict__ kv_layer,
                        size_t kv_seq_stride, int kvdim) {
  pdl_enter();
  const int r = blockIdx.x;
  if (r >= R) return;
  const int4 m = rows[r];
  if (m.z == ROW_NONE) return;
  const int half = dh / 2, qdim = H * dh, hq = half / 4;  // 4-pair items per head
  const float* src = qkv + (size_t)r * ldq;
  const float2* tab = rope_tab + (size_t)m.y * half;
  const bool rot = (m.z != ROW_PROXY);
  const bool wkv = (m.z == ROW_ACTIVE || m.z == ROW_OTHER) || (m.z == ROW_WINDOW && (!write_kv || write_kv[r]));
  const int nq = H * hq, nk = wkv ? Hkv * hq : 0, nv = wkv ? kvdim / 4 : 0;
  T* qo = qout + (size_t)r * qdim;
  T* kdst = kv_layer + (size_t)m.x * kv_seq_stride + (size_t)m.y * 2 * kvdim;
  T* vdst = kdst + kvdim;
  // items: [0, nq) Q pairs, [nq, nq + nk) K pairs, then V groups of 4; up to
  // MAXI items per thread and pass (one pass for the LLaDA-8B / Dream-7B rows)
  constexpr int MAXI = 4;
  const int total = nq + nk + nv;
  for (int base = 0; base < total; base += MAXI * ROW_THREADS) {
  float4 x1[MAXI], x2[MAXI], c4[MAXI], s4[MAXI];
  int kind[MAXI], off[MAXI];
#pragma unroll
  for (int q = 0; q < MAXI; ++q) {
    const int it = base + q * ROW_THREADS + threadIdx.x;
    kind[q] = -1;
    if (it < nq || (it >= nq && it < nq + nk)) {
      const bool isq = it < nq;
      const int i2 = isq ? it : it - nq;
      const int hh = i2 / hq, k = (i2 % hq) * 4;
      const float* base = isq ? src + hh * dh : src + qdim + hh * dh;
      off[q] = hh * dh + k;
      kind[q] = isq ? 0 : 1;
      x1[q] = ld4(base + k);
      x2[q] = ld4(base + k + half);
      const float4 t0 = *(const float4*)(tab + k), t1 = *(const float4*)(tab + k + 2);  // (c,s) x 4
      c4[q] = make_float4(t0.x, t0.z, t1.x, t1.z);
      s4[q] = make_float4(t0.y, t0.w, t1.y, t1.w);
    } else if (it >= nq + nk && it < nq + nk + nv) {
      off[q] = (it - nq - nk) * 4;
      kind[q] = 2;
      x1[q] = ld4(src + qdim + kvdim + off[q]);
    }
  }
#pragma unroll
  for (int q = 0; q < MAXI; ++q) {
    if (kind[q] < 0) continue;
    if (kind[q] == 2) {
      st4t<T>(vdst + off[q], x1[q]);
      continue;
    }
    float4 y1 = x1[q], y2 = x2[q];
    if (kind[q] == 1 || rot) {
      const float4 a = x1[q], b = x2[q], c = c4[q], s = s4[q];
      rope_rotate(a.x, b.x, c.x, s.x, y1.x, y2.x);
      rope_rotate(a.y, b.y, c.y, s.y, y1.y, y2.y);
      rope_rotate(a.z, b.z, c.z, s.z, y1.z, y2.z);
      rope_rotate(a.w, b.w, c.w, s.w, y1.w, y2.w);
    }
    T* o = kind[q] == 0 ? qo : kdst;
    st4t<T>(o + off[q], y1);
    st4t<T>(o + off[q] + half, y2);
  }
  }
}

// h1[i] = h[src_i] + y[i];  a[i] = T(RMSNorm(h1[i]) * g).  (attention residual +
// FFN pre-norm).  With src == nullptr the row is i itself and h1 may alias h.
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS)
    residual_rmsnorm_kernel(const float* h, const int* __restrict__ src, const int* __restrict__ m_dev, int R,
                            const float* __restrict__ y, int ldy, const T* __restrict__ gain, int d, float eps,
                            float* h1, T* __restrict__ a) {
  pdl_enter();
  __shared__ float red[32];
  const int i = blockIdx.x;
  const int Rm = m_dev ? min(R, *m_dev) : R;
  if (i >= Rm) return;
  const float* x = h + (size_t)(src ? src[i] : i) * d;
  const float* yy = y + (size_t)i * ldy;
  float* o = h1 + (size_t)i * d;
  float4 v[ROW_V4], w[ROW_V4];
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j) {
    v[j] = grp(j) < d ? ld4(x + grp(j)) : make_float4(0.f, 0.f, 0.f, 0.f);
    w[j] = grp(j) < d ? ld4(yy + grp(j)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j) {
    v[j] = add4(v[j], w[j]);
    ss += dot4(v[j]);
  }
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j)
    if (grp(j) < d) st4(o + grp(j), v[j]);
  ss = block_sum(ss, red);
  const float inv = 1.f / sqrtf(ss / (float)d + eps);
  T* ao = a + (size_t)i * d;
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j)
    if (grp(j) < d) st4t<T>(ao + grp(j), scale4(v[j], inv, ld4t<T>(gain + grp(j))));
}

// act[i, f] = T(silu(g) * u) with g = gu[i, f], u = gu[i, F + f]; one 4-group
// of f per thread (grid: column blocks x rows).
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS)
    swiglu_kernel(const float* __restrict__ gu, int ldg, const int* __restrict__ m_dev, int R, int F,
                  T* __restrict__ act) {
  pdl_enter();
  const int i = blockIdx.y;
  const int Rm = m_dev ? min(R, *m_dev) : R;
  if (i >= Rm) return;
  const int f = (blockIdx.x * ROW_THREADS + threadIdx.x) * 4;
  if (f >= F) return;
  const float* g = gu + (size_t)i * ldg;
  const float4 gv = ld4(g + f), uv = ld4(g + F + f);
  const float4 out = make_float4(gv.x / (1.f + expf(-gv.x)) * uv.x, gv.y / (1.f + expf(-gv.y)) * uv.y,
                                 gv.z / (1.f + expf(-gv.z)) * uv.z, gv.w / (1.f + expf(-gv.w)) * uv.w);
  st4t<T>(act + (size_t)i * F + f, out);
}

// Final FFN residual: out = h1[i] + y[i]; written to h[src_i] when that row is an
// active/other row (input of the next layer), or to the update packet
// U[seq, widx] when it is a window row (U(t, l+1), the update packet of §4.1).
// With `gain` (the next layer's attention-norm gain), rows written to h also
// get a[src_i] = T(RMSNorm(out) * gain), the next projection's input.
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS)
    residual_scatter_kernel(const float* __restrict__ h1, const float* __restrict__ y, int ldy,
                            const int* __restrict__ src, const int* __restrict__ m_dev, int R,
                            const int4* __restrict__ rows, int d, int Wmax, float* h, float* __restrict__ U,
                            const T* __restrict__ gain, float eps, T* __restrict__ an) {
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
  float4 v[ROW_V4], w[ROW_V4];
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j) {
    v[j] = grp(j) < d ? ld4(a + grp(j)) : make_float4(0.f, 0.f, 0.f, 0.f);
    w[j] = grp(j) < d ? ld4(b + grp(j)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j) {
    v[j] = add4(v[j], w[j]);
    ss += dot4(v[j]);
    if (grp(j) < d) st4(dst + grp(j), v[j]);
  }
  if (!gain || to_u) return;  // uniform per block
  ss = block_sum(ss, red);
  const float inv = 1.f / sqrtf(ss / (float)d + eps);
  T* ao = an + (size_t)r * d;
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j)
    if (grp(j) < d) st4t<T>(ao + grp(j), scale4(v[j], inv, ld4t<T>(gain + grp(j))));
}

// dst[i, :] = src[idx[i], :] (storage type rows)
template <typename T>
__global__ void __launch_bounds__(ROW_THREADS)
    gather_T_kernel(const T* __restrict__ src, const int* __restrict__ idx, const int* __restrict__ m_dev, int R,
                    int w, T* __restrict__ dst) {
  pdl_enter();
  const int i = blockIdx.x;
  const int Rm = m_dev ? min(R, *m_dev) : R;
  if (i >= Rm) return;
  const T* s = src + (size_t)idx[i] * w;
  T* o = dst + (size_t)i * w;
  float4 v[ROW_V4];
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j) v[j] = grp(j) < w ? ld4t<T>(s + grp(j)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j)
    if (grp(j) < w) st4t<T>(o + grp(j), v[j]);
}

// Block-entry capture of the layer inputs of window rows: Hw[seq, widx, :] = h[r].
__global__ void __launch_bounds__(ROW_THREADS)
    capture_window_kernel(const float* __restrict__ h, const int4* __restrict__ rows, int R, int d, int Wmax,
                          float* __restrict__ Hw_layer, size_t seq_stride) {
  pdl_enter();
  const int r = blockIdx.x;
  if (r >= R) return;
  const int4 m = rows[r];
  if (m.z != ROW_WINDOW) return;
  float* dst = Hw_layer + (size_t)m.x * seq_stride + (size_t)m.w * d;
  const float* s = h + (size_t)r * d;
  float4 v[ROW_V4];
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j) v[j] = grp(j) < d ? ld4(s + grp(j)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < ROW_V4; ++j)
    if (grp(j) < d) st4(dst + grp(j), v[j]);
}

// ------------------------------------------------------------------ launchers
template <typename T>
void launch_gather_input(const void* x0, const int4* rows, int R, int N, int d, float* h, cudaStream_t st,
                         const void* gain, float eps, void* a) {
  launch_pdl(gather_input_kernel<T>, dim3(R), dim3(ROW_THREADS), 0, st, (const T*)x0, rows, R, N, d, h,
             (const T*)gain, eps, (T*)a);
}
template <typename T>
void launch_gather_window(const void* x0, const int* win_pos, int nw, const int* fire_seqs, int n_fire,
                          int N, int d, int Wmax, float* U, uint8_t* sel, cudaStream_t st) {
  launch_pdl(gather_window_kernel<T>, dim3(nw, n_fire), dim3(ROW_THREADS), 0, st, (const T*)x0, win_pos, nw,
             fire_seqs, N, d, Wmax, U, sel);
}
template <typename T>
void launch_rmsnorm(const float* h, const int* src, const int* m_dev, const int4* rows, const float* z,
                    int K, const void* gain, int R, int d, float eps, void* a, cudaStream_t st) {
  launch_pdl(rmsnorm_kernel<T>, dim3(R), dim3(ROW_THREADS), 0, st, h, src, m_dev, rows, z, K, (const T*)gain, R,
             d, eps, (T*)a);
}
template <typename T>
void launch_rope_scatter(const float* qkv, int ldq, const int4* rows, const uint8_t* write_kv, int R, int H,
                         int Hkv, int dh, const float2* tab, void* qout, void* kv_layer, size_t kv_seq_stride,
                         int kvdim, cudaStream_t st) {
  launch_pdl(rope_scatter_kernel<T>, dim3(R), dim3(ROW_THREADS), 0, st, qkv, ldq, rows, write_kv, R, H, Hkv, dh,
             tab, (T*)qout, (T*)kv_layer, kv_seq_stride, kvdim);
}
template <typename T>
void launch_residual_rmsnorm(const float* h, const int* src, const int* m_dev, int R, const float* y, int ldy,
                             const void* gain, int d, float eps, float* h1, void* a, cudaStream_t st) {
  launch_pdl(residual_rmsnorm_kernel<T>, dim3(R), dim3(ROW_THREADS), 0, st, h, src, m_dev, R, y, ldy,
             (const T*)gain, d, eps, h1, (T*)a);
}
template <typename T>
void launch_swiglu(const float* gu, int ldg, const int* m_dev, int R, int F, void* act, cudaStream_t st) {
  dim3 grid((F + 4 * ROW_THREADS - 1) / (4 * ROW_THREADS), R);
  launch_pdl(swiglu_kernel<T>, grid, dim3(ROW_THREADS), 0, st, gu, ldg, m_dev, R, F, (T*)act);
}
template <typename T>
void launch_residual_scatter(const float* h1, const float* y, int ldy, const int* src, const int* m_dev, int R,
                             const int4* rows, int d, int Wmax, float* h, float* U, cudaStream_t st,
                             const void* gain, float eps, void* an) {
  launch_pdl(residual_scatter_kernel<T>, dim3(R), dim3(ROW_THREADS), 0, st, h1, y, ldy, src, m_dev, R, rows, d,
             Wmax, h, U, (const T*)gain, eps, (T*)an);
}
template <typename T>
void launch_gather_T(const void* src, const int* idx, const int* m_dev, int R, int w, void* dst,
                     cudaStream_t st) {
  launch_pdl(gather_T_kernel<T>, dim3(R), dim3(ROW_THREADS), 0, st, (const T*)src, idx, m_dev, R, w, (T*)dst);
}
void launch_capture_window(const float* h, const int4* rows, int R, int d, int Wmax, float* Hw_layer,
                           size_t seq_stride, cudaStream_t st) {
  launch_pdl(capture_window_kernel, dim3(R), dim3(ROW_THREADS), 0, st, h, rows, R, d, Wmax, Hw_layer, seq_stride);
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
