// Row attention over the whole cached sequence, with the KL drift epilogue.
//
// Every query row (active block, window rows, centroid proxies) attends
// bidirectionally to all N cached keys of its sequence (Eq. 3; proxies use
// "cached KV and recomputed KV tensors for the active block", §4.1).  For
// tracked rows the kernel also measures the drift of Eq. 4,
// KL(softmax(s) || softmax(s')), against the scores s' the same row produced at
// the previous measurement, and replaces s' by the new scores:
//   - proxy rows at every layer (per-cluster drift D, §4.1 "Measuring Drift");
//   - active rows at the last layer (token drift delta_j, §4.2 and the
//     last-layer drift step of Algorithm 1).
//
// KL is evaluated in the cancellation-free form
//   KL = sum_j p_j d_j - log1p( sum_j q~_j expm1(d_j) / sum_j q~_j ),
// d_j = s_j - s'_j, q~_j = exp(s'_j - lse'), which equals sum_j p_j log(p_j/q_j)
// exactly (lse - lse' = log sum_j q_j e^{d_j}) but keeps fp32 accuracy when the
// two distributions are close.
//
// This file: the fp32 path on the CUDA cores (exact fp32 arithmetic; the bf16
// path is the pipelined tensor-core kernel of k_attn_pipe.cu).  One CTA = 8
// query rows (one per warp) x one query head; K/V tiles of 64 keys are staged
// in shared memory as fp32 (odd row pitch: conflict-free for both the per-key
// dot products and the per-dimension P.V sums).
#include "kernels.h"

namespace polestar {

constexpr int ATT_ROWS = 8;   // rows per CTA (one warp each)
constexpr int ATT_TK = 64;    // keys per tile

template <typename T, int DH>
__global__ void __launch_bounds__(256) row_attention_kernel(AttnArgs p) {
  pdl_enter();
  extern __shared__ float smem[];
  constexpr int PITCH = DH + 1;
  float* Ks = smem;                       // [TK][PITCH]
  float* Vs = Ks + ATT_TK * PITCH;        // [TK][PITCH]
  float* Qs = Vs + ATT_TK * PITCH;        // [ROWS][DH]
  float* Ps = Qs + ATT_ROWS * DH;         // [ROWS][TK]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int r0 = blockIdx.x * ATT_ROWS;
  const int r = r0 + warp;
  const int grp = p.H / p.Hkv;
  const int kvh = h / grp;

  // the CTA's sequence: rows of one CTA never mix sequences (host layout rule)
  const int4 m0 = p.rows[r0];
  const int seq = m0.x;
  const T* kvbase = (const T*)p.kv_layer + (size_t)seq * p.kv_seq_stride;

  int4 m = make_int4(0, 0, ROW_NONE, 0);
  if (r < p.R) m = p.rows[r];
  const bool live = (m.z != ROW_NONE) && (m.z != ROW_OTHER || p.other_live);
  const bool need_out = live && m.z != ROW_PROXY;

  // tracking: where the previous scores of this (row, head) live
  float* prev = nullptr;
  float* prev_lse = nullptr;
  // where the new scores / log-sum-exp go: the deferred-drift buffers when the
  // drift pass measures the KL, else over the previous ones
  float* sdst = nullptr;
  float* ldst = nullptr;
  const bool deferred = p.measure && (p.proxy_new != nullptr || p.active_new != nullptr);
  if (live && m.z == ROW_PROXY && p.proxy_prev) {
    const size_t idx = ((size_t)seq * p.K + m.w) * p.H + h;
    prev = p.proxy_prev + idx * p.N;
    prev_lse = p.proxy_prev_lse + idx;
    sdst = deferred ? p.proxy_new + idx * p.N : prev;
    ldst = deferred ? p.proxy_new_lse + idx : prev_lse;
  } else if (live && m.z == ROW_ACTIVE && p.active_prev) {
    const size_t idx = ((size_t)seq * p.B + m.w) * p.H + h;
    prev = p.active_prev + idx * p.N;
    prev_lse = p.active_prev_lse + idx;
    sdst = deferred ? p.active_new + idx * p.N : prev;
    ldst = deferred ? p.active_new_lse + idx : prev_lse;
  }
  const bool do_kl = prev && p.measure && !deferred;
  const bool put = p.store || deferred;
  const float shift_prev = do_kl ? *prev_lse : 0.f;

  // stage this warp's query (fp32)
  if (live) {
    const T* q = (const T*)p.q + (size_t)r * p.ldq + h * DH;
    for (int i = lane; i < DH; i += 32) Qs[warp * DH + i] = to_f<T>(q[i]);
  }

  constexpr int NV = DH / 32;
  float acc[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) acc[i] = 0.f;
  float mrun = -INFINITY, l_part = 0.f, a_part = 0.f, sq_part = 0.f, e_part = 0.f;

  // K/V tiles are fetched with 16-byte loads, one tile ahead of the compute
  constexpr int VEC = 16 / sizeof(T);                 // elements per 16-byte chunk
  constexpr int CPR = DH / VEC;                        // chunks per key row
  constexpr int PER_T = ATT_TK * CPR / 256;            // chunks per thread per matrix
  uint4 kreg[PER_T], vreg[PER_T];
  auto fetch = [&](int j0) {
#pragma unroll
    for (int i = 0; i < PER_T; ++i) {
      const int chunk = threadIdx.x + i * 256;
      const int kk = chunk / CPR, cv = chunk % CPR;
      const int j = j0 + kk;
      if (j < p.N) {
        const T* rowp = kvbase + (size_t)j * 2 * p.kvdim + kvh * DH + cv * VEC;
        kreg[i] = __ldg((const uint4*)rowp);
        vreg[i] = __ldg((const uint4*)(rowp + p.kvdim));
      } else {
        kreg[i] = make_uint4(0, 0, 0, 0);
        vreg[i] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  auto stash = [&]() {
#pragma unroll
    for (int i = 0; i < PER_T; ++i) {
      const int chunk = threadIdx.x + i * 256;
      const int kk = chunk / CPR, cv = chunk % CPR;
      const T* kv8 = (const T*)&kreg[i];
      const T* vv8 = (const T*)&vreg[i];
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        Ks[kk * PITCH + cv * VEC + e] = to_f<T>(kv8[e]);
        Vs[kk * PITCH + cv * VEC + e] = to_f<T>(vv8[e]);
      }
    }
  };

  fetch(0);
  for (int j0 = 0; j0 < p.N; j0 += ATT_TK) {
    __syncthreads();
    stash();
    __syncthreads();
    if (j0 + ATT_TK < p.N) fetch(j0 + ATT_TK);
    if (!live) continue;
    // scores of keys j0+lane and j0+lane+32
    float s[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int kk = lane + 32 * t;
      const float* kr = Ks + kk * PITCH;
      const float* qr = Qs + warp * DH;
      float dot = 0.f;
#pragma unroll 16
      for (int i = 0; i < DH; ++i) dot = fmaf(qr[i], kr[i], dot);
      s[t] = (j0 + kk < p.N) ? dot * p.scale : -INFINITY;
    }
    const float tmax = warp_max(fmaxf(s[0], s[1]));
    const float mnew = fmaxf(mrun, tmax);
    const float corr = expf(mrun - mnew);  // 0 on the first tile (mrun = -inf)
    l_part *= corr;
    a_part *= corr;
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] *= corr;
    mrun = mnew;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int kk = lane + 32 * t;
      const int j = j0 + kk;
      const float pj = (j < p.N) ? expf(s[t] - mnew) : 0.f;
      Ps[warp * ATT_TK + kk] = pj;
      l_part += pj;
      if (prev && j < p.N) {
        if (do_kl) {
          const float sp = prev[j];
          const float dj = s[t] - sp;
          const float qt = expf(sp - shift_prev);
          a_part += pj * dj;
          sq_part += qt;
          e_part += qt * expm1f(dj);
        }
        if (put) sdst[j] = s[t];
      }
    }
    __syncwarp();
    if (need_out) {
      for (int kk = 0; kk < ATT_TK; ++kk) {
        const float pk = Ps[warp * ATT_TK + kk];
        const float* vr = Vs + kk * PITCH;
#pragma unroll
        for (int i = 0; i < NV; ++i) acc[i] = fmaf(pk, vr[lane + 32 * i], acc[i]);
      }
    }
    __syncwarp();
  }
  if (!live) return;
  const float l_tot = warp_sum(l_part);
  if (need_out) {
    T* o = (T*)p.out + (size_t)r * p.ldo + h * DH;
    const float inv = 1.f / l_tot;
#pragma unroll
    for (int i = 0; i < NV; ++i) o[lane + 32 * i] = from_f<T>(acc[i] * inv);
  }
  if (prev) {
    const float a_tot = warp_sum(a_part);
    const float sq_tot = warp_sum(sq_part);
    const float e_tot = warp_sum(e_part);
    if (lane == 0) {
      if (do_kl)
        p.kl_out[(size_t)r * p.H + h] = a_tot / l_tot - kl_log_mass(e_tot / sq_tot, mrun + logf(l_tot), shift_prev);
      if (put) *ldst = mrun + logf(l_tot);
    }
  }
}

int attention_items(int4* w, int n, int a0, int na, int b0, int nb, int max_rows) {
  const int tot = na + nb;
  if (tot <= 0) return n;
  const int k = (tot + max_rows - 1) / max_rows;
  for (int i = 0; i < k; ++i) {
    const int lo = (int)((long long)i * tot / k), hi = (int)((long long)(i + 1) * tot / k);
    if (hi <= na)
      w[n++] = make_int4(a0 + lo, hi - lo, 0, 0);
    else if (lo >= na)
      w[n++] = make_int4(b0 + (lo - na), hi - lo, 0, 0);
    else
      w[n++] = make_int4(a0 + lo, na - lo, b0, hi - na);
  }
  return n;
}

static int g_attention_impl = 0;

int attention_set_impl(int impl) {
  const int old = g_attention_impl;
  g_attention_impl = impl;
  return old;
}

int attention_item_rows(bool bf16, int dh, long long items128, int H, bool measures, bool deferred) {
  if (!bf16 || dh != 128) return ATT_ITEM_ROWS;
  // the tcgen05 kernel leaves KL drift to the deferred drift pass
  if (measures && !deferred) return ATT_ITEM_ROWS;
  if (g_attention_impl == 1) return ATT_ITEM_ROWS;
  if (g_attention_impl == 2) return ATT_TC_ROWS;
  // Library's choice: the tcgen05 kernel when its items fill every SM twice
  // (two CTAs per SM); below that the pipelined mma.sync kernel, whose smaller
  // items and key splits keep all SMs busy.  Measured on GB300 at LLaDA-8B
  // batch 32 (N = 2048): 270 vs 398 us per layer for attention + drift pass.
  static int nsm_of[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int nsm = dev >= 0 && dev < 64 ? nsm_of[dev] : 0;
  if (nsm <= 0) {
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) nsm_of[dev] = nsm;
  }
  return items128 * H >= 2LL * nsm ? ATT_TC_ROWS : ATT_ITEM_ROWS;
}

template <typename T>
cudaError_t launch_row_attention(const AttnArgs& a, cudaStream_t st) {
  if (sizeof(T) == 2 && a.work && a.item_rows == ATT_TC_ROWS) return launch_attention_tc(a, a.batch, st);
  if (sizeof(T) == 2 && a.work) {
    AttnArgs b = a;
    // SM count per device, queried once (a driver query per launch costs host time)
    static int nsm_of[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int nsm = dev >= 0 && dev < 64 ? nsm_of[dev] : 0;
    if (nsm <= 0) {
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
      if (dev >= 0 && dev < 64) nsm_of[dev] = nsm;
    }
    b.splits = attention_pipe_config(a.n_work, a.H, a.N, a.dh, nsm, &b.stages);
    return launch_attention_pipe(b, a.batch, st);
  }
  const dim3 grid((a.R + ATT_ROWS - 1) / ATT_ROWS, a.H);
  if (a.dh == 128) {
    const size_t sm = (2 * ATT_TK * 129 + ATT_ROWS * 128 + ATT_ROWS * ATT_TK) * sizeof(float);
    static PerDeviceOnce cfg;
    const cudaError_t e = func_attr_once(cfg, (const void*)row_attention_kernel<T, 128>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    launch_pdl(row_attention_kernel<T, 128>, dim3(grid), dim3(256), sm, st, a);
  } else {
    const size_t sm = (2 * ATT_TK * 65 + ATT_ROWS * 64 + ATT_ROWS * ATT_TK) * sizeof(float);
    launch_pdl(row_attention_kernel<T, 64>, dim3(grid), dim3(256), sm, st, a);
  }
  return cudaGetLastError();
}

template cudaError_t launch_row_attention<float>(const AttnArgs&, cudaStream_t);
template cudaError_t launch_row_attention<__nv_bfloat16>(const AttnArgs&, cudaStream_t);

}  // namespace polestar
