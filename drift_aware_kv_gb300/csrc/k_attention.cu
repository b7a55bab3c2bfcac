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
// Work split: one CTA = 8 query rows (one per warp) x one query head; K/V tiles
// of 64 keys are staged in shared memory as fp32 (odd row pitch: conflict-free
// for both the per-key dot products and the per-dimension P.V sums).
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
  if (live && m.z == ROW_PROXY && p.proxy_prev) {
    const size_t idx = ((size_t)seq * p.K + m.w) * p.H + h;
    prev = p.proxy_prev + idx * p.N;
    prev_lse = p.proxy_prev_lse + idx;
  } else if (live && m.z == ROW_ACTIVE && p.active_prev) {
    const size_t idx = ((size_t)seq * p.B + m.w) * p.H + h;
    prev = p.active_prev + idx * p.N;
    prev_lse = p.active_prev_lse + idx;
  }
  const bool do_kl = prev && p.measure;
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
        if (p.store) prev[j] = s[t];
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
      if (do_kl) p.kl_out[(size_t)r * p.H + h] = a_tot / l_tot - log1pf(e_tot / sq_tot);
      if (p.store) *prev_lse = mrun + logf(l_tot);
    }
  }
}

// ---------------------------------------------------------------------------
// bf16 path on the tensor cores (mma.sync m16n8k16, fp32 accumulation).
// One CTA = 4 warps x 16 query rows of one row segment (host work list: a
// segment never mixes sequences) x one query head.  K/V tiles of 64 keys are
// double-buffered in shared memory with cp.async; S = Q K^T and O += P V run on
// the tensor cores with the online softmax and the KL epilogue in registers.
// ---------------------------------------------------------------------------
constexpr int AM_TK = 64;

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 2^x with the hardware approximation (relative error ~2^-22; 2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *(const uint32_t*)&v;
}

template <int DH>
__global__ void __launch_bounds__(128) attn_mma_kernel(AttnArgs p) {
  pdl_enter();
  constexpr int KP = DH + 8;  // smem pitch (elements): 16-byte rows, conflict-free ldmatrix
  extern __shared__ __align__(16) __nv_bfloat16 sm_kv[];
  __nv_bfloat16* Ks = sm_kv;                   // [2][TK][KP]
  __nv_bfloat16* Vs = Ks + 2 * AM_TK * KP;     // [2][TK][KP]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int4 wk = p.work[blockIdx.x];          // {row_start, row_count, seq, 0}
  const int seq = wk.z;
  const int kvh = h / (p.H / p.Hkv);
  const __nv_bfloat16* kvbase = (const __nv_bfloat16*)p.kv_layer + (size_t)seq * p.kv_seq_stride + kvh * DH;

  const int qr = lane >> 2, qc = lane & 3;     // fragment row / column group
  const int rl0 = warp * 16 + qr, rl1 = rl0 + 8;
  const int rows[2] = {wk.x + rl0, wk.x + rl1};
  bool live[2], outp[2];
  float* prev[2] = {nullptr, nullptr};
  float* prev_lse[2] = {nullptr, nullptr};
  float shift[2] = {0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int rl = i ? rl1 : rl0;
    int4 m = make_int4(0, 0, ROW_NONE, 0);
    if (rl < wk.y) m = p.rows[rows[i]];
    live[i] = m.z != ROW_NONE;
    outp[i] = live[i] && m.z != ROW_PROXY;
    if (live[i] && m.z == ROW_PROXY && p.proxy_prev) {
      const size_t idx = ((size_t)seq * p.K + m.w) * p.H + h;
      prev[i] = p.proxy_prev + idx * p.N;
      prev_lse[i] = p.proxy_prev_lse + idx;
    } else if (live[i] && m.z == ROW_ACTIVE && p.active_prev) {
      const size_t idx = ((size_t)seq * p.B + m.w) * p.H + h;
      prev[i] = p.active_prev + idx * p.N;
      prev_lse[i] = p.active_prev_lse + idx;
    }
    if (prev[i] && p.measure) shift[i] = *prev_lse[i];
  }
  const bool warp_live = __any_sync(0xffffffffu, live[0] || live[1]);
  const bool warp_tracked = __any_sync(0xffffffffu, prev[0] != nullptr || prev[1] != nullptr);

  // Q fragments (A operand) straight from global memory
  constexpr int KT = DH / 16;
  uint32_t qa[KT][4];
  {
    const __nv_bfloat16* q0 = (const __nv_bfloat16*)p.q + (size_t)rows[0] * p.ldq + h * DH;
    const __nv_bfloat16* q1 = (const __nv_bfloat16*)p.q + (size_t)rows[1] * p.ldq + h * DH;
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      const int c = kt * 16 + qc * 2;
      qa[kt][0] = live[0] ? *(const uint32_t*)(q0 + c) : 0u;
      qa[kt][1] = live[1] ? *(const uint32_t*)(q1 + c) : 0u;
      qa[kt][2] = live[0] ? *(const uint32_t*)(q0 + c + 8) : 0u;
      qa[kt][3] = live[1] ? *(const uint32_t*)(q1 + c + 8) : 0u;
    }
  }

  auto load_tile = [&](int buf, int j0) {
    __nv_bfloat16* kd = Ks + buf * AM_TK * KP;
    __nv_bfloat16* vd = Vs + buf * AM_TK * KP;
    constexpr int CPR = DH / 8;  // 16-byte chunks per row
    for (int ch = threadIdx.x; ch < AM_TK * CPR; ch += 128) {
      const int kk = ch / CPR, cv = ch % CPR;
      const int j = j0 + kk;
      const bool v = j < p.N;
      const __nv_bfloat16* src = kvbase + (size_t)(v ? j : 0) * 2 * p.kvdim + cv * 8;
      cp_async16(kd + kk * KP + cv * 8, src, v);
      cp_async16(vd + kk * KP + cv * 8, src + p.kvdim, v);
    }
    cp_async_commit();
  };

  constexpr int NT = DH / 8;  // output n-tiles
  float acc[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float mrun[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
  float asum[2] = {0.f, 0.f}, sqs[2] = {0.f, 0.f}, esum[2] = {0.f, 0.f};

  const int ntiles_all = (p.N + AM_TK - 1) / AM_TK;
  const int nsplit = gridDim.z, split = blockIdx.z;
  const int tbeg = split * ntiles_all / nsplit, tend = (split + 1) * ntiles_all / nsplit;
  load_tile(0, tbeg * AM_TK);
  for (int t = tbeg; t < tend; ++t) {
    const int buf = (t - tbeg) & 1;
    if (t + 1 < tend) {
      load_tile(buf ^ 1, (t + 1) * AM_TK);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const __nv_bfloat16* kt_s = Ks + buf * AM_TK * KP;
    const __nv_bfloat16* vt_s = Vs + buf * AM_TK * KP;
    const int j0 = t * AM_TK;
    if (warp_live) {
      // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
      float sc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int kt = 0; kt < KT; kt += 2) {
          const int mi = lane >> 3, ri = lane & 7;
          const __nv_bfloat16* ad = kt_s + (nt * 8 + ri) * KP + kt * 16 + (mi & 1) * 8 + (mi >> 1) * 16;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(b0, b1, b2, b3, ad);
          mma16816(sc[nt], qa[kt], b0, b1);
          mma16816(sc[nt], qa[kt + 1], b2, b3);
        }
      }
      // scores in log2 units (s2 = q.k * scale * log2 e): the attention weights
      // use the hardware exp2; tracked rows convert back to natural units for
      // the stored scores and the KL terms
      const float sl2 = p.scale * 1.4426950408889634f;
      const bool full = (j0 + AM_TK <= p.N);
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = sc[nt][e] * sl2;
          if (!full && j0 + nt * 8 + qc * 2 + (e & 1) >= p.N) v = -INFINITY;
          sc[nt][e] = v;
          tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
        }
      }
      float corr[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 1));
        tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 2));
        const float mnew = fmaxf(mrun[i], tmax[i]);
        corr[i] = ex2_approx(mrun[i] - mnew);
        mrun[i] = mnew;
        lsum[i] *= corr[i];
        asum[i] *= corr[i];
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        acc[nt][0] *= corr[0];
        acc[nt][1] *= corr[0];
        acc[nt][2] *= corr[1];
        acc[nt][3] *= corr[1];
      }
      // tracked rows: fetch the whole tile's previous scores before any store
      float spv[8][4];
      if (warp_tracked) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = e >> 1;
            const int j = j0 + nt * 8 + qc * 2 + (e & 1);
            spv[nt][e] = (prev[i] && p.measure && j < p.N) ? __ldcg(prev[i] + j) : 0.f;
          }
      }
      uint32_t pa[4][4];  // P as A fragments: 4 k-steps of 16 keys
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pv[e] = ex2_approx(sc[nt][e] - mrun[e >> 1]);  // exp2(-inf) = 0 for masked keys
          lsum[e >> 1] += pv[e];
        }
        if (warp_tracked) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = e >> 1;
            const int j = j0 + nt * 8 + qc * 2 + (e & 1);
            if (prev[i] && j < p.N) {
              const float s_nat = sc[nt][e] * 0.6931471805599453f;
              if (p.measure) {
                const float sp = spv[nt][e];
                const float dj = s_nat - sp;
                const float qt = expf(sp - shift[i]);
                asum[i] += pv[e] * dj;
                sqs[i] += qt;
                esum[i] += qt * expm1f(dj);
              }
              spv[nt][e] = s_nat;
            }
          }
        }
        const int kt = nt >> 1;
        if ((nt & 1) == 0) {
          pa[kt][0] = pack_bf16(pv[0], pv[1]);
          pa[kt][1] = pack_bf16(pv[2], pv[3]);
        } else {
          pa[kt][2] = pack_bf16(pv[0], pv[1]);
          pa[kt][3] = pack_bf16(pv[2], pv[3]);
        }
      }
      if (warp_tracked && p.store) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            // two adjacent keys per row: one 8-byte store
            const int i = e;
            const int j = j0 + nt * 8 + qc * 2;
            if (prev[i] && j < p.N) {
              float* dst = prev[i] + j;
              if (j + 1 < p.N && (((uintptr_t)dst) & 7) == 0) {
                *(float2*)dst = make_float2(spv[nt][2 * e], spv[nt][2 * e + 1]);
              } else {
                dst[0] = spv[nt][2 * e];
                if (j + 1 < p.N) dst[1] = spv[nt][2 * e + 1];
              }
            }
          }
      }
      // O += P V
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
          const int mi = lane >> 3, ri = lane & 7;
          const __nv_bfloat16* ad = vt_s + (kt * 16 + (mi & 1) * 8 + ri) * KP + (nt + (mi >> 1)) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3, ad);
          mma16816(acc[nt], pa[kt], b0, b1);
          mma16816(acc[nt + 1], pa[kt], b2, b3);
        }
      }
    }
    __syncthreads();
  }
  // finalize: row sums across the 4 threads sharing a row
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      lsum[i] += __shfl_xor_sync(0xffffffffu, lsum[i], o);
      asum[i] += __shfl_xor_sync(0xffffffffu, asum[i], o);
      sqs[i] += __shfl_xor_sync(0xffffffffu, sqs[i], o);
      esum[i] += __shfl_xor_sync(0xffffffffu, esum[i], o);
    }
  }
  if (nsplit > 1) {
    // partial results of this key slice; the combine kernel finishes the rows
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int rl = i ? rl1 : rl0;
      if (rl >= wk.y || !live[i]) continue;
      float* pp = p.part + (((size_t)split * p.R + rows[i]) * p.H + h) * (5 + DH);
      if (qc == 0) {
        pp[0] = mrun[i];
        pp[1] = lsum[i];
        pp[2] = asum[i];
        pp[3] = sqs[i];
        pp[4] = esum[i];
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        pp[5 + nt * 8 + qc * 2] = acc[nt][2 * i];
        pp[5 + nt * 8 + qc * 2 + 1] = acc[nt][2 * i + 1];
      }
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (outp[i]) {
      __nv_bfloat16* o = (__nv_bfloat16*)p.out + (size_t)rows[i] * p.ldo + h * DH;
      const float inv = 1.f / lsum[i];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *(uint32_t*)(o + nt * 8 + qc * 2) = pack_bf16(acc[nt][2 * i] * inv, acc[nt][2 * i + 1] * inv);
    }
    if (prev[i] && qc == 0) {
      if (p.measure) p.kl_out[(size_t)rows[i] * p.H + h] = asum[i] / lsum[i] - log1pf(esum[i] / sqs[i]);
      if (p.store) *prev_lse[i] = mrun[i] * 0.6931471805599453f + logf(lsum[i]);
    }
  }
}

// Merge the key-split partials of attn_mma_kernel: one warp per (row, head).
template <int DH>
__global__ void attn_combine_kernel(AttnArgs p) {
  pdl_enter();
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (gw >= p.R * p.H) return;
  const int r = gw / p.H, h = gw % p.H;
  const int4 m = p.rows[r];
  if (m.z == ROW_NONE) return;
  const int seq = m.x;
  const size_t stride = (size_t)p.R * p.H * (5 + DH);
  const float* base = p.part + ((size_t)r * p.H + h) * (5 + DH);
  float M = -INFINITY;
  for (int s = 0; s < p.splits; ++s) M = fmaxf(M, base[s * stride]);
  float l = 0.f, a = 0.f, sq = 0.f, e = 0.f;
  constexpr int NV = DH / 32;
  float acc[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) acc[i] = 0.f;
  for (int s = 0; s < p.splits; ++s) {
    const float* pp = base + s * stride;
    const float w = ex2_approx(pp[0] - M);  // partial maxima are in log2 units
    l += pp[1] * w;
    a += pp[2] * w;
    sq += pp[3];
    e += pp[4];
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] += pp[5 + lane + 32 * i] * w;
  }
  if (m.z != ROW_PROXY) {
    __nv_bfloat16* o = (__nv_bfloat16*)p.out + (size_t)r * p.ldo + h * DH;
    const float inv = 1.f / l;
#pragma unroll
    for (int i = 0; i < NV; ++i) o[lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
  }
  float* prev_lse = nullptr;
  if (m.z == ROW_PROXY && p.proxy_prev)
    prev_lse = p.proxy_prev_lse + ((size_t)seq * p.K + m.w) * p.H + h;
  else if (m.z == ROW_ACTIVE && p.active_prev)
    prev_lse = p.active_prev_lse + ((size_t)seq * p.B + m.w) * p.H + h;
  if (prev_lse && lane == 0) {
    if (p.measure) p.kl_out[(size_t)r * p.H + h] = a / l - log1pf(e / sq);
    if (p.store) *prev_lse = M * 0.6931471805599453f + logf(l);
  }
}

int attention_splits(int R, int H, int N, int dh, size_t part_floats, int num_sms) {
  const int ctas = ((R + 63) / 64) * H;
  const int tiles = (N + AM_TK - 1) / AM_TK;
  int s = 1;
  while (s < 8 && ctas * s * 2 <= 4 * num_sms && tiles >= 2 * s * 2 &&
         (size_t)(2 * s) * R * H * (5 + dh) <= part_floats)
    s *= 2;
  return s;
}

template <typename T>
void launch_row_attention(const AttnArgs& a, cudaStream_t st) {
  if (sizeof(T) == 2 && a.work) {
    const int splits = (a.splits > 1 && a.part) ? a.splits : 1;
    AttnArgs b = a;
    b.splits = splits;
    const dim3 grid(a.n_work, a.H, splits);
    const int cw = (a.R * a.H * 32 + 255) / 256;
    if (a.dh == 128) {
      const size_t sm = 4 * AM_TK * (128 + 8) * sizeof(__nv_bfloat16);
      static bool cfg = false;
      if (!cfg) {
        cudaFuncSetAttribute(attn_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        cfg = true;
      }
      launch_pdl(attn_mma_kernel<128>, dim3(grid), dim3(128), sm, st, b);
      if (splits > 1) launch_pdl(attn_combine_kernel<128>, dim3(cw), dim3(256), 0, st, b);
    } else {
      const size_t sm = 4 * AM_TK * (64 + 8) * sizeof(__nv_bfloat16);
      launch_pdl(attn_mma_kernel<64>, dim3(grid), dim3(128), sm, st, b);
      if (splits > 1) launch_pdl(attn_combine_kernel<64>, dim3(cw), dim3(256), 0, st, b);
    }
    return;
  }
  const dim3 grid((a.R + ATT_ROWS - 1) / ATT_ROWS, a.H);
  if (a.dh == 128) {
    const size_t sm = (2 * ATT_TK * 129 + ATT_ROWS * 128 + ATT_ROWS * ATT_TK) * sizeof(float);
    static bool cfg = false;
    if (!cfg) {
      cudaFuncSetAttribute(row_attention_kernel<T, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
      cfg = true;
    }
    launch_pdl(row_attention_kernel<T, 128>, dim3(grid), dim3(256), sm, st, a);
  } else {
    const size_t sm = (2 * ATT_TK * 65 + ATT_ROWS * 64 + ATT_ROWS * ATT_TK) * sizeof(float);
    launch_pdl(row_attention_kernel<T, 64>, dim3(grid), dim3(256), sm, st, a);
  }
}

template void launch_row_attention<float>(const AttnArgs&, cudaStream_t);
template void launch_row_attention<__nv_bfloat16>(const AttnArgs&, cudaStream_t);

}  // namespace polestar
