// KL drift of tracked rows (Eq. 4 of "Polestar: Drift-Aware Cache Calibration
// and Token Commitment for Efficient Inference of Diffusion LLMs", §4.1
// "Measuring Drift") from two stored score rows: the new scores s and
// log-sum-exp an attention launch wrote in deferred mode, and the previous
// ones sp, lse_p kept from the last measurement.  With p = softmax(s),
// q = softmax(sp) and d = s - sp:
//   KL(p || q) = sum_j p_j d_j - log sum_j q_j e^(d_j),
// the second term as log1p(sum_j q_j expm1(d_j) / sum_j q_j) while that stays
// accurate, else as lse - lse_p (kl_log_mass).  One warp per (tracked row,
// head): its lanes stride over the N keys with 16-byte loads, then
// fixed-order butterfly sums (deterministic).  With store, the new scores and
// log-sum-exp then replace the previous ones.  Memory-bound: 8 bytes read (+ 4
// written with store) per key.
#include "kernels.h"

namespace polestar {

constexpr int DRIFT_WARPS = 8;  // (tracked row, head) pairs per CTA, one warp each

__global__ void __launch_bounds__(DRIFT_WARPS * 32) drift_kernel(DriftArgs a) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long u = (long long)blockIdx.x * DRIFT_WARPS + warp;  // (tracked row, head) index
  if (u >= (long long)a.n_track * a.H) return;
  const int4 t = a.track[u / a.H];
  const int h = (int)(u % a.H);
  const bool proxy = t.z == ROW_PROXY;
  const size_t idx = proxy ? ((size_t)t.y * a.K + t.w) * a.H + h : ((size_t)t.y * a.B + t.w) * a.H + h;
  float* prev = (proxy ? a.proxy_prev : a.active_prev) + idx * a.N;
  float* prev_lse = (proxy ? a.proxy_prev_lse : a.active_prev_lse) + idx;
  const float* cur = (proxy ? a.proxy_new : a.active_new) + idx * a.N;
  const float lse = (proxy ? a.proxy_new_lse : a.active_new_lse)[idx];
  const float lse_p = *prev_lse;
  float pd = 0.f, qs = 0.f, qe = 0.f;
  const bool vec = (a.N & 3) == 0 && ((((uintptr_t)prev) | ((uintptr_t)cur)) & 15) == 0;
  if (vec) {
    for (int j = lane * 4; j < a.N; j += 32 * 4) {
      const float4 s4 = *(const float4*)(cur + j);
      const float4 p4 = *(const float4*)(prev + j);
      const float s[4] = {s4.x, s4.y, s4.z, s4.w}, sp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float d = s[e] - sp[e];
        const float q = expf(sp[e] - lse_p);
        pd = fmaf(expf(s[e] - lse), d, pd);
        qs += q;
        qe = fmaf(q, expm1f(d), qe);
      }
      if (a.store) *(float4*)(prev + j) = s4;
    }
  } else {
    for (int j = lane; j < a.N; j += 32) {
      const float s = cur[j], sp = prev[j];
      const float d = s - sp;
      const float q = expf(sp - lse_p);
      pd = fmaf(expf(s - lse), d, pd);
      qs += q;
      qe = fmaf(q, expm1f(d), qe);
      if (a.store) prev[j] = s;
    }
  }
  // fixed-order butterfly sums (deterministic)
  const float PD = warp_sum(pd), QS = warp_sum(qs), QE = warp_sum(qe);
  if (lane == 0) {
    a.kl_out[(size_t)t.x * a.H + h] = PD - kl_log_mass(QE / QS, lse, lse_p);
    if (a.store) *prev_lse = lse;
  }
}

void launch_drift(const DriftArgs& a, cudaStream_t st) {
  if (a.n_track <= 0) return;
  const long long pairs = (long long)a.n_track * a.H;
  launch_pdl(drift_kernel, dim3((unsigned)((pairs + DRIFT_WARPS - 1) / DRIFT_WARPS)), dim3(DRIFT_WARPS * 32), 0, st, a);
}

}  // namespace polestar
