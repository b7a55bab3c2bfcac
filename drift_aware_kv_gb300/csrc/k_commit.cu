// Polestar-Commit (§4.2; the commit phases of Algorithm 1).
//
//   conf_partial_kernel  split-V online (max, sum exp) of every logit row
//                        (the logits read dominates: 2B rows x V fp32 per sequence)
//   commit_gate_kernel   c_j = max softmax; current block: Delta_j = delta_j minus
//                        the mean of the last h drifts (current one excluded),
//                        tau_d = alpha (tau_s - c_j)^2, commit iff masked and
//                        (c_j >= tau_s or Delta_j >= tau_d); suffix block: commit
//                        iff masked, in the last layer's selected clusters and
//                        c_j >= tau_suf.  Block entry: confidence only.
#include "kernels.h"

namespace polestar {

__global__ void conf_partial_kernel(CommitArgs a) {
  pdl_enter();
  __shared__ float sm_m[32], sm_s[32];
  const int row = blockIdx.x, sp = blockIdx.y;
  const int chunk = (a.V + a.splits - 1) / a.splits;
  const int v0 = sp * chunk, v1 = min(a.V, v0 + chunk);
  const float* l = a.logits + (size_t)row * a.V;
  float m = -INFINITY, s = 0.f;
  const bool vec = ((a.V & 3) == 0) && ((v0 & 3) == 0) && ((((uintptr_t)a.logits) & 15) == 0);
  if (vec) {
    const int n4 = (v1 - v0) >> 2;
    const float4* l4 = (const float4*)(l + v0);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
      const float4 x = l4[i];
      const float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
      if (mx > m) {
        s *= expf(m - mx);
        m = mx;
      }
      s += expf(x.x - m) + expf(x.y - m) + expf(x.z - m) + expf(x.w - m);
    }
    for (int v = v0 + (n4 << 2) + threadIdx.x; v < v1; v += blockDim.x) {
      const float x = l[v];
      if (x > m) {
        s *= expf(m - x);
        m = x;
      }
      s += expf(x - m);
    }
  } else {
    for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
      const float x = l[v];
      if (x > m) {
        s *= expf(m - x);
        m = x;
      }
      s += expf(x - m);
    }
  }
  // combine (m, s) pairs over the block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float mm = fmaxf(m, m2);
    s = (mm == -INFINITY) ? 0.f : s * expf(m - mm) + s2 * expf(m2 - mm);
    m = mm;
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_s[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY, S = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      const float mm = fmaxf(M, sm_m[w]);
      S = (mm == -INFINITY) ? 0.f : S * expf(M - mm) + sm_s[w] * expf(sm_m[w] - mm);
      M = mm;
    }
    a.part[((size_t)row * a.splits + sp) * 2 + 0] = M;
    a.part[((size_t)row * a.splits + sp) * 2 + 1] = S;
  }
}

__global__ void commit_gate_kernel(CommitArgs a) {
  pdl_enter();
  const int s = blockIdx.x, j = threadIdx.x;
  const int B = a.B;
  if (j >= 2 * B) return;
  const int row = s * 2 * B + j;
  float M = -INFINITY, S = 0.f;
  for (int sp = 0; sp < a.splits; ++sp) {
    const float m2 = a.part[((size_t)row * a.splits + sp) * 2 + 0];
    const float s2 = a.part[((size_t)row * a.splits + sp) * 2 + 1];
    const float mm = fmaxf(M, m2);
    S = (mm == -INFINITY) ? 0.f : S * expf(M - mm) + s2 * expf(m2 - mm);
    M = mm;
  }
  const float c = 1.f / S;
  a.conf[row] = c;
  if (a.conf_user) a.conf_user[row] = c;
  const int p = a.start + j;
  const bool valid = p < a.N;
  const bool msk = valid && a.masked[(size_t)s * a.N + p] != 0;
  bool commit = false;
  float drel = 0.f, taud = 0.f;
  if (j < B) {
    if (a.block_entry) {
      commit = msk && (c >= a.tau_s);
      a.theta_n[s * B + j] = 0;
    } else {
      float* th = a.theta + ((size_t)s * B + j) * (a.hist > 0 ? a.hist : 1);
      int n = a.theta_n[s * B + j];
      float mean = 0.f;
      if (n > 0) {
        float sum = 0.f;
        for (int i = 0; i < n; ++i) sum += th[i];
        mean = sum / (float)n;
      }
      const float dj = a.delta[s * B + j];
      drel = dj - mean;
      if (a.hist > 0) {
        if (n < a.hist) {
          th[n] = dj;
          ++n;
        } else {
          for (int i = 0; i + 1 < a.hist; ++i) th[i] = th[i + 1];
          th[a.hist - 1] = dj;
        }
        a.theta_n[s * B + j] = n;
      }
      const float g = a.tau_s - c;
      taud = a.alpha * g * g;
      commit = msk && ((c >= a.tau_s) || (drel >= taud));
    }
  } else if (!a.block_entry && valid && a.fire[s]) {
    int widx = -1;
    for (int w = 0; w < a.nw; ++w)
      if (a.win_pos[w] == p) widx = w;
    const bool sel = widx >= 0 && a.sel_last[(size_t)s * a.Wmax + widx];
    commit = msk && sel && (c >= a.tau_suf);
  }
  a.commit[row] = commit;
  a.drel[row] = drel;
  a.taud[row] = taud;
}

void launch_commit(const CommitArgs& a, cudaStream_t st) {
  launch_pdl(conf_partial_kernel, dim3(a.batch * 2 * a.B, a.splits), dim3(256), 0, st, a);
  launch_pdl(commit_gate_kernel, dim3(a.batch), dim3(2 * a.B), 0, st, a);
}

}  // namespace polestar
