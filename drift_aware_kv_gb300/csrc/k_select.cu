// Drift aggregation, top-k cluster selection and gathered-row compaction
// (Polestar-Cache, §4.1 "Measuring Drift and Layer-wise KV Updates";
// Algorithm 1, drift / TopK / member-index steps).
//
// One CTA serves the whole batch (at most a few thousand window rows): per
// refreshing sequence it averages the per-head proxy KL into D_c, picks the k
// largest (ties to the lower cluster id), marks the member rows S, and writes
// the compact row list [active rows of every sequence, then S of each
// refreshing sequence in window order] with its length on the device, so the
// following projections run on exactly those rows without a host round trip.
#include "kernels.h"

namespace polestar {

constexpr int SEL_MAX_SEQ = 32;    // sequences one launch serves
constexpr int SEL_MAX_WORDS = 4;   // 32-row words of a sequence's window (up to 128 rows)

__global__ void select_kernel(SelectArgs a) {
  __shared__ int s_taken[SEL_MAX_SEQ];
  __shared__ int s_count[SEL_MAX_SEQ + 1];
  __shared__ unsigned s_sel[SEL_MAX_SEQ][SEL_MAX_WORDS];  // selection ballots, reused by the compaction
  __shared__ uint8_t s_lab[SEL_MAX_SEQ][SEL_MAX_WORDS * 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  // window labels are written at the block entry, never by a kernel of this
  // step: they are read before waiting for the attention kernel
  for (int i = tid; i < a.batch * a.nw; i += blockDim.x) {
    const int s = i / a.nw, j = i % a.nw;
    s_lab[s][j] = (uint8_t)a.labels[(size_t)s * a.Wmax + j];
  }
  pdl_enter();
  // 1. per sequence (one warp): D_c = mean over heads of the proxy KL (lanes
  //    over heads, every cluster's loads in flight together), then top-k
  for (int s = warp; s < a.batch; s += nwarps) {
    const int pr = a.proxy_row[s];
    float* D = a.drift + (size_t)s * a.K;
    int* tk = a.topk_out + (size_t)s * a.topk;
    if (pr < 0) {
      if (lane < a.K) D[lane] = 0.f;
      if (lane < a.topk) tk[lane] = -1;
      continue;
    }
    float Dv[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) Dv[c] = 0.f;
    for (int h0 = 0; h0 < a.H; h0 += 32) {
      const int h = h0 + lane;
      float v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) v[c] = (c < a.K && h < a.H) ? a.kl_rows[(size_t)(pr + c) * a.H + h] : 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) Dv[c] += v[c];
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      Dv[c] = warp_sum(Dv[c]) / (float)a.H;
      if (lane == 0 && c < a.K) D[c] = Dv[c];
    }
    if (lane == 0) {
      unsigned taken = 0;
      for (int i = 0; i < a.topk; ++i) {
        int best = -1;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (c >= a.K || (taken & (1u << c))) continue;
          if (best < 0 || Dv[c] > Dv[best]) best = c;
        }
        taken |= 1u << best;
        tk[i] = best;
      }
      s_taken[s] = (int)taken;
    }
  }
  __syncthreads();
  // 2. selection masks and per-sequence counts (warp per sequence)
  for (int s = warp; s < a.batch; s += nwarps) {
    const bool fire = a.proxy_row[s] >= 0;
    const unsigned taken = fire ? (unsigned)s_taken[s] : 0u;
    int count = 0;
    for (int j0 = 0; j0 < a.Wmax; j0 += 32) {
      const int j = j0 + lane;
      bool sel = false;
      if (fire && j < a.nw) sel = (taken >> s_lab[s][j]) & 1u;
      if (j < a.Wmax) {
        a.selected[(size_t)s * a.Wmax + j] = sel;
        a.sel_cur[(size_t)s * a.Wmax + j] = sel;
      }
      const unsigned bal = __ballot_sync(0xffffffffu, sel);
      if (lane == 0 && j0 / 32 < SEL_MAX_WORDS) s_sel[s][j0 / 32] = bal;
      count += __popc(bal);
    }
    if (lane == 0) s_count[s] = count;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = a.n_active;
    for (int s = 0; s < a.batch; ++s) {
      const int c = s_count[s];
      s_count[s] = acc;
      acc += c;
    }
    *a.m_o = acc;
  }
  __syncthreads();
  for (int i = tid; i < a.n_active; i += blockDim.x) a.o_src[i] = i;
  // 3. compact row list
  for (int s = warp; s < a.batch; s += nwarps) {
    if (a.proxy_row[s] < 0) continue;
    int base = s_count[s];
    for (int j0 = 0; j0 < a.nw; j0 += 32) {
      const unsigned bal = s_sel[s][j0 / 32];
      if ((bal >> lane) & 1u) a.o_src[base + __popc(bal & ((1u << lane) - 1u))] = a.win_row[s] + j0 + lane;
      base += __popc(bal);
    }
  }
}

void launch_select(const SelectArgs& a, cudaStream_t st) { launch_pdl(select_kernel, dim3(1), dim3(1024), 0, st, a); }

// delta_j = mean over heads of the last-layer active-row KL (§4.2; Algorithm 1, last-layer drift step)
__global__ void delta_kernel(const float* __restrict__ kl_rows, int batch, int B, int H,
                             float* __restrict__ delta) {
  pdl_enter();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= batch * B) return;
  float sum = 0.f;
  for (int h = 0; h < H; ++h) sum += kl_rows[(size_t)i * H + h];
  delta[i] = sum / (float)H;
}

void launch_delta_finalize(const float* kl_rows, int batch, int B, int H, float* delta, cudaStream_t st) {
  launch_pdl(delta_kernel, dim3((batch * B + 127) / 128), dim3(128), 0, st, kl_rows, batch, B, H, delta);
}

}  // namespace polestar
