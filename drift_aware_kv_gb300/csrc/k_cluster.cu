// Window clustering and the NVFP4 residual store (Polestar-Cache, §4.1
// "Cluster and Quantize Hidden States"; App. C.3; Algorithm 1's clustering,
// quantisation, dequantisation, patch and update steps).
//
//   kmeans_encode_kernel  one CTA per (layer, sequence): spherical K-means on the
//                         block-entry window inputs, member sums, residual
//                         anchors, then NVFP4 encoding of every row's residual.
//   window_patch_kernel   within-block: decode a window row, swap in its update
//                         packet when the previous layer selected it, re-encode
//                         it and record the change of its unit direction.
//   centroid_sum/norm     s_c += sum of those changes (window order),
//                         z_c = s_c / |s_c| (incremental centroid update).
#include "kernels.h"

namespace polestar {

constexpr int KM_THREADS = 512;
constexpr int KM_MAXK = 8;
constexpr int KM_DPT = 8;      // dims per thread in the update step (d <= 4096)
constexpr int KM_MAXW = 128;   // rows per problem

__device__ __forceinline__ uint64_t splitmix64_next(uint64_t& x) {
  x += 0x9E3779B97F4A7C15ull;
  uint64_t z = x;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void __launch_bounds__(KM_THREADS) kmeans_encode_kernel(KmeansArgs a) {
  pdl_enter();
  extern __shared__ float sm[];
  float* zs = sm;                                  // [K][d] centroids, later anchors
  float* inv = zs + (size_t)a.K * a.d;             // [KM_MAXW] 1/|x_i|
  float* red = inv + KM_MAXW;                      // [32 * KM_MAXK]
  int* lab = (int*)(red + 32 * KM_MAXK);           // [KM_MAXW]
  int* perm = lab + KM_MAXW;                       // [KM_MAXW]
  int* cnt = perm + KM_MAXW;                       // [KM_MAXK]

  const int prob = blockIdx.x;                     // = layer * batch + seq
  const int layer = prob / a.batch, seq = prob % a.batch;
  const int d = a.d, K = a.K, nw = a.nw;
  const float* X = a.Hw + (size_t)prob * a.Wmax * d;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = KM_THREADS / 32;

  // 1/|x_i|
  for (int i = warp; i < nw; i += nwarps) {
    float ss = 0.f;
    for (int k = lane; k < d; k += 32) ss = fmaf(X[(size_t)i * d + k], X[(size_t)i * d + k], ss);
    ss = warp_sum(ss);
    if (lane == 0) inv[i] = 1.f / sqrtf(ss);
  }
  // seeded initialisation: first K entries of a Fisher-Yates permutation
  if (tid == 0) {
    uint64_t st = a.seed ^ ((uint64_t)seq << 40) ^ ((uint64_t)a.block << 20) ^ (uint64_t)layer;
    for (int i = 0; i < nw; ++i) perm[i] = i;
    for (int i = nw - 1; i > 0; --i) {
      const int j = (int)(splitmix64_next(st) % (uint64_t)(i + 1));
      const int t = perm[i];
      perm[i] = perm[j];
      perm[j] = t;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < K * d; idx += KM_THREADS) {
    const int c = idx / d, k = idx % d;
    const int src = perm[c];
    zs[idx] = X[(size_t)src * d + k] * inv[src];
  }
  __syncthreads();

  float acc[KM_MAXK][KM_DPT];
  for (int it = 0; it < a.iters; ++it) {
    // assignment: argmax cosine, ties to the lower id
    if (tid < K) cnt[tid] = 0;
    __syncthreads();
    for (int i = warp; i < nw; i += nwarps) {
      float dot[KM_MAXK];
#pragma unroll
      for (int c = 0; c < KM_MAXK; ++c) dot[c] = 0.f;
      for (int k = lane; k < d; k += 32) {
        const float x = X[(size_t)i * d + k];
#pragma unroll
        for (int c = 0; c < KM_MAXK; ++c)
          if (c < K) dot[c] = fmaf(x, zs[c * d + k], dot[c]);
      }
      int best = 0;
      float bv = -INFINITY;
#pragma unroll
      for (int c = 0; c < KM_MAXK; ++c) {
        if (c < K) {
          const float cs = warp_sum(dot[c]) * inv[i];
          if (cs > bv) {
            bv = cs;
            best = c;
          }
        }
      }
      if (lane == 0) {
        lab[i] = best;
        atomicAdd(&cnt[best], 1);
      }
    }
    __syncthreads();
    // update: s_c = sum of member unit vectors (row order), z_c = s_c / |s_c|
#pragma unroll
    for (int c = 0; c < KM_MAXK; ++c)
#pragma unroll
      for (int t = 0; t < KM_DPT; ++t) acc[c][t] = 0.f;
    for (int i = 0; i < nw; ++i) {
      const int c = lab[i];
      const float w = inv[i];
#pragma unroll
      for (int t = 0; t < KM_DPT; ++t) {
        const int k = tid + t * KM_THREADS;
        if (k < d) {
          const float v = X[(size_t)i * d + k] * w;
#pragma unroll
          for (int cc = 0; cc < KM_MAXK; ++cc)
            if (cc == c) acc[cc][t] += v;
        }
      }
    }
    const bool last = (it == a.iters - 1);
    for (int c = 0; c < K; ++c) {
      float ss = 0.f;
#pragma unroll
      for (int t = 0; t < KM_DPT; ++t) ss = fmaf(acc[c][t], acc[c][t], ss);
      ss = block_sum(ss, red);
      const float nrm = sqrtf(ss);
      float* csum = a.csum + ((size_t)prob * K + c) * d;
#pragma unroll
      for (int t = 0; t < KM_DPT; ++t) {
        const int k = tid + t * KM_THREADS;
        if (k < d) {
          if (cnt[c] > 0) zs[c * d + k] = acc[c][t] / nrm;
          if (last) csum[k] = (cnt[c] > 0) ? acc[c][t] : zs[c * d + k];
        }
      }
    }
    __syncthreads();
  }
  // outputs: labels, centroids
  for (int i = tid; i < nw; i += KM_THREADS) a.labels[(size_t)prob * a.Wmax + i] = (uint8_t)lab[i];
  for (int idx = tid; idx < K * d; idx += KM_THREADS) a.z[(size_t)prob * K * d + idx] = zs[idx];
  __syncthreads();
  // anchors A_c: raw member means (reuse zs)
#pragma unroll
  for (int c = 0; c < KM_MAXK; ++c)
#pragma unroll
    for (int t = 0; t < KM_DPT; ++t) acc[c][t] = 0.f;
  for (int i = 0; i < nw; ++i) {
    const int c = lab[i];
#pragma unroll
    for (int t = 0; t < KM_DPT; ++t) {
      const int k = tid + t * KM_THREADS;
      if (k < d) {
        const float v = X[(size_t)i * d + k];
#pragma unroll
        for (int cc = 0; cc < KM_MAXK; ++cc)
          if (cc == c) acc[cc][t] += v;
      }
    }
  }
  for (int c = 0; c < K; ++c) {
    float* an = a.anchor + ((size_t)prob * K + c) * d;
#pragma unroll
    for (int t = 0; t < KM_DPT; ++t) {
      const int k = tid + t * KM_THREADS;
      if (k < d) {
        const float v = (cnt[c] > 0) ? acc[c][t] / (float)cnt[c] : 0.f;
        zs[c * d + k] = v;
        an[k] = v;
      }
    }
  }
  __syncthreads();
  // NVFP4 residual encoding: one warp per row, one lane per 16-element group
  const int ng = d / 16;
  for (int i = warp; i < nw; i += nwarps) {
    const int c = lab[i];
    uint8_t* crow = a.codes + ((size_t)prob * a.Wmax + i) * (d / 2);
    uint8_t* srow = a.scales + ((size_t)prob * a.Wmax + i) * ng;
    for (int g = lane; g < ng; g += 32) {
      float r[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) r[e] = X[(size_t)i * d + g * 16 + e] - zs[c * d + g * 16 + e];
      uint8_t packed[8];
      srow[g] = nvfp4_encode16(r, packed);
      uint2 pk;
      pk.x = packed[0] | (packed[1] << 8) | (packed[2] << 16) | ((uint32_t)packed[3] << 24);
      pk.y = packed[4] | (packed[5] << 8) | (packed[6] << 16) | ((uint32_t)packed[7] << 24);
      *(uint2*)(crow + g * 8) = pk;
    }
  }
}

void launch_kmeans_encode(const KmeansArgs& a, cudaStream_t st) {
  const size_t sm = (size_t)a.K * a.d * sizeof(float) + KM_MAXW * sizeof(float) +
                    32 * KM_MAXK * sizeof(float) + (2 * KM_MAXW + KM_MAXK) * sizeof(int);
  cudaFuncSetAttribute(kmeans_encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  launch_pdl(kmeans_encode_kernel, dim3(a.L * a.batch), dim3(KM_THREADS), sm, st, a);
}

// ---------------------------------------------------------------- within-block
__global__ void window_patch_kernel(PatchArgs a) {
  pdl_enter();
  __shared__ float red[32];
  const int j = blockIdx.x, f = blockIdx.y;
  const int s = a.fire_seqs[f];
  const int d = a.d, ng = d / 16;
  const int row = a.win_row[s] + j;
  const int c = a.labels[s * a.Wmax + j];
  const float* A = a.anchor + ((size_t)s * a.K + c) * d;
  uint8_t* crow = a.codes + ((size_t)s * a.Wmax + j) * (d / 2);
  uint8_t* srow = a.scales + ((size_t)s * a.Wmax + j) * ng;
  const bool patched = a.sel_prev[s * a.Wmax + j] != 0;
  const float* Urow = a.U + ((size_t)s * a.Wmax + j) * d;
  float* hrow = a.h_rows + (size_t)row * d;
  float* dnrow = a.dn + ((size_t)s * a.Wmax + j) * d;

  float ss_old = 0.f, ss_new = 0.f;
  // pass 1: decode, write the patched row, norms
  for (int g = threadIdx.x; g < ng; g += blockDim.x) {
    const float sc = e4m3_decode(srow[g]);
    const uint2 pk = *(const uint2*)(crow + g * 8);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t word = (e < 8) ? pk.x : pk.y;
      const uint32_t code = (word >> (4 * (e & 7))) & 0xF;
      const float old = A[g * 16 + e] + e2m1_decode(code) * sc;
      const float nv = patched ? Urow[g * 16 + e] : old;
      ss_old = fmaf(old, old, ss_old);
      ss_new = fmaf(nv, nv, ss_new);
      hrow[g * 16 + e] = nv;
      if (patched) dnrow[g * 16 + e] = old;  // stash old value; finished below
    }
  }
  if (!patched) {
    if (threadIdx.x == 0) a.write_kv[row] = 0;
    return;
  }
  ss_old = block_sum(ss_old, red);
  ss_new = block_sum(ss_new, red);
  const float io = 1.f / sqrtf(ss_old), in = 1.f / sqrtf(ss_new);
  // pass 2: direction change and re-encoding of the new residual
  for (int g = threadIdx.x; g < ng; g += blockDim.x) {
    float r[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int k = g * 16 + e;
      const float nv = Urow[k];
      dnrow[k] = nv * in - dnrow[k] * io;
      r[e] = nv - A[k];
    }
    uint8_t packed[8];
    srow[g] = nvfp4_encode16(r, packed);
    uint2 pk;
    pk.x = packed[0] | (packed[1] << 8) | (packed[2] << 16) | ((uint32_t)packed[3] << 24);
    pk.y = packed[4] | (packed[5] << 8) | (packed[6] << 16) | ((uint32_t)packed[7] << 24);
    *(uint2*)(crow + g * 8) = pk;
  }
  if (threadIdx.x == 0) a.write_kv[row] = 1;
}

// s_c += sum over the patched member rows (window order) of their direction
// change; one thread per channel, all clusters of one sequence per CTA column.
__global__ void centroid_sum_kernel(PatchArgs a) {
  pdl_enter();
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  const int s = a.fire_seqs[blockIdx.y];
  if (k >= a.d) return;
  const uint8_t* lab = a.labels + (size_t)s * a.Wmax;
  const uint8_t* sel = a.sel_prev + (size_t)s * a.Wmax;
  float acc[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) acc[c] = 0.f;
  for (int j = 0; j < a.nw; ++j) {
    if (!sel[j]) continue;  // uniform across the CTA
    const int c = lab[j];
    const float v = a.dn[((size_t)s * a.Wmax + j) * a.d + k];
#pragma unroll
    for (int cc = 0; cc < 8; ++cc)
      if (cc == c) acc[cc] += v;
  }
  float* cs = a.csum + (size_t)s * a.K * a.d;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    if (c < a.K) cs[(size_t)c * a.d + k] += acc[c];
}

// z_c = s_c / |s_c| for every cluster of a refreshing sequence
__global__ void centroid_norm_kernel(PatchArgs a) {
  pdl_enter();
  __shared__ float red[32];
  const int c = blockIdx.x, s = a.fire_seqs[blockIdx.y];
  const float* cs = a.csum + ((size_t)s * a.K + c) * a.d;
  float* z = a.z + ((size_t)s * a.K + c) * a.d;
  float ss = 0.f;
  for (int k = threadIdx.x; k < a.d; k += blockDim.x) ss = fmaf(cs[k], cs[k], ss);
  ss = block_sum(ss, red);
  const float nrm = sqrtf(ss);
  for (int k = threadIdx.x; k < a.d; k += blockDim.x) z[k] = cs[k] / nrm;
}

void launch_window_patch(const PatchArgs& a, cudaStream_t st) {
  launch_pdl(window_patch_kernel, dim3(a.nw, a.n_fire), dim3(256), 0, st, a);
}
void launch_centroid_update(const PatchArgs& a, cudaStream_t st) {
  launch_pdl(centroid_sum_kernel, dim3((a.d + 127) / 128, a.n_fire), dim3(128), 0, st, a);
  launch_pdl(centroid_norm_kernel, dim3(a.K, a.n_fire), dim3(256), 0, st, a);
}

}  // namespace polestar
