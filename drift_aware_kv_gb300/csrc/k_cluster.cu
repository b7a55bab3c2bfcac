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

constexpr int KM_THREADS = 256;
constexpr int KM_MAXK = 8;
constexpr int KM_MAXW = 128;   // rows per problem
constexpr int KM_SMEM_CAP = 220 * 1024;

__device__ __forceinline__ uint64_t splitmix64_next(uint64_t& x) {
  x += 0x9E3779B97F4A7C15ull;
  uint64_t z = x;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint32_t km_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void km_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float km_ld_remote(const float* local, uint32_t rank) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(local), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// out[i] = sum over the cluster's CTAs (rank order) of part[i], i < n.  Every
// CTA ends with the same values; `part` may be rewritten after the call.
__device__ __forceinline__ void km_allreduce(const float* part, float* out, int n, int cs) {
  km_cluster_sync();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    float v[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = (q < cs) ? km_ld_remote(part + i, (uint32_t)q) : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q) acc += v[q];  // rank order; absent ranks add +0
    out[i] = acc;
  }
  km_cluster_sync();
}

// One thread-block cluster per (layer, sequence) problem; CTA r of the cluster
// owns channels [r*ds, (r+1)*ds) of the window rows, held in shared memory for
// the whole K-means, so the rows are read from memory once.
__global__ void __launch_bounds__(KM_THREADS) kmeans_encode_kernel(KmeansArgs a, int cs) {
  pdl_enter();
  extern __shared__ __align__(16) float sm[];
  const int d = a.d, K = a.K, nw = a.nw;
  const int ds = d / cs;
  const uint32_t rank = km_rank();
  const int prob = blockIdx.x / cs;                    // = layer * batch + seq
  const int layer = prob / a.batch, seq = prob % a.batch;
  const int c0 = (int)rank * ds;
  float* Xs = sm;                                      // [nw][ds]
  float* zs = Xs + (size_t)nw * ds;                    // [K][ds]
  float* part = zs + (size_t)K * ds;                   // [KM_MAXW * KM_MAXK] partial sums
  float* full = part + KM_MAXW * KM_MAXK;              // [KM_MAXW * KM_MAXK] reduced sums
  float* inv = full + KM_MAXW * KM_MAXK;               // [KM_MAXW]
  float* red = inv + KM_MAXW;                          // [32] block-reduction scratch
  int* lab = (int*)(red + 32);                         // [KM_MAXW]
  int* perm = lab + KM_MAXW;                           // [KM_MAXW]
  int* cnt = perm + KM_MAXW;                           // [KM_MAXK]
  const int tid = threadIdx.x;
  const float* X = a.Hw + (size_t)prob * a.Wmax * d;

  // stage the channel slice of every row
  for (int idx = tid; idx < nw * (ds / 4); idx += KM_THREADS) {
    const int i = idx / (ds / 4), k4 = idx % (ds / 4);
    *(float4*)(Xs + (size_t)i * ds + k4 * 4) = *(const float4*)(X + (size_t)i * d + c0 + k4 * 4);
  }
  __syncthreads();
  // 1/|x_i|: slice partials (warp per row, lanes across channels), cluster sum
  {
    const int lane = tid & 31, warp = tid >> 5;
    for (int i = warp; i < nw; i += KM_THREADS / 32) {
      float ss = 0.f;
      for (int k = lane; k < ds; k += 32) ss = fmaf(Xs[(size_t)i * ds + k], Xs[(size_t)i * ds + k], ss);
      ss = warp_sum(ss);
      if (lane == 0) part[i] = ss;
    }
  }
  __syncthreads();
  km_allreduce(part, full, nw, cs);
  for (int i = tid; i < nw; i += KM_THREADS) inv[i] = 1.f / sqrtf(full[i]);
  // seeded initialisation (every CTA draws the same permutation)
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
  for (int idx = tid; idx < K * ds; idx += KM_THREADS) {
    const int c = idx / ds, k = idx % ds;
    zs[idx] = Xs[(size_t)perm[c] * ds + k] * inv[perm[c]];
  }
  __syncthreads();

  constexpr int DPT = 2;  // channels per thread in the update (ds <= 512)
  float acc[KM_MAXK][DPT];
  for (int it = 0; it < a.iters; ++it) {
    // assignment: cosine = (sum over slices of x.z) / |x|, argmax, ties to the lower id.
    // Warp per row, lanes across channels (conflict-free shared-memory reads).
    {
      const int lane = tid & 31, warp = tid >> 5;
      for (int i = warp; i < nw; i += KM_THREADS / 32) {
        float dot[KM_MAXK];
#pragma unroll
        for (int c = 0; c < KM_MAXK; ++c) dot[c] = 0.f;
        for (int k = lane; k < ds; k += 32) {
          const float x = Xs[(size_t)i * ds + k];
#pragma unroll
          for (int c = 0; c < KM_MAXK; ++c)
            if (c < K) dot[c] = fmaf(x, zs[c * ds + k], dot[c]);
        }
#pragma unroll
        for (int c = 0; c < KM_MAXK; ++c) {
          const float v = warp_sum(dot[c]);
          if (lane == 0 && c < K) part[i * K + c] = v;
        }
      }
    }
    __syncthreads();
    km_allreduce(part, full, nw * K, cs);
    if (tid < K) cnt[tid] = 0;
    __syncthreads();
    for (int i = tid; i < nw; i += KM_THREADS) {
      int best = 0;
      float bv = -INFINITY;
      for (int c = 0; c < K; ++c) {
        const float v = full[i * K + c] * inv[i];
        if (v > bv) {
          bv = v;
          best = c;
        }
      }
      lab[i] = best;
      atomicAdd(&cnt[best], 1);
    }
    __syncthreads();
    // update: s_c = sum of member unit rows (row order) on this slice
#pragma unroll
    for (int c = 0; c < KM_MAXK; ++c)
#pragma unroll
      for (int t = 0; t < DPT; ++t) acc[c][t] = 0.f;
    for (int i = 0; i < nw; ++i) {
      const int c = lab[i];
      const float w = inv[i];
#pragma unroll
      for (int t = 0; t < DPT; ++t) {
        const int k = tid + t * KM_THREADS;
        if (k < ds) {
          const float v = Xs[(size_t)i * ds + k] * w;
#pragma unroll
          for (int cc = 0; cc < KM_MAXK; ++cc)
            if (cc == c) acc[cc][t] += v;
        }
      }
    }
    // |s_c|^2: per-thread partials, block reduce per cluster, cluster sum
    for (int c = 0; c < K; ++c) {
      float ss = 0.f;
#pragma unroll
      for (int t = 0; t < DPT; ++t) ss = fmaf(acc[c][t], acc[c][t], ss);
      ss = block_sum(ss, red);
      if (tid == 0) part[c] = ss;
    }
    __syncthreads();
    km_allreduce(part, full, K, cs);
    const bool last = (it == a.iters - 1);
    for (int c = 0; c < K; ++c) {
      const float nrm = sqrtf(full[c]);
      float* csum = a.csum + ((size_t)prob * K + c) * d + c0;
#pragma unroll
      for (int t = 0; t < DPT; ++t) {
        const int k = tid + t * KM_THREADS;
        if (k < ds) {
          if (cnt[c] > 0) zs[c * ds + k] = acc[c][t] / nrm;
          if (last) csum[k] = (cnt[c] > 0) ? acc[c][t] : zs[c * ds + k];
        }
      }
    }
    __syncthreads();
  }
  // outputs: labels, centroid slices
  if (rank == 0)
    for (int i = tid; i < nw; i += KM_THREADS) a.labels[(size_t)prob * a.Wmax + i] = (uint8_t)lab[i];
  for (int idx = tid; idx < K * ds; idx += KM_THREADS) {
    const int c = idx / ds, k = idx % ds;
    a.z[((size_t)prob * K + c) * d + c0 + k] = zs[idx];
  }
  __syncthreads();
  // anchors A_c: raw member means on this slice (reuse zs)
#pragma unroll
  for (int c = 0; c < KM_MAXK; ++c)
#pragma unroll
    for (int t = 0; t < DPT; ++t) acc[c][t] = 0.f;
  for (int i = 0; i < nw; ++i) {
    const int c = lab[i];
#pragma unroll
    for (int t = 0; t < DPT; ++t) {
      const int k = tid + t * KM_THREADS;
      if (k < ds) {
        const float v = Xs[(size_t)i * ds + k];
#pragma unroll
        for (int cc = 0; cc < KM_MAXK; ++cc)
          if (cc == c) acc[cc][t] += v;
      }
    }
  }
  for (int c = 0; c < K; ++c) {
    float* an = a.anchor + ((size_t)prob * K + c) * d + c0;
#pragma unroll
    for (int t = 0; t < DPT; ++t) {
      const int k = tid + t * KM_THREADS;
      if (k < ds) {
        const float v = (cnt[c] > 0) ? acc[c][t] / (float)cnt[c] : 0.f;
        zs[c * ds + k] = v;
        an[k] = v;
      }
    }
  }
  __syncthreads();
  // NVFP4 residual encoding of this slice: one thread per 16-channel group
  const int ngs = ds / 16, ng = d / 16;
  for (int idx = tid; idx < nw * ngs; idx += KM_THREADS) {
    const int i = idx / ngs, g = idx % ngs;
    const int c = lab[i];
    float r[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) r[e] = Xs[(size_t)i * ds + g * 16 + e] - zs[c * ds + g * 16 + e];
    uint8_t packed[8];
    const int gg = c0 / 16 + g;
    a.scales[((size_t)prob * a.Wmax + i) * ng + gg] = nvfp4_encode16(r, packed);
    uint2 pk;
    pk.x = packed[0] | (packed[1] << 8) | (packed[2] << 16) | ((uint32_t)packed[3] << 24);
    pk.y = packed[4] | (packed[5] << 8) | (packed[6] << 16) | ((uint32_t)packed[7] << 24);
    *(uint2*)(a.codes + ((size_t)prob * a.Wmax + i) * (d / 2) + gg * 8) = pk;
  }
}

// Cluster size: the smallest divisor of d/16 (<= 16) whose channel slice fits
// in shared memory and keeps <= 2 channels per thread.
int kmeans_cluster_size(int d, int nw, int K) {
  const int groups = d / 16;
  for (int cs = 1; cs <= 16; ++cs) {
    if (groups % cs) continue;
    const int ds = d / cs;
    const size_t sm = ((size_t)nw * ds + (size_t)K * ds + 2 * KM_MAXW * KM_MAXK + KM_MAXW + 32) * sizeof(float) +
                      (3 * KM_MAXW + KM_MAXK) * sizeof(int);
    if (ds <= 2 * KM_THREADS && sm <= (size_t)KM_SMEM_CAP) return cs;
  }
  return -1;
}

void launch_kmeans_encode(const KmeansArgs& a, cudaStream_t st) {
  const int cs = kmeans_cluster_size(a.d, a.nw, a.K);
  const int ds = a.d / cs;
  const size_t sm = ((size_t)a.nw * ds + (size_t)a.K * ds + 2 * KM_MAXW * KM_MAXK + KM_MAXW + 32) * sizeof(float) +
                    (3 * KM_MAXW + KM_MAXK) * sizeof(int);
  cudaFuncSetAttribute(kmeans_encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (cs > 8) cudaFuncSetAttribute(kmeans_encode_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.L * a.batch * cs);
  cfg.blockDim = dim3(KM_THREADS);
  cfg.dynamicSmemBytes = sm;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, kmeans_encode_kernel, a, cs);
}

// ---------------------------------------------------------------- within-block
template <typename T>
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
  ss_old = block_sum(ss_old, red);
  ss_new = block_sum(ss_new, red);
  // fused input of the layer's projections: RMSNorm of the (patched) row
  {
    const float inv = 1.f / sqrtf(ss_new / (float)d + a.eps);
    const T* gain = (const T*)a.gain;
    T* ao = (T*)a.a_out + (size_t)row * d;
    for (int k = threadIdx.x; k < d; k += blockDim.x) ao[k] = from_f<T>(hrow[k] * inv * to_f<T>(gain[k]));
  }
  if (!patched) {
    if (threadIdx.x == 0) a.write_kv[row] = 0;
    return;
  }
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

// z_c = s_c / |s_c| for every cluster of a refreshing sequence, and the proxy
// row's projection input T(RMSNorm(z_c) * gain)
template <typename T>
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
  float zz = 0.f;
  for (int k = threadIdx.x; k < a.d; k += blockDim.x) {
    const float v = cs[k] / nrm;
    z[k] = v;
    zz = fmaf(v, v, zz);
  }
  zz = block_sum(zz, red);
  const float inv = 1.f / sqrtf(zz / (float)a.d + a.eps);
  const T* gain = (const T*)a.gain;
  T* ao = (T*)a.a_out + (size_t)(a.proxy_row[s] + c) * a.d;
  for (int k = threadIdx.x; k < a.d; k += blockDim.x) ao[k] = from_f<T>(z[k] * inv * to_f<T>(gain[k]));
}

template <typename T>
void launch_window_patch(const PatchArgs& a, cudaStream_t st) {
  launch_pdl(window_patch_kernel<T>, dim3(a.nw, a.n_fire), dim3(256), 0, st, a);
}
template <typename T>
void launch_centroid_update(const PatchArgs& a, cudaStream_t st) {
  launch_pdl(centroid_sum_kernel, dim3((a.d + 127) / 128, a.n_fire), dim3(128), 0, st, a);
  launch_pdl(centroid_norm_kernel<T>, dim3(a.K, a.n_fire), dim3(256), 0, st, a);
}
template void launch_window_patch<float>(const PatchArgs&, cudaStream_t);
template void launch_window_patch<__nv_bfloat16>(const PatchArgs&, cudaStream_t);
template void launch_centroid_update<float>(const PatchArgs&, cudaStream_t);
template void launch_centroid_update<__nv_bfloat16>(const PatchArgs&, cudaStream_t);

}  // namespace polestar
