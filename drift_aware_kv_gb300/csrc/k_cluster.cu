// Window clustering and the NVFP4 residual store (Polestar-Cache, §4.1
// "Cluster and Quantize Hidden States"; App. C.3; Algorithm 1's clustering,
// quantisation, dequantisation, patch and update steps).
//
//   kmeans_encode_kernel    one thread-block cluster per (layer, sequence),
//                           channel slices per CTA: spherical K-means on the
//                           block-entry window inputs, member sums, residual
//                           anchors, then NVFP4 encoding of every row's residual.
//   window_patch_kernel     within-block: decode a window row, swap in its update
//                           packet when the previous layer selected it, re-encode
//                           it and record the change of its unit direction.
//   centroid_update_kernel  one cluster per firing sequence: s_c += sum of those
//                           changes, z_c = s_c / |s_c| (incremental centroid
//                           update) and the proxy rows' projection inputs.
#include "kernels.h"

namespace polestar {

constexpr int KM_THREADS = 512;
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

// One reduce-scatter step of a warp over 2H values v[0 .. 2H) (H a power of
// two), exchanging with lane ^ o: the lane keeps the half selected by bit o of
// its lane index and adds its partner's copy of that half into v[0 .. H).
constexpr int KM_ROWS = 6;  // rows per warp pass of the assignment (6 * KM_MAXK values per lane)
static_assert(KM_MAXK == 8 && KM_ROWS == 6, "the assignment's butterflies map 32 + 16 values onto the lanes");
template <int H>
__device__ __forceinline__ void km_bfly(float* v, int lane, int o = H) {
  const bool up = (lane & o) != 0;
#pragma unroll
  for (int j = 0; j < H; ++j) {
    const float send = up ? v[j] : v[j + H];
    const float keep = up ? v[j + H] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
  }
}

// Floats of each of the kernel's two reduction buffers: the assignment's row x
// cluster dot products, and at least one value per (warp, cluster) for the
// norm reduction.
__host__ __device__ constexpr int km_pair_floats(int nw, int K) {
  return nw * KM_MAXK > (KM_THREADS / 32) * KM_MAXK ? nw * KM_MAXK : (KM_THREADS / 32) * KM_MAXK;
}
__host__ __device__ constexpr size_t km_smem_bytes(int nw, int ds, int K) {
  return ((size_t)nw * ds + (size_t)K * ds + 2 * (size_t)km_pair_floats(nw, K) + KM_MAXW + 32) * sizeof(float) +
         (3 * KM_MAXW + 2 * KM_MAXK + 1) * sizeof(int);
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
  const int local = blockIdx.x / cs;                   // problem of this launch
  const int prob = a.layer0 * a.batch + local;         // = layer * batch + seq
  const int layer = prob / a.batch, seq = prob % a.batch;
  const int c0 = (int)rank * ds;
  float* Xs = sm;                                      // [nw][ds]
  float* zs = Xs + (size_t)nw * ds;                    // [K][ds]
  const int pk = km_pair_floats(nw, K);
  float* part = zs + (size_t)K * ds;                   // [pk] partial sums
  float* full = part + pk;                             // [pk] reduced sums
  float* inv = full + pk;                              // [KM_MAXW]
  float* red = inv + KM_MAXW;                          // [32] block-reduction scratch
  int* lab = (int*)(red + 32);                         // [KM_MAXW]
  int* perm = lab + KM_MAXW;                           // [KM_MAXW]
  int* cnt = perm + KM_MAXW;                           // [KM_MAXK] counts, then [KM_MAXK + 1] list starts
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
  // seeded initialisation (every CTA draws the same permutation).  Fisher-Yates
  // step t (i = nw-1-t, swap perm[i] with perm[j], j = draw_t mod (i+1)) takes
  // output t of splitmix64; output t is the mix of state st0 + (t+1) * golden,
  // so the targets are computed in parallel (into lab, free until the first
  // assignment) and only the swaps run in order.
  {
    const uint64_t st0 = a.seed ^ ((uint64_t)seq << 40) ^ ((uint64_t)a.block << 20) ^ (uint64_t)layer;
    for (int t = tid; t < nw - 1; t += KM_THREADS) {
      uint64_t st = st0 + (uint64_t)t * 0x9E3779B97F4A7C15ull;
      const uint64_t x = splitmix64_next(st);
      // x mod m with 32-bit operations (exact: m <= KM_MAXW): x = hi * 2^32 + lo,
      // so x mod m = ((hi mod m) * (2^32 mod m) + lo mod m) mod m
      const uint32_t m = (uint32_t)(nw - t), hi = (uint32_t)(x >> 32), lo = (uint32_t)x;
      const uint32_t p32 = (uint32_t)((0x100000000ull) % m);
      lab[t] = (int)(((hi % m) * p32 + lo % m) % m);
    }
    for (int i = tid; i < nw; i += KM_THREADS) perm[i] = i;
    __syncthreads();
    if (tid == 0)
      for (int t = 0; t < nw - 1; ++t) {
        const int i = nw - 1 - t, j = lab[t];
        const int v = perm[i];
        perm[i] = perm[j];
        perm[j] = v;
      }
    __syncthreads();
  }
  for (int idx = tid; idx < K * ds; idx += KM_THREADS) {
    const int c = idx / ds, k = idx % ds;
    zs[idx] = Xs[(size_t)perm[c] * ds + k] * inv[perm[c]];
  }
  __syncthreads();

  // member lists of the last assignment: rows of cluster c, in row order, at
  // mem[mstart[c] .. mstart[c + 1])
  int* mem = perm;  // the permutation is only needed for the initialisation
  int* mstart = cnt + KM_MAXK;
  const int lane = tid & 31, warp = tid >> 5;
  const int k = tid;  // this thread's channel of the slice in the updates (ds <= KM_THREADS)
  float accv[KM_MAXK];
  for (int it = 0; it < a.iters; ++it) {
    // assignment: cosine = (sum over slices of x.z) / |x|, argmax, ties to the lower id.
    // A warp takes KM_ROWS rows at a time, lanes across channels (conflict-free
    // shared-memory reads), so each centroid element is read once per KM_ROWS
    // rows; the per-lane partial dot products are summed over the warp by
    // reduce-scatter butterflies (rows 0-3: 32 values, lane L ends with the
    // total of value L; rows 4-5: 16 values, lanes 2v and 2v+1 with value v).
    for (int i0 = warp * KM_ROWS; i0 < nw; i0 += (KM_THREADS / 32) * KM_ROWS) {
      float dv[KM_ROWS * KM_MAXK];  // dv[r * KM_MAXK + c]
#pragma unroll
      for (int q = 0; q < KM_ROWS * KM_MAXK; ++q) dv[q] = 0.f;
      for (int kk = lane; kk < ds; kk += 32) {
        float zc[KM_MAXK];
#pragma unroll
        for (int c = 0; c < KM_MAXK; ++c) zc[c] = (c < K) ? zs[c * ds + kk] : 0.f;
#pragma unroll
        for (int r = 0; r < KM_ROWS; ++r) {
          const float x = (i0 + r < nw) ? Xs[(size_t)(i0 + r) * ds + kk] : 0.f;
#pragma unroll
          for (int c = 0; c < KM_MAXK; ++c) dv[r * KM_MAXK + c] = fmaf(x, zc[c], dv[r * KM_MAXK + c]);
        }
      }
      km_bfly<16>(dv, lane);
      km_bfly<8>(dv, lane);
      km_bfly<4>(dv, lane);
      km_bfly<2>(dv, lane);
      km_bfly<1>(dv, lane);
      float* d2 = dv + 32;
      km_bfly<8>(d2, lane, 16);
      km_bfly<4>(d2, lane, 8);
      km_bfly<2>(d2, lane, 4);
      km_bfly<1>(d2, lane, 2);
      d2[0] += __shfl_xor_sync(0xffffffffu, d2[0], 1);
      {
        const int r = lane >> 3, c = lane & 7;
        if (i0 + r < nw) part[(i0 + r) * KM_MAXK + c] = dv[0];
      }
      {
        const int v = lane >> 1, r = 4 + (v >> 3), c = v & 7;
        if (!(lane & 1) && i0 + r < nw) part[(i0 + r) * KM_MAXK + c] = d2[0];
      }
    }
    __syncthreads();
    km_allreduce(part, full, nw * KM_MAXK, cs);
    // argmax and the member lists (stable counting sort by label): warp w
    // takes rows 32w + lane; its per-cluster counts go to wcnt, and after one
    // barrier each warp places its members behind those of the earlier
    // clusters and of the earlier warps of the same cluster
    int* wcnt = (int*)red;  // [KM_MAXW / 32][KM_MAXK]
    const int nch = (nw + 31) / 32;
    int best = -1;
    unsigned bal[KM_MAXK];
    if (warp < nch) {
      const int i = warp * 32 + lane;
      if (i < nw) {
        float bv = -INFINITY;
        best = 0;
        const float4 f0 = *(const float4*)(full + i * KM_MAXK), f1 = *(const float4*)(full + i * KM_MAXK + 4);
        const float fr[KM_MAXK] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
        const float w = inv[i];
#pragma unroll
        for (int c = 0; c < KM_MAXK; ++c) {
          const float v = fr[c] * w;
          if (c < K && v > bv) {
            bv = v;
            best = c;
          }
        }
        lab[i] = best;
      }
#pragma unroll
      for (int c = 0; c < KM_MAXK; ++c) {
        bal[c] = __ballot_sync(0xffffffffu, best == c);
        if (lane == 0) wcnt[warp * KM_MAXK + c] = __popc(bal[c]);
      }
    }
    __syncthreads();
    if (warp < nch) {
      int off = 0;  // members of clusters < c, then of earlier warps in cluster c
      const unsigned lt = (1u << lane) - 1u;
#pragma unroll
      for (int c = 0; c < KM_MAXK; ++c) {
        int before = 0, total = 0;
        for (int w2 = 0; w2 < nch; ++w2) {
          const int n = wcnt[w2 * KM_MAXK + c];
          total += n;
          if (w2 < warp) before += n;
        }
        if (best == c) mem[off + before + __popc(bal[c] & lt)] = warp * 32 + lane;
        if (warp == 0 && lane == 0) {
          cnt[c] = total;
          mstart[c] = off;
        }
        off += total;
      }
      if (warp == 0 && lane == 0) mstart[KM_MAXK] = off;
    }
    __syncthreads();
    // update: s_c = sum of member unit rows (row order) on this slice
#pragma unroll
    for (int c = 0; c < KM_MAXK; ++c) {
      accv[c] = 0.f;
      if (c < K && k < ds)
        for (int j = mstart[c]; j < mstart[c + 1]; ++j) {
          const int i = mem[j];
          accv[c] += Xs[(size_t)i * ds + k] * inv[i];
        }
    }
    // |s_c|^2: warp partials (xor tree), then the warps' values (xor tree), cluster sum
#pragma unroll
    for (int c = 0; c < KM_MAXK; ++c) {
      const float v = warp_sum(accv[c] * accv[c]);
      if (lane == 0 && c < K) full[warp * K + c] = v;
    }
    __syncthreads();
    if (warp == 0)
      for (int c = 0; c < K; ++c) {
        const float t = warp_sum(lane < KM_THREADS / 32 ? full[lane * K + c] : 0.f);
        if (lane == 0) part[c] = t;
      }
    __syncthreads();
    km_allreduce(part, full, K, cs);
    const bool last = (it == a.iters - 1);
    if (k < ds)
#pragma unroll
      for (int c = 0; c < KM_MAXK; ++c) {
        if (c >= K) continue;
        float* csum = a.csum + ((size_t)prob * K + c) * d + c0;
        if (cnt[c] > 0) zs[c * ds + k] = accv[c] / sqrtf(full[c]);
        if (last) csum[k] = (cnt[c] > 0) ? accv[c] : zs[c * ds + k];
      }
    __syncthreads();
  }
  // outputs: labels, centroid slices
  if (rank == 0)
    for (int i = tid; i < nw; i += KM_THREADS) a.labels[(size_t)prob * a.Wmax + i] = (uint8_t)lab[i];
  for (int idx = tid; idx < K * ds; idx += KM_THREADS) {
    const int c = idx / ds, kk = idx % ds;
    a.z[((size_t)prob * K + c) * d + c0 + kk] = zs[idx];
  }
  __syncthreads();
  // anchors A_c: raw member means on this slice (reuse zs)
  if (k < ds)
#pragma unroll
    for (int c = 0; c < KM_MAXK; ++c) {
      if (c >= K) continue;
      float acc = 0.f;
      for (int j = mstart[c]; j < mstart[c + 1]; ++j) acc += Xs[(size_t)mem[j] * ds + k];
      const float v = (cnt[c] > 0) ? acc / (float)cnt[c] : 0.f;
      zs[c * ds + k] = v;
      a.anchor[((size_t)prob * K + c) * d + c0 + k] = v;
    }
  __syncthreads();
  // NVFP4 residual encoding of this slice: one thread per 16-channel group,
  // groups of a row on consecutive threads (coalesced code writes).  The four
  // 16-byte quarters of a group are read starting at quarter (g / 2) mod 4, so
  // the eight groups of a quarter-warp hit eight different bank quads.
  const int ngs = ds / 16, ng = d / 16;
  for (int idx = tid; idx < nw * ngs; idx += KM_THREADS) {
    const int i = idx / ngs, g = idx % ngs;
    const int c = lab[i];
    const int rot = (g >> 1) & 3;
    const float* xr = Xs + (size_t)i * ds + g * 16;
    const float* zr = zs + c * ds + g * 16;
    float4 r4[4];  // r4[qq] = quarter (qq + rot) & 3 of the group
    float amax = 0.f;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const int q = (qq + rot) & 3;
      const float4 xv = *(const float4*)(xr + q * 4), zv = *(const float4*)(zr + q * 4);
      r4[qq] = make_float4(xv.x - zv.x, xv.y - zv.y, xv.z - zv.z, xv.w - zv.w);
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(r4[qq].x), fabsf(r4[qq].y)), fmaxf(fabsf(r4[qq].z), fabsf(r4[qq].w))));
    }
    const uint8_t sb = e4m3_encode_rne(__fdiv_rn(amax, 6.f));
    const float sc = e4m3_decode(sb);
    uint64_t pk = 0;
    if (sc > 0.f)
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const int q = (qq + rot) & 3;
        const uint32_t e0 = e2m1_encode_rne(__fdiv_rn(r4[qq].x, sc)), e1 = e2m1_encode_rne(__fdiv_rn(r4[qq].y, sc));
        const uint32_t e2 = e2m1_encode_rne(__fdiv_rn(r4[qq].z, sc)), e3 = e2m1_encode_rne(__fdiv_rn(r4[qq].w, sc));
        const uint64_t bits = (uint64_t)(e0 | (e1 << 4) | (e2 << 8) | (e3 << 12));
        pk |= bits << (16 * q);  // elements 4q .. 4q+3 are bytes 2q, 2q+1
      }
    const int gg = c0 / 16 + g;
    a.scales[((size_t)local * a.Wmax + i) * ng + gg] = sb;
    *(uint2*)(a.codes + ((size_t)local * a.Wmax + i) * (d / 2) + gg * 8) =
        make_uint2((uint32_t)pk, (uint32_t)(pk >> 32));
  }
}

// Cluster size: the smallest divisor of d/16 (<= 16) whose channel slice fits
// in shared memory and gives each thread at most one channel in the updates.
int kmeans_cluster_size(int d, int nw, int K) {
  const int groups = d / 16;
  for (int cs = 1; cs <= 16; ++cs) {
    if (groups % cs) continue;
    const int ds = d / cs;
    if (ds <= KM_THREADS && km_smem_bytes(nw, ds, K) <= (size_t)KM_SMEM_CAP) return cs;
  }
  return -1;
}

void launch_kmeans_encode(const KmeansArgs& a, cudaStream_t st) {
  const int cs = kmeans_cluster_size(a.d, a.nw, a.K);
  const int ds = a.d / cs;
  const size_t sm = km_smem_bytes(a.nw, ds, a.K);
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
__device__ __forceinline__ float4 cl_ld4t(const T* p);
template <>
__device__ __forceinline__ float4 cl_ld4t<float>(const float* p) {
  return *(const float4*)p;
}
template <>
__device__ __forceinline__ float4 cl_ld4t<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *(const uint2*)p;
  const float2 fa = __bfloat1622float2(*(const __nv_bfloat162*)&u.x), fb = __bfloat1622float2(*(const __nv_bfloat162*)&u.y);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
template <typename T>
__device__ __forceinline__ void cl_st4t(T* p, float4 v);
template <>
__device__ __forceinline__ void cl_st4t<float>(float* p, float4 v) {
  *(float4*)p = v;
}
template <>
__device__ __forceinline__ void cl_st4t<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *(const uint32_t*)&a;
  u.y = *(const uint32_t*)&b;
  *(uint2*)p = u;
}

// One window row per CTA; thread g owns NVFP4 group g (16 channels, d <= 4096
// so one group per thread) and keeps its decoded and patched values in
// registers through the decode, the RMSNorm of the projection input and the
// re-encoding.
template <typename T>
__global__ void __launch_bounds__(256) window_patch_kernel(PatchArgs a) {
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
  const int g = threadIdx.x;
  const bool act = g < ng;
  float av[16], old[16], nv[16];
  float ss_old = 0.f, ss_new = 0.f;
  if (act) {
    const float sc = e4m3_decode(srow[g]);
    const uint2 pk = *(const uint2*)(crow + g * 8);
#pragma unroll
    for (int q = 0; q < 4; ++q) *(float4*)&av[4 * q] = *(const float4*)(A + g * 16 + 4 * q);
    if (patched) {
#pragma unroll
      for (int q = 0; q < 4; ++q) *(float4*)&nv[4 * q] = *(const float4*)(Urow + g * 16 + 4 * q);
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t word = (e < 8) ? pk.x : pk.y;
      const uint32_t code = (word >> (4 * (e & 7))) & 0xF;
      old[e] = av[e] + e2m1_decode(code) * sc;
      if (!patched) nv[e] = old[e];
      ss_old = fmaf(old[e], old[e], ss_old);
      ss_new = fmaf(nv[e], nv[e], ss_new);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) *(float4*)(hrow + g * 16 + 4 * q) = *(const float4*)&nv[4 * q];
  }
  ss_old = block_sum(ss_old, red);
  ss_new = block_sum(ss_new, red);
  // fused input of the layer's projections: RMSNorm of the (patched) row
  if (act) {
    const float inv = 1.f / sqrtf(ss_new / (float)d + a.eps);
    const T* gain = (const T*)a.gain + g * 16;
    T* ao = (T*)a.a_out + (size_t)row * d + g * 16;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 gv = cl_ld4t<T>(gain + 4 * q);
      cl_st4t<T>(ao + 4 * q, make_float4(nv[4 * q] * inv * gv.x, nv[4 * q + 1] * inv * gv.y,
                                         nv[4 * q + 2] * inv * gv.z, nv[4 * q + 3] * inv * gv.w));
    }
  }
  if (!patched) {
    if (threadIdx.x == 0) a.write_kv[row] = 0;
    return;
  }
  const float io = 1.f / sqrtf(ss_old), in = 1.f / sqrtf(ss_new);
  if (act) {
    // direction change and re-encoding of the new residual
    float r[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) r[e] = nv[e] - av[e];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *(float4*)(dnrow + g * 16 + 4 * q) =
          make_float4(nv[4 * q] * in - old[4 * q] * io, nv[4 * q + 1] * in - old[4 * q + 1] * io,
                      nv[4 * q + 2] * in - old[4 * q + 2] * io, nv[4 * q + 3] * in - old[4 * q + 3] * io);
    uint8_t packed[8];
    srow[g] = nvfp4_encode16(r, packed);
    uint2 pk;
    pk.x = packed[0] | (packed[1] << 8) | (packed[2] << 16) | ((uint32_t)packed[3] << 24);
    pk.y = packed[4] | (packed[5] << 8) | (packed[6] << 16) | ((uint32_t)packed[7] << 24);
    *(uint2*)(crow + g * 8) = pk;
  }
  if (threadIdx.x == 0) a.write_kv[row] = 1;
}

// Incremental centroid update of one firing sequence on a thread-block cluster
// of `nc` CTAs, CTA r owning channels [r*cw, (r+1)*cw):
//   s_c += sum over selected window rows j with label c of dn_j   (window order
//          within each of the RL row lanes, lanes added in order),
//   z_c  = s_c / |s_c|   (|s_c| summed over the cluster in rank order),
//   a_out[proxy_row + c] = T(RMSNorm(z_c) * gain)   (the proxy row's projection input).
constexpr int CU_THREADS = 256;

template <typename T>
__global__ void __launch_bounds__(CU_THREADS, 2) centroid_update_kernel(PatchArgs a, int nc, int cw) {
  __shared__ float4 part[CU_THREADS][KM_MAXK];  // [row lane * groups + group][cluster]
  __shared__ float nrm_part[1][KM_MAXK], nrm_full[1][KM_MAXK];
  __shared__ float wsum[CU_THREADS / 32][KM_MAXK];
  __shared__ uint8_t sl[KM_MAXW], lb[KM_MAXW];
  const int rank = (int)km_rank();
  const int s = a.fire_seqs[blockIdx.y];
  const int d = a.d, K = a.K, nw = a.nw;
  const int c0 = rank * cw;
  const int G = cw / 4;                              // channel groups of this CTA
  const int RL = G >= CU_THREADS ? 1 : CU_THREADS / G;  // row lanes sharing a group
  const int t = threadIdx.x;
  // inputs that no preceding kernel of the step writes (the block's labels, the
  // norm gain) are read before waiting for the window patch
  const T* gain = (const T*)a.gain;
  const bool one_pass = G <= CU_THREADS;  // each thread finishes at most one channel group
  float4 gv0 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (one_pass && t < G) gv0 = cl_ld4t<T>(gain + c0 + t * 4);
  for (int i = t; i < nw; i += CU_THREADS) lb[i] = a.labels[s * a.Wmax + i];
  pdl_enter();
  for (int i = t; i < nw; i += CU_THREADS) sl[i] = a.sel_prev[s * a.Wmax + i];
  __syncthreads();
  float* cs_base = a.csum + (size_t)s * K * d;
  float ssl[KM_MAXK];
  // this thread's group sums; after the last pass (the only one when one_pass)
  // the updated member sums, reused for z
  float4 acc[KM_MAXK];
#pragma unroll
  for (int c = 0; c < KM_MAXK; ++c) ssl[c] = 0.f;
  // RL > 1: one pass, thread t = lane rl * G + group cg.  RL == 1: group
  // cg = t + k * CU_THREADS in pass k.  Either way the thread that finishes
  // group cg (rl == 0) is thread cg % CU_THREADS, which also normalises it below.
  for (int cgb = 0; cgb < G; cgb += (RL > 1 ? G : CU_THREADS)) {
    const int cg = RL > 1 ? t % G : cgb + t;
    const int rl = RL > 1 ? t / G : 0;
    const bool act = RL > 1 ? t < RL * G : cg < G;
#pragma unroll
    for (int c = 0; c < KM_MAXK; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (act) {
      const float* dn = a.dn + (size_t)s * a.Wmax * d + c0 + cg * 4;
      constexpr int DEPTH = 8;  // row loads in flight per thread
      for (int j0 = rl; j0 < nw; j0 += DEPTH * RL) {
        float4 v[DEPTH];
#pragma unroll
        for (int u = 0; u < DEPTH; ++u) {
          const int j = j0 + u * RL;
          v[u] = (j < nw && sl[j]) ? *(const float4*)(dn + (size_t)j * d) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < DEPTH; ++u) {
          const int j = j0 + u * RL;
          if (j >= nw || !sl[j]) continue;
          const int lab = lb[j];
#pragma unroll
          for (int c = 0; c < KM_MAXK; ++c)
            if (c == lab) {
              acc[c].x += v[u].x;
              acc[c].y += v[u].y;
              acc[c].z += v[u].z;
              acc[c].w += v[u].w;
            }
        }
      }
    }
    // combine the row lanes in order through shared memory
    if (RL > 1) {
      __syncthreads();
      if (act) {
#pragma unroll
        for (int c = 0; c < KM_MAXK; ++c) part[rl * G + cg][c] = acc[c];
      }
      __syncthreads();
      if (act && rl == 0) {
#pragma unroll
        for (int c = 0; c < KM_MAXK; ++c) acc[c] = part[cg][c];
        for (int q = 1; q < RL; ++q) {
#pragma unroll
          for (int c = 0; c < KM_MAXK; ++c) {
            const float4 w = part[q * G + cg][c];
            acc[c].x += w.x;
            acc[c].y += w.y;
            acc[c].z += w.z;
            acc[c].w += w.w;
          }
        }
      }
    }
    if (act && rl == 0) {
#pragma unroll
      for (int c = 0; c < KM_MAXK; ++c) {
        if (c >= K) continue;
        float* cs = cs_base + (size_t)c * d + c0 + cg * 4;
        float4 v = *(const float4*)cs;
        v.x += acc[c].x;
        v.y += acc[c].y;
        v.z += acc[c].z;
        v.w += acc[c].w;
        *(float4*)cs = v;
        acc[c] = v;
        ssl[c] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
    }
  }
  // |s_c|^2 of this CTA's channels, then over the cluster (rank order)
  const int lane = t & 31, wid = t >> 5;
#pragma unroll
  for (int c = 0; c < KM_MAXK; ++c) {
    float v = ssl[c];
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) wsum[wid][c] = v;
  }
  __syncthreads();
  if (t < KM_MAXK) {
    float v = 0.f;
    for (int w = 0; w < CU_THREADS / 32; ++w) v += wsum[w][t];
    nrm_part[0][t] = v;
  }
  km_allreduce(&nrm_part[0][0], &nrm_full[0][0], KM_MAXK, nc);
  // z_c = s_c / |s_c| for this CTA's channels, and the proxy rows' projection
  // input RMSNorm(z_c) * gain.  z_c is a unit vector, so its mean square over
  // the d channels is 1/d: no second reduction over the cluster.
  const float inv = 1.f / sqrtf(1.f / (float)d + a.eps);
  for (int cg = t; cg < G; cg += CU_THREADS) {
    const float4 gv = one_pass ? gv0 : cl_ld4t<T>(gain + c0 + cg * 4);
#pragma unroll
    for (int c = 0; c < KM_MAXK; ++c) {
      if (c >= K) continue;
      const float nrm = sqrtf(nrm_full[0][c]);
      const float4 v = one_pass ? acc[c] : *(const float4*)(cs_base + (size_t)c * d + c0 + cg * 4);
      const float4 zv = make_float4(v.x / nrm, v.y / nrm, v.z / nrm, v.w / nrm);
      *(float4*)(a.z + ((size_t)s * K + c) * d + c0 + cg * 4) = zv;
      T* ao = (T*)a.a_out + (size_t)(a.proxy_row[s] + c) * d + c0 + cg * 4;
      cl_st4t<T>(ao, make_float4(zv.x * inv * gv.x, zv.y * inv * gv.y, zv.z * inv * gv.z, zv.w * inv * gv.w));
    }
  }
}

// Cluster size of the centroid update: the fewest CTAs (at most 8, a portable
// cluster) that give each CTA at most 512 channels in whole 4-channel groups,
// else the most CTAs up to 8 with whole groups.  At two CTAs per SM every
// sequence of a batch of 32 then has its cluster resident at once on GB300
// (16-CTA clusters at one CTA per SM ran the batch in four waves).
int centroid_cluster_size(int d) {
  for (int nc = 1; nc <= 8; ++nc)
    if (d % (4 * nc) == 0 && d / nc <= 512) return nc;
  for (int nc = 8; nc >= 1; --nc)
    if (d % (4 * nc) == 0) return nc;
  return 1;
}

template <typename T>
void launch_window_patch(const PatchArgs& a, cudaStream_t st) {
  launch_pdl(window_patch_kernel<T>, dim3(a.nw, a.n_fire), dim3(256), 0, st, a);
}
template <typename T>
void launch_centroid_update(const PatchArgs& a, cudaStream_t st) {
  const int nc = centroid_cluster_size(a.d);
  const int cw = a.d / nc;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(nc, a.n_fire);
  cfg.blockDim = dim3(CU_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = nc;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  cudaLaunchKernelEx(&cfg, centroid_update_kernel<T>, a, nc, cw);
}
template void launch_window_patch<float>(const PatchArgs&, cudaStream_t);
template void launch_window_patch<__nv_bfloat16>(const PatchArgs&, cudaStream_t);
template void launch_centroid_update<float>(const PatchArgs&, cudaStream_t);
template void launch_centroid_update<__nv_bfloat16>(const PatchArgs&, cudaStream_t);

}  // namespace polestar
