// KV-cache staleness (Polestar, App. C.2 "KV-Cache Staleness Metric").
//
// For a cached K/V row i and the fully recomputed row of the same position,
//   E_i = 1 - (mean_h cos(K_i^h, Kref_i^h) + mean_h cos(V_i^h, Vref_i^h)) / 2,
// the cosine taken per KV head and averaged over heads.  Rows are laid out as
// the library's cache: [rows][2][Hkv * dh], K first, then V.
//
// Memory-bound: every element of both caches is read once (4 * Hkv * dh
// elements per row).  One CTA of 8 warps per row; a warp takes one head at a
// time, lanes 0-15 its K vectors and lanes 16-31 its V vectors, each lane 8
// consecutive elements (one 16-byte load per cache for bf16, two for fp32)
// per 128-element stride.  Sums are fp32; the half-warp reduction and the sum
// over heads run in a fixed order, so results are deterministic.
#include "kernels.h"

namespace polestar {
namespace {

constexpr int kStaleWarps = 8;

template <typename T>
struct Vec8;
template <>
struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* out) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load(const float* p, float* out) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
  }
};

// cos(a, b) from <a,b>, |a|^2, |b|^2.  Zero vectors: two zero vectors count as
// identical (cos 1), one zero vector as orthogonal (cos 0).
__device__ __forceinline__ float cosine(float dot, float na, float nb) {
  if (na > 0.f && nb > 0.f) return dot / (sqrtf(na) * sqrtf(nb));
  return (na == 0.f && nb == 0.f) ? 1.f : 0.f;
}

template <typename T>
__global__ void __launch_bounds__(kStaleWarps * 32)
    kv_staleness_kernel(const T* __restrict__ kv, const T* __restrict__ ref, int Hkv, int dh,
                        float* __restrict__ E) {
  __shared__ float part[kStaleWarps][2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane >> 4, l16 = lane & 15;
  const size_t kvdim = (size_t)Hkv * dh;
  const size_t base = (size_t)blockIdx.x * 2 * kvdim + (size_t)half * kvdim;
  float acc = 0.f;  // lane 0: sum of K cosines of this warp's heads; lane 16: V
  for (int h = warp; h < Hkv; h += kStaleWarps) {
    float dot = 0.f, na = 0.f, nb = 0.f;
    for (int e = l16 * 8; e < dh; e += 128) {
      float a[8], b[8];
      Vec8<T>::load(kv + base + (size_t)h * dh + e, a);
      Vec8<T>::load(ref + base + (size_t)h * dh + e, b);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dot = fmaf(a[i], b[i], dot);
        na = fmaf(a[i], a[i], na);
        nb = fmaf(b[i], b[i], nb);
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {  // stays inside the 16-lane half
      dot += __shfl_xor_sync(0xffffffffu, dot, o);
      na += __shfl_xor_sync(0xffffffffu, na, o);
      nb += __shfl_xor_sync(0xffffffffu, nb, o);
    }
    acc += cosine(dot, na, nb);
  }
  if (l16 == 0) part[warp][half] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float sk = 0.f, sv = 0.f;
    for (int w = 0; w < kStaleWarps; ++w) {
      sk += part[w][0];
      sv += part[w][1];
    }
    E[blockIdx.x] = 1.f - 0.5f * (sk / (float)Hkv + sv / (float)Hkv);
  }
}

}  // namespace

template <typename T>
cudaError_t launch_kv_staleness(const void* kv, const void* ref, long long rows, int Hkv, int dh, float* E,
                                cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  kv_staleness_kernel<T><<<(unsigned)rows, kStaleWarps * 32, 0, st>>>((const T*)kv, (const T*)ref, Hkv, dh, E);
  return cudaGetLastError();
}

template cudaError_t launch_kv_staleness<float>(const void*, const void*, long long, int, int, float*,
                                                cudaStream_t);
template cudaError_t launch_kv_staleness<__nv_bfloat16>(const void*, const void*, long long, int, int, float*,
                                                        cudaStream_t);

}  // namespace polestar
