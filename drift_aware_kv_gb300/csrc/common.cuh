// Shared device helpers of the Polestar library (storage-type loads/stores,
// warp/block reductions, the NVFP4 number formats).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace polestar {

// ---- kernel attributes, once per device -------------------------------------------
// A kernel attribute (dynamic shared memory limit, non-portable cluster size)
// applies to the device that is current when it is set, so each launch site
// keeps one flag per device and sets the attribute the first time it launches
// on that device.
struct PerDeviceOnce {
  static constexpr int kDevices = 64;
  std::atomic<bool> done[kDevices] = {};
};
inline cudaError_t func_attr_once(PerDeviceOnce& once, const void* func, cudaFuncAttribute attr, int value) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= PerDeviceOnce::kDevices) return cudaFuncSetAttribute(func, attr, value);
  if (once.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, attr, value);
  if (e == cudaSuccess) once.done[dev].store(true, std::memory_order_release);
  return e;
}

// ---- storage types: fp32 or bf16, arithmetic always fp32 ---------------------
template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// ---- reductions ----------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Sum over the block; `red` holds >= 32 floats of shared memory.  All threads
// get the result.  Deterministic (fixed tree).
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = (threadIdx.x < nw) ? red[threadIdx.x] : 0.f;
  if (wid == 0) t = warp_sum(t);
  if (threadIdx.x == 0) red[0] = t;
  __syncthreads();
  return red[0];
}

// ---- NVFP4 formats (App. C.3: E2M1 elements, E4M3 scale per 16 elements) -------
// E4M3 (bias 7, max finite 448, subnormal quantum 2^-9), round to nearest even,
// saturating.  Input is a non-negative fp32 value.
__device__ __forceinline__ uint8_t e4m3_encode_rne(float v) {
  if (!(v > 0.f)) return 0;
  if (v >= 448.f) return 0x7E;
  int e2;
  frexpf(v, &e2);        // v = f * 2^e2, f in [0.5, 1)  => floor(log2 v) = e2 - 1
  int E = e2 - 1;
  if (E < -6) E = -6;    // subnormal range shares the quantum of the first binade
  const float q = ldexpf(v, 3 - E);  // v / 2^(E-3), exact
  const float n = rintf(q);          // nearest, ties to even
  // n in [0, 16]; n == 16 carries into the next binade
  int exp_field, mant;
  if (n == 0.f) return 0;
  if (E == -6 && n < 8.f) {  // subnormal: value n * 2^-9
    exp_field = 0;
    mant = (int)n;
  } else if (n >= 16.f) {
    exp_field = E + 1 + 7;
    mant = 0;
  } else {
    exp_field = E + 7;
    mant = (int)n - 8;
  }
  if (exp_field > 15 || (exp_field == 15 && mant > 6)) return 0x7E;
  return (uint8_t)((exp_field << 3) | mant);
}

__device__ __forceinline__ float e4m3_decode(uint8_t b) {
  const int e = (b >> 3) & 0xF, m = b & 7;
  const float mag = (e == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
  return (b & 0x80) ? -mag : mag;
}

// E2M1 code of an fp32 value: bit 3 = sign, bits 0-2 index into
// {0, .5, 1, 1.5, 2, 3, 4, 6}; nearest with ties to the even index; saturating.
__device__ __forceinline__ uint32_t e2m1_encode_rne(float x) {
  const float a = fabsf(x);
  uint32_t idx = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                 (a >= 3.5f) + (a > 5.f);
  return ((__float_as_uint(x) >> 31) << 3) | idx;
}

__device__ __forceinline__ float e2m1_decode(uint32_t c) {
  // magnitude table as bit patterns of {0, .5, 1, 1.5, 2, 3, 4, 6}
  const uint32_t i = c & 7u;
  const float mag = (i < 4) ? 0.5f * (float)i : (float)(1u << ((i - 2) >> 1)) * (1.f + 0.5f * (float)(i & 1u));
  return (c & 8u) ? -mag : mag;
}

// Encode one group of 16 residual values.  Returns the scale byte, writes 8
// packed bytes (element 2i in the low nibble).
__device__ __forceinline__ uint8_t nvfp4_encode16(const float* r, uint8_t* out8) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(r[i]));
  const uint8_t sb = e4m3_encode_rne(__fdiv_rn(amax, 6.f));
  const float s = e4m3_decode(sb);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t lo = 0, hi = 0;
    if (s > 0.f) {
      lo = e2m1_encode_rne(__fdiv_rn(r[2 * i], s));
      hi = e2m1_encode_rne(__fdiv_rn(r[2 * i + 1], s));
    }
    out8[i] = (uint8_t)(lo | (hi << 4));
  }
  return sb;
}

// ---- programmatic dependent launch ------------------------------------------
// Every kernel of the layer loop is launched with programmatic stream
// serialisation: it lets its successor start launching right away and waits
// for its predecessor's results before touching memory the predecessor writes.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_launch_dependents();
  pdl_wait();
}

// ---- row metadata -------------------------------------------------------------
enum RowKind : int { ROW_NONE = 0, ROW_ACTIVE = 1, ROW_WINDOW = 2, ROW_PROXY = 3, ROW_OTHER = 4 };

// log sum_j q_j e^(d_j) of the KL drift (Eq. 4 with q = the previous softmax and
// d = new minus previous score), from x = sum_j q_j expm1(d_j) / sum_j q_j:
// log1p(x) while x > -1/2.  Below that the sum is the ratio e^(lse_new - lse_prev)
// near zero, and 1 + x would cancel the digits that matter, so the difference
// of the two log-sum-exps (natural units) is taken instead.
__device__ __forceinline__ float kl_log_mass(float x, float lse_new, float lse_prev) {
  return x > -0.5f ? log1pf(x) : lse_new - lse_prev;
}

// Rotate-half rotary embedding of one pair (x_k, x_{k+dh/2}) by (cos, sin):
// explicit fused multiply-adds, so every kernel that applies it (the row
// kernel and the projection epilogue) rounds identically.
__device__ __forceinline__ void rope_rotate(float a, float b, float c, float s, float& y1, float& y2) {
  y1 = fmaf(a, c, -(b * s));
  y2 = fmaf(b, c, a * s);
}

}  // namespace polestar
