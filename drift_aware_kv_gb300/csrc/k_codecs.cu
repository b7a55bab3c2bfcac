// Storage formats of the window hidden states compared in the quantization
// ablation of "Polestar: Drift-Aware Cache Calibration and Token Commitment for
// Efficient Inference of Diffusion LLMs" (Table 11; NVFP4 as in App. C.3).
//
// A format stores either the hidden state h itself ("plain") or its residual
// r = h - A_label against the row's cluster anchor ("residual", App. C.3 /
// §4.1), and decoding adds the anchor back.  The paper names the formats but
// fixes only NVFP4's layout; the others follow their usual definitions:
//   FP16   binary16 of every element, nearest even;
//   FP8    E4M3 elements (nearest even, saturating at 448), one fp32 scale per
//          row s = fp32(amax / 448);
//   INT8   integers in [-127, 127] (nearest even), one fp32 scale per row
//          s = fp32(amax / 127);
//   MXFP4  OCP microscaling: blocks of 32 elements share a power-of-two scale
//          2^e, e = floor(log2 amax) - 2 (E8M0 byte e + 127, e clamped to
//          [-127, 127]), E2M1 elements nearest even, saturating at 6;
//   INT2   ternary {-1, 0, +1} with one fp32 scale per row s = amax: an element
//          is +-s when |r| > s / 2, else 0 (a tie goes to the even value 0);
//   NVFP4  E2M1 elements with one E4M3 scale per 16 (App. C.3).
// Every division is IEEE fp32 round-to-nearest, every rounding to a grid
// nearest-even, as the definitions state; all-zero rows or blocks store zero
// codes and a zero scale.
//
// One 256-thread CTA per row; a thread owns 16 consecutive elements (one NVFP4
// group, half an MXFP4 block) per pass, loaded with 16-byte vector loads; the
// per-row maxima are block reductions.  Memory-bound: a row is read once and its
// codes written once.
#include <cuda_fp16.h>

#include "../../include/polestar.h"
#include "kernels.h"

namespace polestar {
namespace {

constexpr int CT = 256;  // threads per row

struct CodecArgs {
  int fmt, rows, d;
  const float* h;        // [rows, d] encode input / decode output
  float* out;
  const float* anchors;  // [K, d] or null (plain)
  const uint8_t* labels; // [rows]
  uint8_t* codes;        // layout per format (see polestar.h)
  uint8_t* scales;
};

__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = (threadIdx.x < CT / 32) ? red[threadIdx.x] : 0.f;
  if (wid == 0) t = warp_max(t);
  if (threadIdx.x == 0) red[0] = t;
  __syncthreads();
  return red[0];
}

// E4M3 of a signed fp32 value: sign bit 7, magnitude nearest even, saturating
__device__ __forceinline__ uint8_t e4m3_signed(float q) {
  return (uint8_t)(e4m3_encode_rne(fabsf(q)) | ((__float_as_uint(q) >> 31) << 7));
}

// the 16 values of chunk c of row `row` (residual against the anchor when given)
__device__ __forceinline__ void load16(const CodecArgs& a, int row, int c, float* v) {
  const float4* src = (const float4*)(a.h + (size_t)row * a.d + c * 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 x = src[i];
    v[4 * i] = x.x;
    v[4 * i + 1] = x.y;
    v[4 * i + 2] = x.z;
    v[4 * i + 3] = x.w;
  }
  if (a.anchors) {
    const float4* an = (const float4*)(a.anchors + (size_t)a.labels[row] * a.d + c * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 x = an[i];
      v[4 * i] -= x.x;
      v[4 * i + 1] -= x.y;
      v[4 * i + 2] -= x.z;
      v[4 * i + 3] -= x.w;
    }
  }
}

__global__ void __launch_bounds__(CT) codec_encode_kernel(CodecArgs a) {
  __shared__ float red[CT / 32];
  const int row = blockIdx.x, d = a.d, nch = d / 16;
  const int fmt = a.fmt;
  // per-row scale formats: the row maximum first
  float s = 0.f;
  if (fmt == POLESTAR_CODEC_FP8 || fmt == POLESTAR_CODEC_INT8 || fmt == POLESTAR_CODEC_INT2) {
    float m = 0.f;
    for (int c = threadIdx.x; c < nch; c += CT) {
      float v[16];
      load16(a, row, c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
    }
    const float amax = block_max(m, red);
    s = fmt == POLESTAR_CODEC_FP8 ? __fdiv_rn(amax, 448.f) : (fmt == POLESTAR_CODEC_INT8 ? __fdiv_rn(amax, 127.f) : amax);
    if (threadIdx.x == 0) ((float*)a.scales)[row] = s;
  }
  // MXFP4 pairs chunks 2k, 2k + 1 into one block: both sit in one warp when
  // the chunk stride is a multiple of 2, so every pass keeps the pairing
  for (int c0 = 0; c0 < nch; c0 += CT) {
    const int c = c0 + threadIdx.x;
    const bool live = c < nch;
    float v[16];
    if (live) load16(a, row, c, v);
    else
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.f;
    if (fmt == POLESTAR_CODEC_FP16) {
      if (live) {
        uint16_t* dst = (uint16_t*)a.codes + (size_t)row * d + c * 16;
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i] = (uint32_t)__half_as_ushort(__float2half_rn(v[2 * i])) |
                 ((uint32_t)__half_as_ushort(__float2half_rn(v[2 * i + 1])) << 16);
        ((uint4*)dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        ((uint4*)dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    } else if (fmt == POLESTAR_CODEC_FP8 || fmt == POLESTAR_CODEC_INT8) {
      if (live) {
        uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t b = 0;
          if (s > 0.f) {
            const float q = __fdiv_rn(v[i], s);
            if (fmt == POLESTAR_CODEC_FP8) {
              b = e4m3_signed(q);
            } else {
              const float n = fminf(fmaxf(rintf(q), -127.f), 127.f);
              b = (uint32_t)(uint8_t)(int8_t)(int)n;
            }
          }
          w[i >> 2] |= b << (8 * (i & 3));
        }
        *(uint4*)(a.codes + (size_t)row * d + c * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else if (fmt == POLESTAR_CODEC_INT2) {
      if (live) {
        uint32_t w = 0;
        const float half = 0.5f * s;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t t = 0;  // 2-bit two's complement: 0 -> 00, +1 -> 01, -1 -> 11
          if (s > 0.f && fabsf(v[i]) > half) t = v[i] > 0.f ? 1u : 3u;
          w |= t << (2 * i);
        }
        *(uint32_t*)(a.codes + (size_t)row * (d / 4) + c * 4) = w;
      }
    } else if (fmt == POLESTAR_CODEC_NVFP4) {
      if (live) {
        uint8_t packed[8];
        const uint8_t sb = nvfp4_encode16(v, packed);
        uint2 w;
        memcpy(&w, packed, 8);
        *(uint2*)(a.codes + (size_t)row * (d / 2) + c * 8) = w;
        a.scales[(size_t)row * (d / 16) + c] = sb;
      }
    } else {  // MXFP4
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));  // the block's other half
      int e = 0;
      if (m > 0.f) {
        int e2;
        frexpf(m, &e2);  // m = f 2^e2, f in [0.5, 1): floor(log2 m) = e2 - 1
        e = min(max(e2 - 1 - 2, -127), 127);
      }
      if (live) {
        uint32_t w[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t code = m > 0.f ? e2m1_encode_rne(ldexpf(v[i], -e)) : 0u;
          w[i >> 3] |= code << (4 * (i & 7));
        }
        *(uint2*)(a.codes + (size_t)row * (d / 2) + c * 8) = make_uint2(w[0], w[1]);
        if ((c & 1) == 0) a.scales[(size_t)row * (d / 32) + (c >> 1)] = (uint8_t)(e + 127);
      }
    }
  }
}

__global__ void __launch_bounds__(CT) codec_decode_kernel(CodecArgs a) {
  const int row = blockIdx.x, d = a.d, nch = d / 16;
  const int fmt = a.fmt;
  float s = 0.f;
  if (fmt == POLESTAR_CODEC_FP8 || fmt == POLESTAR_CODEC_INT8 || fmt == POLESTAR_CODEC_INT2)
    s = ((const float*)a.scales)[row];
  for (int c = threadIdx.x; c < nch; c += CT) {
    float v[16];
    if (fmt == POLESTAR_CODEC_FP16) {
      const uint4* src = (const uint4*)((const uint16_t*)a.codes + (size_t)row * d + c * 16);
      const uint4 p0 = src[0], p1 = src[1];
      const uint32_t w[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xFFFF)));
        v[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
      }
    } else if (fmt == POLESTAR_CODEC_FP8 || fmt == POLESTAR_CODEC_INT8) {
      const uint4 p = *(const uint4*)(a.codes + (size_t)row * d + c * 16);
      const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint8_t b = (uint8_t)(w[i >> 2] >> (8 * (i & 3)));
        v[i] = fmt == POLESTAR_CODEC_FP8 ? e4m3_decode(b) * s : (float)(int8_t)b * s;
      }
    } else if (fmt == POLESTAR_CODEC_INT2) {
      const uint32_t w = *(const uint32_t*)(a.codes + (size_t)row * (d / 4) + c * 4);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t t = (w >> (2 * i)) & 3u;
        v[i] = t == 1u ? s : (t == 3u ? -s : 0.f);
      }
    } else {  // NVFP4, MXFP4: packed E2M1 pairs, element 2i in the low nibble
      const uint2 p = *(const uint2*)(a.codes + (size_t)row * (d / 2) + c * 8);
      float sc;
      if (fmt == POLESTAR_CODEC_NVFP4)
        sc = e4m3_decode(a.scales[(size_t)row * (d / 16) + c]);
      else
        sc = ldexpf(1.f, (int)a.scales[(size_t)row * (d / 32) + (c >> 1)] - 127);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = e2m1_decode(((i < 8 ? p.x : p.y) >> (4 * (i & 7))) & 0xFu) * sc;
    }
    if (a.anchors) {
      const float* an = a.anchors + (size_t)a.labels[row] * d + c * 16;
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] += an[i];
    }
    float4* dst = (float4*)(a.out + (size_t)row * d + c * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

bool codec_shape_ok(int fmt, int rows, int d) {
  return fmt >= POLESTAR_CODEC_FP16 && fmt <= POLESTAR_CODEC_NVFP4 && rows >= 0 && d >= 32 && d % 32 == 0;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

int64_t codec_code_bytes(int fmt, int64_t rows, int64_t d) {
  switch (fmt) {
    case POLESTAR_CODEC_FP16: return rows * d * 2;
    case POLESTAR_CODEC_FP8:
    case POLESTAR_CODEC_INT8: return rows * d;
    case POLESTAR_CODEC_MXFP4:
    case POLESTAR_CODEC_NVFP4: return rows * d / 2;
    case POLESTAR_CODEC_INT2: return rows * d / 4;
  }
  return -1;
}

int64_t codec_scale_bytes(int fmt, int64_t rows, int64_t d) {
  switch (fmt) {
    case POLESTAR_CODEC_FP16: return 0;
    case POLESTAR_CODEC_FP8:
    case POLESTAR_CODEC_INT8:
    case POLESTAR_CODEC_INT2: return rows * 4;
    case POLESTAR_CODEC_MXFP4: return rows * d / 32;
    case POLESTAR_CODEC_NVFP4: return rows * d / 16;
  }
  return -1;
}

}  // namespace polestar

using namespace polestar;

extern "C" int64_t polestar_codec_bytes(int32_t fmt, int32_t rows, int32_t d, int64_t* code_bytes,
                                        int64_t* scale_bytes) {
  if (!codec_shape_ok(fmt, rows, d)) return -1;
  const int64_t c = codec_code_bytes(fmt, rows, d), s = codec_scale_bytes(fmt, rows, d);
  if (code_bytes) *code_bytes = c;
  if (scale_bytes) *scale_bytes = s;
  return c + s;
}

extern "C" polestar_status polestar_codec_encode(int32_t fmt, const float* h, int32_t rows, int32_t d,
                                                 const float* anchors, const uint8_t* labels, void* codes,
                                                 void* scales, void* stream) {
  if (!codec_shape_ok(fmt, rows, d)) return POLESTAR_ERR_INVALID_ARG;
  if (rows == 0) return POLESTAR_OK;
  if (!h || !codes || (anchors && !labels) || (fmt != POLESTAR_CODEC_FP16 && !scales)) return POLESTAR_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(codes) || (anchors && !aligned16(anchors))) return POLESTAR_ERR_INVALID_ARG;
  CodecArgs a{};
  a.fmt = fmt;
  a.rows = rows;
  a.d = d;
  a.h = h;
  a.anchors = anchors;
  a.labels = labels;
  a.codes = (uint8_t*)codes;
  a.scales = (uint8_t*)scales;
  codec_encode_kernel<<<rows, CT, 0, (cudaStream_t)stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? POLESTAR_OK : POLESTAR_ERR_CUDA;
}

extern "C" polestar_status polestar_codec_decode(int32_t fmt, const void* codes, const void* scales, int32_t rows,
                                                 int32_t d, const float* anchors, const uint8_t* labels, float* out,
                                                 void* stream) {
  if (!codec_shape_ok(fmt, rows, d)) return POLESTAR_ERR_INVALID_ARG;
  if (rows == 0) return POLESTAR_OK;
  if (!out || !codes || (anchors && !labels) || (fmt != POLESTAR_CODEC_FP16 && !scales)) return POLESTAR_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(codes) || (anchors && !aligned16(anchors))) return POLESTAR_ERR_INVALID_ARG;
  CodecArgs a{};
  a.fmt = fmt;
  a.rows = rows;
  a.d = d;
  a.out = out;
  a.anchors = anchors;
  a.labels = labels;
  a.codes = (uint8_t*)codes;
  a.scales = (uint8_t*)scales;
  codec_decode_kernel<<<rows, CT, 0, (cudaStream_t)stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? POLESTAR_OK : POLESTAR_ERR_CUDA;
}
