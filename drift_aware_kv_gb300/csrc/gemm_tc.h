// tcgen05 (5th-generation tensor core) GEMM for bf16 operands, fp32 output.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <array>
#include <map>
#include <unordered_map>

namespace polestar {

struct TcMapKey {
  const void* ptr;
  int rows, cols, ld, box_rows;
  bool operator==(const TcMapKey& o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && ld == o.ld && box_rows == o.box_rows;
  }
};
struct TcMapKeyHash {
  size_t operator()(const TcMapKey& k) const {
    size_t h = (size_t)k.ptr;
    h ^= (size_t)k.rows * 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
    h ^= (size_t)k.cols * 0xC2B2AE3D27D4EB4Full + (h << 6) + (h >> 2);
    h ^= (size_t)k.ld * 0x165667B19E3779F9ull + (h << 6) + (h >> 2);
    h ^= (size_t)k.box_rows + (h << 6) + (h >> 2);
    return h;
  }
};

// Per-context state of the tensor-core GEMM: encoded TMA descriptors (keyed by
// buffer, shape and box), the device error word of the bounded waits, SM count.
struct TcGemmCache {
  std::unordered_map<TcMapKey, CUtensorMap, TcMapKeyHash> maps;
  int* err = nullptr;
  int num_sms = 0;
  // automatic launch choices by shape {M, K, segments, N0, N1, N2, SMs} ->
  // {kernel, bn, splits, stages}: the search runs once per shape
  std::map<std::array<int, 7>, std::array<int, 4>> picks;
  // pair kernel's split tail (single plain segment): partial tiles and their
  // counters, allocated on first use; launches through one cache run one at a
  // time (stream order)
  float* tail_ws = nullptr;
  int* tail_cnt = nullptr;
};

// Kernel choice for tuning sweeps and tests; zero fields are chosen
// automatically.  kernel: 1 row-tiled (rows on the MMA's M side, up to two
// 128-row sub-tiles per CTA), 2 weight-stationary (W rows on the M side, at most
// 256 activation rows on the N side, one tile per CTA), 5 persistent pair tiles
// (two-CTA clusters over 256-row x bn tiles, the pair's MMA run as one,
// cta_group::2).  stages: ring depth; splits: K split over a thread-block
// cluster (1..8), or for kernel 5 the 64-column k-blocks per stage; bn: columns
// per tile of kernels 1 and 5 (a multiple of 16, at most 256).
struct TcGemmChoice {
  int kernel = 0;
  int stages = 0;
  int splits = 0;
  int bn = 0;
  int kpack = 0;  // row-tiled kernel: 64-column k-blocks per stage (0 = 1)
};

// True when the tensor-core path handles this shape: leading dimensions must
// give 16-byte aligned rows (multiples of 8 bf16 elements).
bool tc_gemm_supported(int K, int lda, int ldw);

// C[M, N] (fp32, ldc) = A[M, K] (bf16, lda) * W[N, K]^T (bf16, ldw); rows at or
// beyond min(M, *m_dev) are not written (m_dev may be null).
cudaError_t tc_gemm_bf16(TcGemmCache* cache, const void* A, int lda, const void* W, int ldw, float* C, int ldc,
                         int M, const int* m_dev, int N, int K, cudaStream_t st,
                         const TcGemmChoice* force = nullptr);

// Up to three projections sharing the A operand in one launch: segment s
// computes C[s][M, N[s]] = A * W[s]^T (all C[s] with row stride ldc).
cudaError_t tc_gemm_bf16_multi(TcGemmCache* cache, const void* A, int lda, int nseg, const void* const* W,
                               const int* ldw, const int* N, float* const* C, int ldc, int M, const int* m_dev,
                               int K, cudaStream_t st, const TcGemmChoice* force = nullptr);

// Q/K/V projection of one layer with the rotary embedding and the scatter
// fused into the two-SM pair kernel's epilogue: segments W[0] (Q, N[0] rows),
// W[1] (K) and W[2] (V) (row stride K); row r of A is the row rows[r]
// {seq, pos, kind, aux}; its Q (rotated unless a proxy row) goes to
// q_out[r, N[0]] bf16, its K (rotated) and V to the cache row (seq, pos) of
// kv_layer (bf16 [.., N, 2, kvdim], seq stride kv_seq_stride elements) when
// the row is active, other, or a window row with write_kv[r] set (every
// window row when write_kv is null).  cudaErrorNotSupported when the
// library's choice for the shape is not the pair kernel or the widths are not
// whole 256-column tiles of whole heads (the caller then runs the projection
// and the row kernel).
struct TcQkvRope {
  const int4* rows = nullptr;
  const uint8_t* write_kv = nullptr;
  const float2* rope = nullptr;  // [N][dh / 2] (cos, sin)
  void* q_out = nullptr;
  void* kv_layer = nullptr;
  size_t kv_seq_stride = 0;
  int kvdim = 0, dh = 0;
};
cudaError_t tc_gemm_bf16_qkv_rope(TcGemmCache* cache, const void* A, int lda, const void* const* W, const int* N,
                                  int M, int K, const TcQkvRope& q, cudaStream_t st);

// Gate and up projections with the SwiGLU activation fused into the
// row-tiled kernel's epilogue: act[m, f] = bf16(silu(g) * u) with
// g = A * Wg^T, u = A * Wu^T (both [F, K], row stride ldw), act row stride
// ld_act.  cudaErrorNotSupported when the library's choice for this shape is
// not the row-tiled kernel (the caller then runs the projections and the
// activation separately); force (kernel 1 only) overrides width/split/depth.
cudaError_t tc_gemm_bf16_swiglu(TcGemmCache* cache, const void* A, int lda, const void* Wg, const void* Wu, int ldw,
                                int F, void* act, int ld_act, int M, const int* m_dev, int K, cudaStream_t st,
                                const TcGemmChoice* force = nullptr);

// The launch the library picks for M rows, nseg weight segments of N[i]
// output columns and inner size K: out = {kernel (1 row-tiled, 2
// weight-stationary, 5 two-SM pair tiles), columns per tile, K split, ring
// depth}.
cudaError_t tc_gemm_choice(TcGemmCache* cache, int M, int nseg, const int* N, int K, int* out);

// Device word holding the code of the first timed-out wait (0 = none).
int* tc_error_word(TcGemmCache* cache);

// Test of the bounded waits: on `st`, shortens the wait bound of this file's
// kernels to limit_cycles, runs one kernel whose mbarrier wait can never be
// satisfied (it gives up after the bound and writes `code` to *err), then
// restores the default bound.  The bound is a per-device variable shared by
// every stream: other work in flight meanwhile sees the short bound too.
cudaError_t tc_debug_stalled_wait(int* err, int code, long long limit_cycles, cudaStream_t st);

void tc_gemm_cache_clear(TcGemmCache* cache);
// After a reported wait timeout: clear the split-tail counters, which a launch
// that gave up may have left counted (stream-ordered on st).
cudaError_t tc_gemm_reset_after_timeout(TcGemmCache* cache, cudaStream_t st);

}  // namespace polestar
