// CUDA-core GEMM C[M, N] = A[M, K] * W[N, K]^T with fp32 accumulation.
// Used for fp32 workloads (no fp32 tensor-core path keeps full fp32 products)
// and as the cross-check of the tensor-core kernel in tests.
#include "kernels.h"

namespace polestar {

constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16;

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T* __restrict__ A, int lda, const T* __restrict__ W,
                                                         int ldw, float* __restrict__ C, int ldc, int M,
                                                         const int* __restrict__ m_dev, int N, int K) {
  pdl_enter();
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Ws[SG_BK][SG_BN + 4];
  const int Mr = m_dev ? min(M, *m_dev) : M;
  const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
  if (m0 >= Mr) return;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += SG_BK) {
    for (int idx = threadIdx.x; idx < SG_BM * SG_BK; idx += 256) {
      const int mm = idx / SG_BK, kk = idx % SG_BK;
      const int gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < Mr && gk < K) ? to_f<T>(A[(size_t)gm * lda + gk]) : 0.f;
      const int gn = n0 + mm;
      Ws[kk][mm] = (gn < N && gk < K) ? to_f<T>(W[(size_t)gn * ldw + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i) b[i] = Ws[kk][tx * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(a[i], b[jj], acc[i][jj]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= Mr) continue;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int gn = n0 + tx * 4 + jj;
      if (gn < N) C[(size_t)gm * ldc + gn] = acc[i][jj];
    }
  }
}

template <typename T>
void launch_gemm_simt(const void* A, int lda, const void* W, int ldw, float* C, int ldc, int M, const int* m_dev,
                      int N, int K, cudaStream_t st) {
  const dim3 grid((N + SG_BN - 1) / SG_BN, (M + SG_BM - 1) / SG_BM);
  launch_pdl(gemm_simt_kernel<T>, dim3(grid), dim3(256), 0, st, (const T*)A, lda, (const T*)W, ldw, C, ldc, M, m_dev, N, K);
}

template void launch_gemm_simt<float>(const void*, int, const void*, int, float*, int, int, const int*, int, int,
                                      cudaStream_t);
template void launch_gemm_simt<__nv_bfloat16>(const void*, int, const void*, int, float*, int, int, const int*,
                                              int, int, cudaStream_t);

}  // namespace polestar
