// tcgen05 (5th-generation tensor core) GEMM for bf16 operands, fp32 output.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace polestar {

struct TcGemmCache {
  struct Entry {
    const void* ptr;
    int rows, cols, ld, box_rows;
    alignas(64) unsigned char map[128];
  };
  std::vector<Entry> maps;
};

// True when the tensor-core path handles this shape (K and leading dimensions
// multiples of 64 elements / 16 bytes).
bool tc_gemm_supported(int K, int lda, int ldw);

// C[M, N] (fp32, ldc) = A[M, K] (bf16, lda) * W[N, K]^T (bf16, ldw); rows at or
// beyond min(M, *m_dev) are neither read meaningfully nor written.
cudaError_t tc_gemm_bf16(TcGemmCache* cache, const void* A, int lda, const void* W, int ldw, float* C, int ldc,
                         int M, const int* m_dev, int N, int K, cudaStream_t st);

void tc_gemm_cache_clear(TcGemmCache* cache);

}  // namespace polestar
