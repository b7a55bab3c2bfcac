// bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
//   C[M, N] (fp32) = A[M, K] (bf16, K-major) * W[N, K]^T (bf16, K-major)
//
// The projections of the Polestar layer loop are weight-stream bound at small
// batch (tens to a few hundred gathered rows against multi-MB weight matrices),
// so the kernel is organised around reading every weight tile exactly once:
//   * a CTA owns one 128-column slice of W and applies each staged W tile to
//     all of its rows: up to MT = 2 row sub-tiles of 128, each with its own
//     fp32 accumulator in TMEM (MT x 128 columns);
//   * when (N / 128) x row-groups gives too few CTAs to keep HBM busy, K is
//     split over the S CTAs of a thread-block cluster; the partial tiles are
//     reduced through distributed shared memory in a fixed order (no atomics,
//     no global workspace, deterministic);
//   * warp 0 issues TMA loads (128B-swizzled boxes of 64 K-elements) into an
//     mbarrier pipeline, warp 1 issues tcgen05.mma (one elected thread), warps
//     2-5 drain TMEM with tcgen05.ld in the epilogue.
// Every mbarrier wait is bounded by a clock-based timeout that records an
// error code instead of spinning forever.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "gemm_tc.h"

namespace polestar {

namespace tc {

constexpr int BM = 128;         // rows per UMMA
constexpr int BN = 128;         // columns per CTA
constexpr int BK = 64;          // K elements per stage (one 128-byte swizzle row)
constexpr int THREADS = 192;    // 6 warps
// dynamic shared memory of a configuration: stages + barriers + alignment slack
constexpr int smem_bytes(int mt, int stages) { return stages * (mt * 128 * 64 * 2 + 128 * 64 * 2) + 2048; }
constexpr long long TIMEOUT_CYCLES = 4000000000LL;  // ~2 s at 2 GHz
constexpr int RED_PITCH = BN + 4;                     // fp32 staging row pitch

struct Params {
  int M, K;
  const int* m_dev;
  int ldc;
  int ktiles;
  int splits;
  int* err;
  // up to three weight segments sharing A: tiles [seg_start[s], seg_start[s+1])
  int nseg;
  int seg_start[4];
  int seg_N[3];
  float* seg_C[3];
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait; on timeout records `code` in *err and in the CTA abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err, int code,
                                          volatile int* abort_flag) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > TIMEOUT_CYCLES) {
      atomicExch(err, code);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;                      // leading-dimension offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride-dimension offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                      // descriptor version
  d |= (uint64_t)2 << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, bf16 x bf16 -> fp32, both K-major, M = 128, N = BN.
__host__ __device__ constexpr uint32_t instr_desc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(instr_desc()), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float4 ld_dsmem4(const float* local_ptr, uint32_t rank) {
  uint32_t a = smem_u32(local_ptr), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(ra)
               : "memory");
  return v;
}

template <int MT, int STAGES>
__global__ void __launch_bounds__(THREADS)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2, Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  constexpr int A_BYTES = BM * BK * 2;  // 16 KB per row sub-tile
  constexpr int B_BYTES = BN * BK * 2;  // 16 KB
  constexpr int STAGE_BYTES = MT * A_BYTES + B_BYTES;
  uint64_t* full = (uint64_t*)(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* accum = empty + STAGES;
  uint32_t* tmem_slot = (uint32_t*)(accum + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int seg = (tile >= p.seg_start[1]) + (tile >= p.seg_start[2]);
  const int n0 = (tile - p.seg_start[seg]) * BN;
  const int segN = p.seg_N[seg];
  float* const Cseg = p.seg_C[seg];
  const CUtensorMap* tmB = seg == 0 ? &tmB0 : (seg == 1 ? &tmB1 : &tmB2);
  const int m0 = blockIdx.y * (MT * BM);
  const int split = blockIdx.z;

  const int kt0 = (int)((long long)split * p.ktiles / p.splits);
  const int kt1 = (int)((long long)(split + 1) * p.ktiles / p.splits);
  const int nk = kt1 - kt0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(accum), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(MT * BN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  // Weights never depend on earlier kernels: the first stages' W tiles are
  // requested before waiting for the predecessor that produces A (and m_dev).
  const int npre = nk < STAGES ? nk : STAGES;
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < npre; ++i) {
      const uint32_t fb = smem_u32(&full[i]);
      mbar_expect_tx(fb, STAGE_BYTES);
      tma_load_2d(smem_u32(smem + i * STAGE_BYTES) + MT * A_BYTES, tmB, (kt0 + i) * BK, n0, fb);
    }
  }
  pdl_launch_dependents();
  pdl_wait();
  const int M_eff = p.m_dev ? min(p.M, *p.m_dev) : p.M;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      for (int i = 0; i < npre; ++i) {
        const uint32_t st = smem_u32(smem + i * STAGE_BYTES);
        const int kx = (kt0 + i) * BK;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) tma_load_2d(st + mt * A_BYTES, &tmA, kx, m0 + mt * BM, smem_u32(&full[i]));
      }
      for (int i = npre; i < nk; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(smem_u32(&empty[s]), ((i / STAGES) - 1) & 1, p.err, 1, abort_flag)) break;
        const uint32_t fb = smem_u32(&full[s]);
        mbar_expect_tx(fb, STAGE_BYTES);
        const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
        const int kx = (kt0 + i) * BK;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) tma_load_2d(st + mt * A_BYTES, &tmA, kx, m0 + mt * BM, fb);
        tma_load_2d(st + MT * A_BYTES, tmB, kx, n0, fb);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(smem_u32(&full[s]), (i / STAGES) & 1, p.err, 2, abort_flag)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
        const uint32_t bst = st + MT * A_BYTES;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            umma(tmem + mt * BN, smem_desc(st + mt * A_BYTES + kk * 32), smem_desc(bst + kk * 32),
                 (i > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(smem_u32(&empty[s]));  // frees the stage once these MMAs have read it
      }
      umma_commit(smem_u32(accum));        // accumulators final
    }
  }
  __syncwarp();

  // ---------------- epilogue
  const bool epi = warp >= 2;
  const int q = warp & 3;              // TMEM lane quarter this warp may access
  bool ok = true;
  if (epi) {
    ok = (nk > 0) && mbar_wait(smem_u32(accum), 0, p.err, 3, abort_flag);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  }
  if (p.splits == 1) {
    if (epi && ok) {
#pragma unroll 1
      for (int mt = 0; mt < MT; ++mt) {
        const int row = m0 + mt * BM + q * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + mt * BN + c, v);
          if (row < M_eff) {
            float* dst = Cseg + (size_t)row * p.ldc + n0 + c;
            if (n0 + c + 32 <= segN && ((p.ldc & 3) == 0) && ((((uintptr_t)Cseg) & 15) == 0)) {
#pragma unroll
              for (int j = 0; j < 32; j += 4) *(float4*)(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (n0 + c + j < segN) dst[j] = v[j];
            }
          }
        }
      }
    }
  } else {
    // split-K: stage partials in shared memory, reduce across the cluster
    float* red = (float*)smem;  // [BM][RED_PITCH] fp32, pipeline buffers are idle now
    const uint32_t rank = cluster_rank();
#pragma unroll 1
    for (int mt = 0; mt < MT; ++mt) {
      __syncthreads();
      if (epi) {
        const int r = q * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          if (ok) tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + mt * BN + c, v);
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *(float4*)(red + r * RED_PITCH + c + j) =
                ok ? make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      cluster_sync();
      // this CTA reduces its share of the sub-tile's rows, splits in fixed order
      const int rbeg = (int)rank * BM / p.splits, rend = ((int)rank + 1) * BM / p.splits;
      for (int idx = threadIdx.x; idx < (rend - rbeg) * (BN / 4); idx += THREADS) {
        const int rr = rbeg + idx / (BN / 4), cc = (idx % (BN / 4)) * 4;
        const int row = m0 + mt * BM + rr;
        if (row >= M_eff) continue;
        float4 acc = ld_dsmem4(red + rr * RED_PITCH + cc, 0u);
        for (int s = 1; s < p.splits; ++s) {
          const float4 v = ld_dsmem4(red + rr * RED_PITCH + cc, (uint32_t)s);
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        float* dst = Cseg + (size_t)row * p.ldc + n0 + cc;
        if (n0 + cc + 4 <= segN && ((p.ldc & 3) == 0) && ((((uintptr_t)Cseg) & 15) == 0)) {
          *(float4*)dst = acc;
        } else {
          const float vv[4] = {acc.x, acc.y, acc.z, acc.w};
          for (int j = 0; j < 4; ++j)
            if (n0 + cc + j < segN) dst[j] = vv[j];
        }
      }
      cluster_sync();
    }
  }
  if (*abort_flag && warp == 0 && lane == 0) {
    // let in-flight bulk copies land before the CTA's shared memory is released
    const long long t0 = clock64();
    while (clock64() - t0 < 20000000LL) {
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(MT * BN));
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

const CUtensorMap* get_map(TcGemmCache* cache, const void* ptr, int rows, int cols, int ld, int box_rows) {
  const TcMapKey key{ptr, rows, cols, ld, box_rows};
  auto it = cache->maps.find(key);
  if (it != cache->maps.end()) return &it->second;
  auto fn = encode_fn();
  if (!fn) return nullptr;
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return nullptr;
  return &cache->maps.emplace(key, m).first->second;
}

template <int MT, int STAGES>
cudaError_t launch(const CUtensorMap* a, const CUtensorMap* const* b, const Params& p, dim3 grid, int splits,
                   cudaStream_t st) {
  auto kern = gemm_kernel<MT, STAGES>;
  constexpr int SMEM_BYTES = smem_bytes(MT, STAGES);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = splits;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, *a, *b[0], *b[1], *b[2], p);
}

}  // namespace tc

int* tc_error_word(TcGemmCache* cache) {
  if (!cache->err) {
    if (cudaMalloc(&cache->err, sizeof(int)) != cudaSuccess) return nullptr;
    cudaMemset(cache->err, 0, sizeof(int));
  }
  return cache->err;
}

bool tc_gemm_supported(int K, int lda, int ldw) {
  return K >= 16 && (lda % 8) == 0 && (ldw % 8) == 0;
}

cudaError_t tc_gemm_bf16_multi(TcGemmCache* cache, const void* A, int lda, int nseg, const void* const* W,
                               const int* ldw, const int* N, float* const* C, int ldc, int M, const int* m_dev,
                               int K, cudaStream_t st) {
  using namespace tc;
  if (M <= 0 || nseg < 1 || nseg > 3) return M <= 0 ? cudaSuccess : cudaErrorInvalidValue;
  if ((uintptr_t)A & 15) return cudaErrorInvalidValue;
  int* err = tc_error_word(cache);
  if (!err) return cudaErrorMemoryAllocation;
  if (cache->num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&cache->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (cache->num_sms <= 0) cache->num_sms = 148;
  }
  const int MT = M > BM ? 2 : 1;
  const int mgroups = (M + MT * BM - 1) / (MT * BM);
  const int ktiles = (K + BK - 1) / BK;
  Params p{};
  p.M = M;
  p.K = K;
  p.m_dev = m_dev;
  p.ldc = ldc;
  p.ktiles = ktiles;
  p.err = err;
  p.nseg = nseg;
  const CUtensorMap* mb[3] = {nullptr, nullptr, nullptr};
  int tiles = 0;
  for (int sgi = 0; sgi < 3; ++sgi) {
    p.seg_start[sgi] = sgi < nseg ? tiles : 0x3FFFFFFF;
    if (sgi < nseg) {
      if (((uintptr_t)W[sgi] & 15) || N[sgi] < 1) return cudaErrorInvalidValue;
      p.seg_N[sgi] = N[sgi];
      p.seg_C[sgi] = C[sgi];
      mb[sgi] = get_map(cache, W[sgi], N[sgi], K, ldw[sgi], BN);
      if (!mb[sgi]) return cudaErrorInvalidValue;
      tiles += (N[sgi] + BN - 1) / BN;
    }
  }
  p.seg_start[3] = 0x3FFFFFFF;
  for (int sgi = nseg; sgi < 3; ++sgi) mb[sgi] = mb[0];
  // split K over a cluster while the doubled grid still fits in one wave and
  // every split keeps at least 8 K-tiles (cluster size <= 8): only grids that
  // would leave most SMs idle pay for the cross-CTA reduction
  const int base = tiles * mgroups, nsm = cache->num_sms;
  int splits = 1;
  while (splits < 8 && base * splits * 2 <= nsm && ktiles >= splits * 2 * 8) splits *= 2;
  p.splits = splits;
  const CUtensorMap* ma = get_map(cache, A, M, K, lda, BM);
  if (!ma) return cudaErrorInvalidValue;
  const dim3 grid(tiles, mgroups, splits);
  // stage rings: deep (one CTA per SM) unless a single row group has more
  // tiles than SMs, where two CTAs per SM (3 stages each) avoid a second wave
  if (MT == 2) return launch<2, 4>(ma, mb, p, grid, splits, st);
  if (mgroups == 1 && splits == 1 && tiles > nsm) return launch<1, 3>(ma, mb, p, grid, splits, st);
  return launch<1, 6>(ma, mb, p, grid, splits, st);
}

cudaError_t tc_gemm_bf16(TcGemmCache* cache, const void* A, int lda, const void* W, int ldw, float* C, int ldc,
                         int M, const int* m_dev, int N, int K, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  return tc_gemm_bf16_multi(cache, A, lda, 1, &W, &ldw, &N, &C, ldc, M, m_dev, K, st);
}

void tc_gemm_cache_clear(TcGemmCache* c) {
  c->maps.clear();
  if (c->err) cudaFree(c->err);
  c->err = nullptr;
}

}  // namespace polestar
