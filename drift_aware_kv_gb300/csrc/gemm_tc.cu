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
#include <map>
#include <mutex>

#include "common.cuh"
#include "gemm_tc.h"

namespace polestar {

namespace tc {

constexpr int BM = 128;         // rows per UMMA
constexpr int BN = 128;         // columns per CTA
constexpr int BK = 64;          // K elements per stage (one 128-byte swizzle row)
constexpr int THREADS = 192;    // 6 warps
// Bound of every mbarrier wait of the kernels in this file, in SM clock cycles
// (default ~2 s at 2 GHz).  A device variable rather than a constant so that a
// test can shorten it and make a wait run out (tc_debug_stalled_wait); it is
// read only while a wait is already spinning.
constexpr long long TIMEOUT_CYCLES = 4000000000LL;
__device__ long long g_wait_limit_cycles = TIMEOUT_CYCLES;
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
  // ring depth and TMEM columns; row-tiled kernel: columns per tile (bn);
  // weight-stationary kernel: row box (np)
  int bn;
  int np;
  int stages;
  int tmem_cols;
  int ntn;    // persistent pair kernels: column tiles over all segments
  int nload;  // loader warps (1, 2 or 4; divides stages)
  // row-tiled kernel, SwiGLU mode: segments 0 (gate) and 1 (up) of equal width
  // seg_N[0]; tile t computes columns [t*bn/2, (t+1)*bn/2) of both (gate in
  // the accumulator's first half, up in the second) and writes
  // act[row, col] = bf16(silu(g) * u) (row stride ld_act) instead of C
  __nv_bfloat16* act;
  int ld_act;
  // two-SM pair kernel: 64-column k-blocks per stage (1, or 2 read by one 3D
  // TMA box per operand: fewer, larger copies per issuing warp)
  int kpack;
  // two-SM pair kernel: tiles walk groups of `group` row pairs, every column
  // block of a group before the next group (so a group's A rows stay in L2
  // while the weights stream past them)
  int group;
  // two-SM pair kernel, Q/K/V mode (segments Q, K, V of one layer, tiles of a
  // whole number of heads): the epilogue applies the rotary embedding and
  // writes bf16 Q rows and the K/V cache entries of the rows (as the row
  // kernel rope_scatter does) instead of C
  __nv_bfloat16* q_out;  // [M, qdim]
  const int4* qkv_rows;  // [M] {seq, pos, kind, aux}
  const uint8_t* qkv_write_kv;
  const float2* rope;    // [N][dh / 2] (cos, sin)
  __nv_bfloat16* kv_layer;
  long long kv_seq_stride;
  int kvdim, dh;
  // two-SM pair kernel, one plain segment: when the tiles leave the last wave
  // partly empty, each of those `rem` tiles is split along K over S clusters
  // (S = clusters / rem, capped).  Every split writes its partial tile to
  // tail_ws and counts it in tail_cnt; once all S are in, split s sums column
  // slice s of the tile over the splits in split order and writes it to C
  // (deterministic); the last split to finish clears the counters.  Null: no
  // split.
  float* tail_ws;  // [rem * S <= clusters][2 CTAs][BM][256] fp32
  int* tail_cnt;   // [rem][2 CTAs][4 lane quarters] x 32 ints (count, done at +16), zero between launches
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
    if (clock64() - t0 > g_wait_limit_cycles) {
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

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar)
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

__host__ __device__ constexpr uint32_t instr_desc_ws(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void umma_id(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// silu(g) * u, as the unfused SwiGLU kernel computes it
__device__ __forceinline__ float swiglu1(float g, float u) { return g / (1.f + expf(-g)) * u; }

// Row-tiled kernel: the gathered rows are the MMA's M side (MT sub-tiles of
// 128), a CTA owns p.bn (a multiple of 16, at most 256) output columns of one
// weight segment as the MMA's N side.  The column width is chosen per launch
// so that the tiles fill the SMs evenly (no second, mostly idle wave).
constexpr int RT_MAX_STAGES = 8;
__host__ __device__ constexpr int rt_stage_bytes(int mt, int bn) { return mt * BM * BK * 2 + bn * BK * 2; }
__host__ __device__ constexpr int rt_smem_bytes(int mt, int bn, int stages) {
  return stages * rt_stage_bytes(mt, bn) + 2048;
}

template <int MT>
__global__ void __launch_bounds__(THREADS)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2, Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  constexpr int A_BLK = BM * BK * 2;  // 16 KB: one row sub-tile x one 64-column k-block
  const int bn = p.bn, STAGES = p.stages;
  const int KP = p.kpack > 1 ? p.kpack : 1;  // k-blocks per stage (KP > 1: one 3D box per operand)
  const int A_BYTES = KP * A_BLK;            // one row sub-tile's k-blocks of a stage
  const int W_BLK = bn * BK * 2;             // one k-block of the W tile
  const int STAGE_BYTES = KP * rt_stage_bytes(MT, bn);
  const int pitch = bn + 4;             // fp32 staging row pitch of the split-K reduction
  uint64_t* full = (uint64_t*)(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + RT_MAX_STAGES;
  uint64_t* accum = empty + RT_MAX_STAGES;
  uint32_t* tmem_slot = (uint32_t*)(accum + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const bool glu = p.act != nullptr;  // SwiGLU mode: gate and up halves of one tile
  const int seg = glu ? 0 : (tile >= p.seg_start[1]) + (tile >= p.seg_start[2]);
  const int n0 = glu ? tile * (bn / 2) : (tile - p.seg_start[seg]) * bn;
  const int segN = p.seg_N[seg];
  float* const Cseg = p.seg_C[seg];
  const CUtensorMap* tmB = seg == 0 ? &tmB0 : (seg == 1 ? &tmB1 : &tmB2);
  const int m0 = blockIdx.y * (MT * BM);
  const int split = blockIdx.z;
  // W tile of a stage: one bn-row box, or in SwiGLU mode the gate and up boxes
  // of bn/2 rows each (the up half at row bn/2 of the tile)
  auto load_w = [&](uint32_t dst, int kb, uint32_t bar) {
    if (glu) {
      tma_load_2d(dst, &tmB0, kb * BK, n0, bar);
      tma_load_2d(dst + (bn / 2) * 128, &tmB1, kb * BK, n0, bar);
    } else if (KP == 1) {
      tma_load_2d(dst, tmB, kb * BK, n0, bar);
    } else {
      tma_load_3d(dst, tmB, 0, n0, kb, bar);
    }
  };
  auto load_a = [&](uint32_t dst, int kb, int row, uint32_t bar) {
    if (KP == 1)
      tma_load_2d(dst, &tmA, kb * BK, row, bar);
    else
      tma_load_3d(dst, &tmA, 0, row, kb, bar);
  };

  const int kt0 = (int)((long long)split * p.ktiles / p.splits);
  const int kt1 = (int)((long long)(split + 1) * p.ktiles / p.splits);
  const int nk = (kt1 - kt0 + KP - 1) / KP;  // stages of this CTA's K range

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
                 "r"(p.tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  // Loaders: warp 0 and, while the mainloop runs, epilogue warps 2-4; loader j
  // owns the stages s with s % nload == j (nload divides the ring depth), so
  // every stage is refilled in order by one warp.  One issuing warp keeps
  // about one TMA box in flight, so several loaders stream faster.
  const int lj = warp == 0 ? 0 : ((warp >= 2 && warp <= 4) ? warp - 1 : -1);
  const bool loader = lj >= 0 && lj < p.nload && lane == 0;
  // Weights never depend on earlier kernels: the first stages' W tiles are
  // requested before waiting for the predecessor that produces A (and m_dev).
  const int npre = nk < STAGES ? nk : STAGES;
  if (loader) {
    for (int i = lj; i < npre; i += p.nload) {
      const uint32_t fb = smem_u32(&full[i]);
      mbar_expect_tx(fb, STAGE_BYTES);
      load_w(smem_u32(smem + i * STAGE_BYTES) + MT * A_BYTES, kt0 + i * KP, fb);
    }
  }
  pdl_launch_dependents();
  pdl_wait();
  const int M_eff = p.m_dev ? min(p.M, *p.m_dev) : p.M;

  if (loader) {
    // ---------------- TMA producers
    for (int i = lj; i < npre; i += p.nload) {
      const uint32_t st = smem_u32(smem + i * STAGE_BYTES);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) load_a(st + mt * A_BYTES, kt0 + i * KP, m0 + mt * BM, smem_u32(&full[i]));
    }
    for (int i = npre; i < nk; ++i) {
      const int s = i % STAGES;
      if (s % p.nload != lj) continue;
      if (!mbar_wait(smem_u32(&empty[s]), ((i / STAGES) - 1) & 1, p.err, 1, abort_flag)) break;
      const uint32_t fb = smem_u32(&full[s]);
      mbar_expect_tx(fb, STAGE_BYTES);
      const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
      const int kb = kt0 + i * KP;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) load_a(st + mt * A_BYTES, kb, m0 + mt * BM, fb);
      load_w(st + MT * A_BYTES, kb, fb);
    }
  }
  if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = instr_desc_ws(bn);  // M = 128, N = bn
      for (int i = 0; i < nk; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(smem_u32(&full[s]), (i / STAGES) & 1, p.err, 2, abort_flag)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
        const uint32_t bst = st + MT * A_BYTES;
        // k-blocks of this stage inside this CTA's K range (a stage past the
        // range's end holds blocks of the next split: not multiplied)
        const int nkb = min(KP, kt1 - (kt0 + i * KP));
#pragma unroll 1
        for (int kb = 0; kb < nkb; ++kb) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              umma_id(tmem + mt * bn, smem_desc(st + mt * A_BYTES + kb * A_BLK + kk * 32),
                      smem_desc(bst + kb * W_BLK + kk * 32), idesc, (i > 0 || kb > 0 || kk > 0) ? 1u : 0u);
            }
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
  const bool vec = ((p.ldc & 3) == 0) && ((((uintptr_t)Cseg) & 15) == 0);
  const int half = bn / 2;
  const bool avec = glu && ((p.ld_act & 7) == 0) && ((((uintptr_t)p.act) & 15) == 0);
  if (p.splits == 1 && glu) {
    // SwiGLU epilogue: gate columns c and up columns half + c of each row
    if (epi && ok) {
#pragma unroll 1
      for (int mt = 0; mt < MT; ++mt) {
        const int row = m0 + mt * BM + q * 32 + lane;
        const uint32_t tr = tmem + ((uint32_t)(q * 32) << 16) + mt * bn;
#pragma unroll 1
        for (int c = 0; c < half; c += 8) {
          float g[8], u[8];
          tmem_ld8(tr + c, g);
          tmem_ld8(tr + half + c, u);
          if (row < M_eff) {
            __nv_bfloat16* dst = p.act + (size_t)row * p.ld_act + n0 + c;
            if (n0 + c + 8 <= segN && avec) {
              uint32_t w[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const __nv_bfloat162 b2 =
                    __floats2bfloat162_rn(swiglu1(g[2 * j], u[2 * j]), swiglu1(g[2 * j + 1], u[2 * j + 1]));
                w[j] = *(const uint32_t*)&b2;
              }
              *(uint4*)dst = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (n0 + c + j < segN) dst[j] = __float2bfloat16_rn(swiglu1(g[j], u[j]));
            }
          }
        }
      }
    }
  } else if (p.splits == 1) {
    if (epi && ok) {
#pragma unroll 1
      for (int mt = 0; mt < MT; ++mt) {
        const int row = m0 + mt * BM + q * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < bn; c += 16) {
          float v[16];
          tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + mt * bn + c, v);
          if (row < M_eff) {
            float* dst = Cseg + (size_t)row * p.ldc + n0 + c;
            if (n0 + c + 16 <= segN && vec) {
#pragma unroll
              for (int j = 0; j < 16; j += 4) *(float4*)(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (n0 + c + j < segN) dst[j] = v[j];
            }
          }
        }
      }
    }
  } else {
    // split-K: stage partials in shared memory, reduce across the cluster
    float* red = (float*)smem;  // [BM][pitch] fp32, pipeline buffers are idle now
    const uint32_t rank = cluster_rank();
#pragma unroll 1
    for (int mt = 0; mt < MT; ++mt) {
      __syncthreads();
      if (epi) {
        const int r = q * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < bn; c += 16) {
          float v[16];
          if (ok) tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + mt * bn + c, v);
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *(float4*)(red + r * pitch + c + j) =
                ok ? make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      cluster_sync();
      // this CTA reduces its share of the sub-tile's rows, splits in fixed order
      const int rbeg = (int)rank * BM / p.splits, rend = ((int)rank + 1) * BM / p.splits;
      if (glu) {
        // SwiGLU: gate columns cc.. and up columns half + cc.. of a row
        const int h4 = half / 4;
        for (int idx = threadIdx.x; idx < (rend - rbeg) * h4; idx += THREADS) {
          const int rr = rbeg + idx / h4, cc = (idx % h4) * 4;
          const int row = m0 + mt * BM + rr;
          if (row >= M_eff) continue;
          float4 ag = ld_dsmem4(red + rr * pitch + cc, 0u), au = ld_dsmem4(red + rr * pitch + half + cc, 0u);
          for (int s = 1; s < p.splits; ++s) {
            const float4 vg = ld_dsmem4(red + rr * pitch + cc, (uint32_t)s);
            const float4 vu = ld_dsmem4(red + rr * pitch + half + cc, (uint32_t)s);
            ag.x += vg.x;
            ag.y += vg.y;
            ag.z += vg.z;
            ag.w += vg.w;
            au.x += vu.x;
            au.y += vu.y;
            au.z += vu.z;
            au.w += vu.w;
          }
          const float a4[4] = {swiglu1(ag.x, au.x), swiglu1(ag.y, au.y), swiglu1(ag.z, au.z), swiglu1(ag.w, au.w)};
          __nv_bfloat16* dst = p.act + (size_t)row * p.ld_act + n0 + cc;
          for (int j = 0; j < 4; ++j)
            if (n0 + cc + j < segN) dst[j] = __float2bfloat16_rn(a4[j]);
        }
        cluster_sync();
        continue;
      }
      const int c4 = bn / 4;
      for (int idx = threadIdx.x; idx < (rend - rbeg) * c4; idx += THREADS) {
        const int rr = rbeg + idx / c4, cc = (idx % c4) * 4;
        const int row = m0 + mt * BM + rr;
        if (row >= M_eff) continue;
        float4 acc = ld_dsmem4(red + rr * pitch + cc, 0u);
        for (int s = 1; s < p.splits; ++s) {
          const float4 v = ld_dsmem4(red + rr * pitch + cc, (uint32_t)s);
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        float* dst = Cseg + (size_t)row * p.ldc + n0 + cc;
        if (n0 + cc + 4 <= segN && vec) {
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols));
  }
}

// ---------------------------------------------------------------- weight-stationary tile
// For at most 256 rows the operands swap roles: the 128 x 64 W tile is the
// MMA's A operand (M = 128 output features) and the activation rows are its B
// operand (N = the live row count rounded up to 16, read from m_dev on the
// device), so the accumulator is [128 features][np tokens] and the tensor work
// per streamed weight byte follows the live rows instead of a 128/256-row
// padding.  The TMA box still covers p.np rows; rows past M are zero-filled.
constexpr int WS_MAX_STAGES = 8;
constexpr int WS_W_BYTES = BN * BK * 2;  // 16 KB weight tile per stage
__host__ __device__ constexpr int ws_stage_bytes(int np) { return WS_W_BYTES + np * BK * 2; }
__host__ __device__ constexpr int ws_smem_bytes(int np, int stages) { return stages * ws_stage_bytes(np) + 2048; }

__global__ void __launch_bounds__(THREADS)
    gemm_ws_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2, Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int NP = p.np, STAGES = p.stages;
  const int STAGE_BYTES = ws_stage_bytes(NP);
  uint64_t* full = (uint64_t*)(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + WS_MAX_STAGES;
  uint64_t* accum = empty + WS_MAX_STAGES;
  uint32_t* tmem_slot = (uint32_t*)(accum + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int seg = (tile >= p.seg_start[1]) + (tile >= p.seg_start[2]);
  const int n0 = (tile - p.seg_start[seg]) * BN;
  const int segN = p.seg_N[seg];
  float* const Cseg = p.seg_C[seg];
  const CUtensorMap* tmB = seg == 0 ? &tmB0 : (seg == 1 ? &tmB1 : &tmB2);
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
                 "r"(p.tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  // loaders as in the row-tiled kernel: warp 0 and epilogue warps 2-4, each
  // owning the stages s with s % nload == its index
  const int lj = warp == 0 ? 0 : ((warp >= 2 && warp <= 4) ? warp - 1 : -1);
  const bool loader = lj >= 0 && lj < p.nload && lane == 0;
  // weight tiles of the first stages go out before waiting for the producer of A
  const int npre = nk < STAGES ? nk : STAGES;
  if (loader) {
    for (int i = lj; i < npre; i += p.nload) {
      const uint32_t fb = smem_u32(&full[i]);
      mbar_expect_tx(fb, STAGE_BYTES);
      tma_load_2d(smem_u32(smem + i * STAGE_BYTES), tmB, (kt0 + i) * BK, n0, fb);
    }
  }
  pdl_launch_dependents();
  pdl_wait();
  const int M_eff = p.m_dev ? min(p.M, *p.m_dev) : p.M;
  const int np_eff = min(NP, max(16, (M_eff + 15) & ~15));

  if (loader) {
    // ---------------- TMA producers
    for (int i = lj; i < npre; i += p.nload)
      tma_load_2d(smem_u32(smem + i * STAGE_BYTES) + WS_W_BYTES, &tmA, (kt0 + i) * BK, 0, smem_u32(&full[i]));
    for (int i = npre; i < nk; ++i) {
      const int s = i % STAGES;
      if (s % p.nload != lj) continue;
      if (!mbar_wait(smem_u32(&empty[s]), ((i / STAGES) - 1) & 1, p.err, 1, abort_flag)) break;
      const uint32_t fb = smem_u32(&full[s]);
      mbar_expect_tx(fb, STAGE_BYTES);
      const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
      const int kx = (kt0 + i) * BK;
      tma_load_2d(st, tmB, kx, n0, fb);
      tma_load_2d(st + WS_W_BYTES, &tmA, kx, 0, fb);
    }
  }
  if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = instr_desc_ws(np_eff);
      for (int i = 0; i < nk; ++i) {
        const int s = i % STAGES;
        if (!mbar_wait(smem_u32(&full[s]), (i / STAGES) & 1, p.err, 2, abort_flag)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_id(tmem, smem_desc(st + kk * 32), smem_desc(st + WS_W_BYTES + kk * 32), idesc,
                  (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(smem_u32(&empty[s]));
      }
      umma_commit(smem_u32(accum));
    }
  }
  __syncwarp();

  // ---------------- epilogue: TMEM lane = output feature, column = row
  const bool epi = warp >= 2;
  const int q = warp & 3;
  bool ok = true;
  if (epi) {
    ok = (nk > 0) && mbar_wait(smem_u32(accum), 0, p.err, 3, abort_flag);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  }
  const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
  if (p.splits == 1) {
    if (epi && ok) {
      const int f = n0 + q * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < np_eff; c += 16) {
        float v[16];
        tmem_ld16(tq + c, v);
        if (f < segN) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c + j < M_eff) Cseg[(size_t)(c + j) * p.ldc + f] = v[j];
        }
      }
    }
  } else {
    // split-K: stage [rows][features] partials, reduce across the cluster in rank order
    float* red = (float*)smem;
    const uint32_t rank = cluster_rank();
    __syncthreads();
    if (epi) {
#pragma unroll 1
      for (int c = 0; c < np_eff; c += 16) {
        float v[16];
        if (ok) tmem_ld16(tq + c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) red[(c + j) * RED_PITCH + q * 32 + lane] = ok ? v[j] : 0.f;
      }
    }
    cluster_sync();
    const int rbeg = (int)rank * np_eff / p.splits, rend = ((int)rank + 1) * np_eff / p.splits;
    for (int idx = threadIdx.x; idx < (rend - rbeg) * (BN / 4); idx += THREADS) {
      const int row = rbeg + idx / (BN / 4), cc = (idx % (BN / 4)) * 4;
      if (row >= M_eff) continue;
      float4 acc = ld_dsmem4(red + row * RED_PITCH + cc, 0u);
      for (int s = 1; s < p.splits; ++s) {
        const float4 v = ld_dsmem4(red + row * RED_PITCH + cc, (uint32_t)s);
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
  if (*abort_flag && warp == 0 && lane == 0) {
    const long long t0 = clock64();
    while (clock64() - t0 < 20000000LL) {
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols));
  }
}

// ---------------------------------------------------------------- two-SM pair tiles
// The same walk over 256-row x bn-column output tiles, with the pair's tensor
// cores working as one (tcgen05 cta_group::2, M = 256): CTA r of the pair stages
// only ITS 128 A rows and ITS half of the W tile, the leader CTA (rank 0)
// issues every MMA, which reads both CTAs' shared memory and writes each CTA's
// 128 accumulator rows into that CTA's TMEM.  Half the W bytes per stage buy a
// deeper ring (up to 7 stages of 32 KB at bn = 256) than staging the whole W
// tile in both CTAs.  Both CTAs' loads complete on the leader's stage barrier;
// the leader's MMA commits release the stage (and, per tile, the accumulator)
// in both CTAs; both CTAs' epilogue warps hand the accumulator back to the
// leader.  TMEM is allocated and freed by the pair together (cta_group::2).
constexpr int P2_MAX_STAGES = 8;
__host__ __device__ constexpr int p2_stage_bytes(int bn) { return BM * BK * 2 + (bn / 2) * BK * 2; }
__host__ __device__ constexpr int p2_smem_bytes(int bn, int stages) { return stages * p2_stage_bytes(bn) + 2048; }

__host__ __device__ constexpr uint32_t instr_desc_m256(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}
// tiled 2D load whose completion is counted on `bar`, an mbarrier of this CTA
// or of its pair peer (shared::cluster address)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void umma_pair(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_smem, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (arrivals from the pair peer);
// sleep_ns > 0 backs off between polls (waits that are long by design, so the
// polling warp leaves the issue slots of its scheduler to the MMA warp).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, int* err, int code,
                                                  volatile int* abort_flag, unsigned sleep_ns = 0) {
  const long long t0 = clock64();
  while (!mbar_try_cluster(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > g_wait_limit_cycles) {
      atomicExch(err, code);
      *abort_flag = 1;
      return false;
    }
    if (sleep_ns) __nanosleep(sleep_ns);
  }
  return true;
}

// Loaders: two issuing warps.  p.nload == 1 (the default): warp 0 issues every
// stage's A box and warp 6 its W half, each in stage order (one warp issuing
// both measured 7 % slower at LLaDA-8B batch 8).  p.nload == 2: warp 0 / 6
// issue both boxes of the stages s with s % 2 == 0 / 1 (the ring depth then
// even), so each stage's uses are issued in order by one warp and its parity
// waits never run more than one phase ahead of the barrier.
constexpr int P2_LOADERS = 2;
constexpr int P2_TAIL_MAX_SPLIT = 8;    // K splits of a tail tile at most
constexpr int P2_TAIL_MIN_SPLIT = 4;    // fewer possible splits: no split
constexpr int P2_TAIL_MIN_STAGES = 32;  // stages per tile below which tails are not split
// Tile t of the pair kernel's walk -> (row pair, column block): groups of g
// row pairs (the last one shorter), row pairs fastest inside a group.
__device__ __forceinline__ void p2_tile(long long t, int mpairs, int ntn, int g, int* mp, int* nb) {
  const long long per = (long long)g * ntn;
  const int grp = (int)(t / per);
  const int rem = (int)(t - (long long)grp * per);
  const int gm = min(g, mpairs - grp * g);
  *mp = grp * g + rem % gm;
  *nb = rem / gm;
}
constexpr int P2_THREADS = (6 + P2_LOADERS - 1) * 32;  // warps 0 and 6.. load, 1 MMA, 2-5 drain
__global__ void __launch_bounds__(P2_THREADS, 1)
    gemm_p2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2, Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  constexpr int A_BLK = BM * BK * 2;  // one 64-column k-block of the A rows
  const int STAGES = p.stages, bn = p.bn, KP = p.kpack;
  const int B_BLK = (bn / 2) * BK * 2;  // one k-block of this CTA's W half
  const int A_BYTES = KP * A_BLK;
  const int SB = KP * p2_stage_bytes(bn);
  uint64_t* full = (uint64_t*)(smem + STAGES * SB);  // used in the leader
  uint64_t* empty = full + P2_MAX_STAGES;
  uint64_t* acc_full = empty + P2_MAX_STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;          // [2], used in the leader
  uint32_t* tmem_slot = (uint32_t*)(acc_empty + 2);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_rank();  // 0 (leader) or 1
  const int cid = (int)blockIdx.x >> 1, ncl = (int)gridDim.x >> 1;
  constexpr uint16_t PAIR = 3;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);   // the leader's expect-tx arrival; bytes of both CTAs
      mbar_init(smem_u32(&empty[s]), 1);  // the leader's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 8);  // four epilogue warps of each CTA
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    // the pair allocates together: one warp of each CTA, same column range
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(p.tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  cluster_sync();
  // the pair's allocation must have given both CTAs the same columns (the MMA
  // writes the same TMEM address in both); otherwise report and do nothing
  if (threadIdx.x == 0) {
    uint32_t peer;
    asm volatile("ld.shared::cluster.u32 %0, [%1];"
                 : "=r"(peer)
                 : "r"(map_to_rank(smem_u32(tmem_slot), (uint32_t)(rank ^ 1)))
                 : "memory");
    if (peer != tmem) {
      atomicExch(p.err, 6);
      *abort_flag = 1;
    }
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();
  const int M_eff = p.m_dev ? min(p.M, *p.m_dev) : p.M;
  const int mpairs = (M_eff + 2 * BM - 1) / (2 * BM);
  const long long ntiles = *abort_flag ? 0 : (long long)mpairs * p.ntn;
  const int nk = (p.ktiles + KP - 1) / KP;  // stages per tile
  // Work of this cluster: its whole tiles t = cid + i ncl below full_tiles,
  // then (with a split tail) one K range of a tail tile.  Every cluster derives
  // the same schedule from the live row count.
  long long full_tiles = ntiles;
  int tail_S = 1, tail_rem = 0;
  if (p.tail_ws && ntiles > 0) {
    const long long full = ntiles / ncl;
    const int rem = (int)(ntiles - full * ncl);
    // measured on GB300: two- and three-way splits lost more to the partial
    // tiles' round trip than the shorter tail gained
    const int S = rem > 0 ? min(ncl / rem, P2_TAIL_MAX_SPLIT) : 1;
    if (S >= P2_TAIL_MIN_SPLIT && nk >= P2_TAIL_MIN_STAGES) {
      full_tiles = full * ncl;
      tail_S = S;
      tail_rem = rem;
    }
  }
  const bool has_tail = tail_S >= 2 && cid < tail_rem * tail_S;
  const int tail_tile = has_tail ? cid / tail_S : 0;  // 0 .. rem-1
  const int tail_s = has_tail ? cid % tail_S : 0;     // split of that tile
  const long long n_dp = full_tiles > cid ? (full_tiles - cid + ncl - 1) / ncl : 0;
  const long long n_units = n_dp + (has_tail ? 1 : 0);
  // unit i -> tile and stage range
  auto unit = [&](long long i, long long* t, int* k0, int* k1) {
    if (i < n_dp) {
      *t = cid + i * ncl;
      *k0 = 0;
      *k1 = nk;
    } else {
      *t = full_tiles + tail_tile;
      *k0 = (int)((long long)tail_s * nk / tail_S);
      *k1 = (int)((long long)(tail_s + 1) * nk / tail_S);
    }
  };

  if (warp == 0 || warp >= 6) {
    // ---------------- TMA producers, completing on the leader's stage barrier.
    // nload == 1: warp 0 issues every k-step's own A rows and warp 6 its own
    // half of the W tile (two issuing threads, each in stage order).  nload >
    // 1: loader j (warp 0, 6, 7, ...) issues both for the stages s with
    // s % nload == j.
    const int lj = warp == 0 ? 0 : warp - 5;
    const bool split_ab = p.nload == 1;
    const bool loads_a = !split_ab || warp == 0, loads_w = !split_ab || warp == 6;
    if (lane == 0 && (split_ab ? (warp == 0 || warp == 6) : lj < p.nload)) {
      long long it = 0;
      bool live = true;
      for (long long ui = 0; ui < n_units && live; ++ui) {
        long long t;
        int k0, k1;
        unit(ui, &t, &k0, &k1);
        int mp, nb;
        p2_tile(t, mpairs, p.ntn, p.group, &mp, &nb);
        const int sg = (nb >= p.seg_start[1]) + (nb >= p.seg_start[2]);
        // W rows of this CTA's half tile: rows n0 + rank bn/2 of segment sg, or
        // in SwiGLU mode gate (rank 0) / up (rank 1) rows of act columns n0..
        const CUtensorMap* tmB = p.act ? (rank == 0 ? &tmB0 : &tmB1) : (sg == 0 ? &tmB0 : (sg == 1 ? &tmB1 : &tmB2));
        const int wrow = p.act ? nb * (bn / 2) : (nb - p.seg_start[sg]) * bn + rank * (bn / 2);
        const int m0 = mp * 2 * BM + rank * BM;
        for (int k = k0; k < k1; ++k, ++it) {
          const int s = (int)(it % STAGES);
          if (!split_ab && s % p.nload != lj) continue;
          if (it >= STAGES && !mbar_wait_cluster(smem_u32(&empty[s]), (uint32_t)((it / STAGES) - 1) & 1u, p.err, 1,
                                                 abort_flag)) {
            live = false;
            break;
          }
          const uint32_t fb_local = smem_u32(&full[s]);
          if (rank == 0 && loads_a) mbar_expect_tx(fb_local, 2 * SB);
          const uint32_t fb = map_to_rank(fb_local, 0);
          const uint32_t st = smem_u32(smem + (size_t)s * SB);
          if (KP == 1) {
            if (loads_a) tma_load_2d_pair(st, &tmA, k * BK, m0, fb);
            if (loads_w) tma_load_2d_pair(st + A_BYTES, tmB, k * BK, wrow, fb);
          } else {
            // {column in the k-block, row, k-block}: KP consecutive k-blocks per box
            if (loads_a) tma_load_3d_pair(st, &tmA, 0, m0, k * KP, fb);
            if (loads_w) tma_load_3d_pair(st + A_BYTES, tmB, 0, wrow, k * KP, fb);
          }
        }
      }
      // the last uses of this loader's stages must be read before this CTA may exit
      if (live)
        for (long long u = (it > STAGES ? it - STAGES : 0); u < it; ++u)
          if ((split_ab || (int)(u % STAGES) % p.nload == lj) &&
              !mbar_wait_cluster(smem_u32(&empty[u % STAGES]), (uint32_t)(u / STAGES) & 1u, p.err, 4, abort_flag))
            break;
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader only): tile i into accumulator i % 2
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = instr_desc_m256(bn);
      long long it = 0;
      int tl = 0;
      bool live = true;
      for (long long ui = 0; ui < n_units && live; ++ui, ++tl) {
        long long t;
        int k0, k1;
        unit(ui, &t, &k0, &k1);
        const int b = tl & 1;
        if (tl >= 2 &&
            !mbar_wait_cluster(smem_u32(&acc_empty[b]), (uint32_t)((tl >> 1) - 1) & 1u, p.err, 5, abort_flag))
          break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + (uint32_t)(b * bn);
        for (int k = k0; k < k1; ++k, ++it) {
          const int s = (int)(it % STAGES);
          if (!mbar_wait_cluster(smem_u32(&full[s]), (uint32_t)(it / STAGES) & 1u, p.err, 2, abort_flag)) {
            live = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t st = smem_u32(smem + (size_t)s * SB);
#pragma unroll 1
          for (int kb = 0; kb < KP; ++kb) {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_pair(d, smem_desc(st + kb * A_BLK + kk * 32), smem_desc(st + A_BYTES + kb * B_BLK + kk * 32), idesc,
                        (k > k0 || kb > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&empty[s]), PAIR);  // stage s free in both CTAs once read
        }
        if (live) umma_commit_pair(smem_u32(&acc_full[b]), PAIR);
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ---------------- epilogue: TMEM lane quarter q = warp & 3 of this CTA's rows
    const int q = warp & 3;
    const bool vec = ((p.ldc & 3) == 0);
    const uint32_t lead_acc_empty0 = map_to_rank(smem_u32(&acc_empty[0]), 0);
    int tl = 0;
    for (long long ui = 0; ui < n_units; ++ui, ++tl) {
      long long t;
      int k0, k1;
      unit(ui, &t, &k0, &k1);
      const bool tail = ui >= n_dp;
      const int b = tl & 1;
      const bool ok =
          mbar_wait_cluster(smem_u32(&acc_full[b]), (uint32_t)(tl >> 1) & 1u, p.err, 3, abort_flag, 256);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (!ok) break;
      int mp, nb;
      p2_tile(t, mpairs, p.ntn, p.group, &mp, &nb);
      const int sg = (nb >= p.seg_start[1]) + (nb >= p.seg_start[2]);
      const int n0 = (nb - p.seg_start[sg]) * bn;
      const int segN = p.seg_N[sg];
      float* const Cseg = p.seg_C[sg];
      const bool vseg = vec && ((((uintptr_t)Cseg) & 15) == 0);
      const int row = mp * 2 * BM + rank * BM + q * 32 + lane;
      const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * bn);
      if (p.q_out) {
        // Q/K/V mode: segment sg 0 = Q, 1 = K (both rotated; proxy rows' Q is
        // not), 2 = V; K and V go to the cache row (seq, pos) of active,
        // other and (when flagged) window rows
        int4 m = make_int4(0, 0, ROW_NONE, 0);
        if (row < M_eff) m = p.qkv_rows[row];
        const bool rot = sg == 1 || m.z != ROW_PROXY;
        const bool wkv = (m.z == ROW_ACTIVE || m.z == ROW_OTHER) ||
                         (m.z == ROW_WINDOW && (!p.qkv_write_kv || p.qkv_write_kv[row]));
        const bool put = m.z != ROW_NONE && (sg == 0 || wkv);
        __nv_bfloat16* dst = sg == 0 ? p.q_out + (size_t)row * p.seg_N[0] + n0
                                     : p.kv_layer + (size_t)m.x * p.kv_seq_stride + (size_t)m.y * 2 * p.kvdim +
                                           (sg == 2 ? p.kvdim : 0) + n0;
        auto put16 = [&](__nv_bfloat16* o, const float* y) {
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const __nv_bfloat162 v2 = __floats2bfloat162_rn(y[2 * e], y[2 * e + 1]);
            w[e] = *(const uint32_t*)&v2;
          }
          *(uint4*)o = make_uint4(w[0], w[1], w[2], w[3]);
          *(uint4*)(o + 8) = make_uint4(w[4], w[5], w[6], w[7]);
        };
        if (sg < 2) {
          const int hd = p.dh / 2;
#pragma unroll 1
          for (int hh = 0; hh < bn / p.dh; ++hh) {
#pragma unroll 1
            for (int c0 = 0; c0 < hd; c0 += 16) {
              float a[16], b2[16];
              tmem_ld16(tq + hh * p.dh + c0, a);
              tmem_ld16(tq + hh * p.dh + hd + c0, b2);
              if (put) {
                if (rot) {
                  const float2* tab = p.rope + (size_t)m.y * hd + c0;
#pragma unroll
                  for (int e = 0; e < 16; ++e) {
                    const float2 cs = tab[e];
                    float y1, y2;
                    rope_rotate(a[e], b2[e], cs.x, cs.y, y1, y2);
                    a[e] = y1;
                    b2[e] = y2;
                  }
                }
                put16(dst + hh * p.dh + c0, a);
                put16(dst + hh * p.dh + hd + c0, b2);
              }
            }
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < bn; c += 16) {
            float v[16];
            tmem_ld16(tq + c, v);
            if (put) put16(dst + c, v);
          }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead_acc_empty0 + (uint32_t)(b * 8));
        continue;
      }
      if (p.act) {
        // SwiGLU mode: gate in the accumulator's first bn/2 columns, up in the
        // second; act[row, nb bn/2 + c] = bf16(silu(g) * u)
        const int a0 = nb * (bn / 2), F = p.seg_N[0];
        const bool va = ((p.ld_act & 7) == 0) && ((((uintptr_t)p.act) & 15) == 0);
#pragma unroll 1
        for (int c = 0; c < bn / 2; c += 16) {
          float g[16], u[16];
          tmem_ld16(tq + c, g);
          tmem_ld16(tq + bn / 2 + c, u);
          if (row < M_eff) {
            __nv_bfloat16* dst = p.act + (size_t)row * p.ld_act + a0 + c;
            if (a0 + c + 16 <= F && va) {
              uint32_t w[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const __nv_bfloat162 v2 = __floats2bfloat162_rn(swiglu1(g[2 * j], u[2 * j]), swiglu1(g[2 * j + 1], u[2 * j + 1]));
                w[j] = *(const uint32_t*)&v2;
              }
              *(uint4*)dst = make_uint4(w[0], w[1], w[2], w[3]);
              *(uint4*)(dst + 8) = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (a0 + c + j < F) dst[j] = __float2bfloat16_rn(swiglu1(g[j], u[j]));
            }
          }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lead_acc_empty0 + (uint32_t)(b * 8));
        continue;
      }
      if (tail) {
        // split tail tile: every split writes its partial rows, waits for the
        // other splits' (bounded), then sums one column slice of the tile over
        // all splits in split order and writes it to C (deterministic)
        int* const cnt = p.tail_cnt + (((size_t)tail_tile * 2 + rank) * 4 + q) * 32;  // own 128-byte line
        int* const done = cnt + 16;
        const size_t wsplit = (size_t)2 * BM * 256;  // floats between consecutive splits' partials
        float* const w0 = p.tail_ws + (((size_t)tail_tile * tail_S * 2 + rank) * BM + q * 32 + lane) * 256;
#pragma unroll 1
        for (int c = 0; c < bn; c += 16) {
          float v[16];
          tmem_ld16(tq + c, v);
          float* w = w0 + tail_s * wsplit + c;
#pragma unroll
          for (int j = 0; j < 16; j += 4) *(float4*)(w + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
        // accumulator drained: the MMA warp may go on
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_cluster(lead_acc_empty0 + (uint32_t)(b * 8));
          __threadfence();
          atomicAdd(cnt, 1);
          const long long t0 = clock64();
          while (true) {
            int got;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(got) : "l"(cnt) : "memory");
            if (got >= tail_S) break;
            if (*abort_flag) break;
            if (clock64() - t0 > g_wait_limit_cycles) {
              atomicExch(p.err, 7);
              *abort_flag = 1;
              break;
            }
            __nanosleep(64);
          }
        }
        __syncwarp();
        int got;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(got) : "l"(cnt) : "memory");
        if (got >= tail_S && row < M_eff) {
          const int n4 = bn / 4;
          const int c4a = (int)((long long)tail_s * n4 / tail_S), c4b = (int)((long long)(tail_s + 1) * n4 / tail_S);
          float* dst = Cseg + (size_t)row * p.ldc + n0;
          // two float4 columns per pass with every split's loads in flight
          // together (up to P2_TAIL_MAX_SPLIT x 2 independent 16-byte loads)
#pragma unroll 1
          for (int c4 = c4a; c4 < c4b; c4 += 2) {
            const bool two = c4 + 1 < c4b;
            float4 x0[P2_TAIL_MAX_SPLIT], x1[P2_TAIL_MAX_SPLIT];
#pragma unroll
            for (int sp = 0; sp < P2_TAIL_MAX_SPLIT; ++sp) {
              if (sp < tail_S) {
                const float* w = w0 + sp * wsplit + c4 * 4;
                x0[sp] = *(const float4*)w;
                x1[sp] = two ? *(const float4*)(w + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
              }
            }
            float4 a0 = x0[0], a1 = x1[0];
#pragma unroll
            for (int sp = 1; sp < P2_TAIL_MAX_SPLIT; ++sp) {
              if (sp < tail_S) {
                a0.x += x0[sp].x;
                a0.y += x0[sp].y;
                a0.z += x0[sp].z;
                a0.w += x0[sp].w;
                a1.x += x1[sp].x;
                a1.y += x1[sp].y;
                a1.z += x1[sp].z;
                a1.w += x1[sp].w;
              }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              if (u == 1 && !two) continue;
              const float4 av = u ? a1 : a0;
              const int col = (c4 + u) * 4;
              if (n0 + col + 4 <= segN && vseg) {
                *(float4*)(dst + col) = av;
              } else {
                const float e[4] = {av.x, av.y, av.z, av.w};
                for (int j = 0; j < 4; ++j)
                  if (n0 + col + j < segN) dst[col + j] = e[j];
              }
            }
          }
        }
        // the last split to finish reading clears both counters for the next launch
        __syncwarp();
        if (lane == 0) {
          const int d = atomicAdd(done, 1);
          if (d == tail_S - 1) {
            *cnt = 0;
            *done = 0;
          }
        }
        continue;
      }
#pragma unroll 1
      for (int c = 0; c < bn; c += 16) {
        float v[16];
        tmem_ld16(tq + c, v);
        if (row < M_eff) {
          float* dst = Cseg + (size_t)row * p.ldc + n0 + c;
          if (n0 + c + 16 <= segN && vseg) {
#pragma unroll
            for (int j = 0; j < 16; j += 4) *(float4*)(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (n0 + c + j < segN) dst[j] = v[j];
          }
        }
      }
      // accumulator drained in this CTA: tell the leader's MMA warp
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lead_acc_empty0 + (uint32_t)(b * 8));
    }
  }
  if (*abort_flag && (warp == 0 || warp >= 6) && lane == 0) {
    // let in-flight bulk copies land before the CTA's shared memory is released
    const long long t0 = clock64();
    while (clock64() - t0 < 20000000LL) {
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  // neither CTA of the pair leaves (or frees TMEM) while the other still works
  cluster_sync();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols));
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

// 3D view {column within a 64-column k-block, row, k-block} of a row-major
// bf16 matrix: a box of `kblocks` k-blocks lands as that many consecutive
// 128B-swizzled [box_rows][64] tiles (the same image as separate 2D boxes).
const CUtensorMap* get_map3(TcGemmCache* cache, const void* ptr, int rows, int cols, int ld, int box_rows,
                            int kblocks) {
  const TcMapKey key{ptr, rows, cols, ld, box_rows | (kblocks << 16)};
  auto it = cache->maps.find(key);
  if (it != cache->maps.end()) return &it->second;
  auto fn = encode_fn();
  if (!fn) return nullptr;
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  const cuuint64_t dims[3] = {(cuuint64_t)BK, (cuuint64_t)rows, (cuuint64_t)((cols + BK - 1) / BK)};
  const cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)BK * 2};
  const cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, (cuuint32_t)kblocks};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return nullptr;
  return &cache->maps.emplace(key, m).first->second;
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

template <int MT>
cudaError_t launch_rt(const CUtensorMap* a, const CUtensorMap* const* b, const Params& p, dim3 grid,
                      cudaStream_t st) {
  static PerDeviceOnce attr;
  {
    const cudaError_t e =
        func_attr_once(attr, (const void*)gemm_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
  }
  // at most 512 / tmem_cols CTAs may share an SM (see launch_ws)
  const int resident = 512 / p.tmem_cols;
  const int kp = p.kpack > 1 ? p.kpack : 1;
  const int smem = std::max(kp * p.stages * rt_stage_bytes(MT, p.bn) + 2048, 233472 / (resident + 1) - 1024 + 16);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = p.splits;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<MT>, *a, *b[0], *b[1], *b[2], p);
}

int rt_tiles(const int* N, int nseg, int bn) {
  int t = 0;
  for (int i = 0; i < nseg; ++i) t += (N[i] + bn - 1) / bn;
  return t;
}

int rt_max_stages(int mt, int bn) { return std::min(RT_MAX_STAGES, (232448 - 2048) / rt_stage_bytes(mt, bn)); }

// Ring depth of the weight-stationary kernel when `ctas` CTAs share an SM.
int ws_stages_for(int np, int ctas, int splits) {
  const int budget = ctas == 1 ? 232448 : 115712;  // per-CTA dynamic shared memory
  int s = std::min(WS_MAX_STAGES, (budget - 2048) / ws_stage_bytes(np));
  // the split-K reduction reuses the ring for np x RED_PITCH fp32 partials
  if (splits > 1 && s * ws_stage_bytes(np) < np * RED_PITCH * 4) s = 0;
  return s;
}

// Stand-in for the occupancy queries below; never launched.  The occupancy
// calculator treats any kernel that allocates tensor memory as one CTA per SM,
// while the hardware runs as many as shared memory allows (measured: a
// 3-stage weight-stationary launch shows no second wave up to 2 CTAs per SM).
// The launchers pad shared memory so co-resident CTAs never ask for more than
// 512 TMEM columns between them, so a kernel without tensor memory, with the
// same threads and the same launch shared memory, gives the true capacity.
__global__ void __launch_bounds__(THREADS) occupancy_standin_kernel(int* p) {
  if (p) p[threadIdx.x] = threadIdx.x;
}

// Clusters of `cluster` CTAs of THREADS threads and `smem` bytes of dynamic
// shared memory that the device runs at once; 0 when the query is unavailable.
int max_active_clusters(int smem, int cluster) {
  static std::map<std::pair<int, int>, int> memo;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  const std::pair<int, int> key{smem, cluster};
  auto it = memo.find(key);
  if (it != memo.end()) return it->second;
  const void* func = (const void*)occupancy_standin_kernel;
  int n = 0;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448) == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1, 1, cluster);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = cluster;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  memo[key] = n;
  return n;
}

// Launch choice for at most 256 rows (one row group).  Candidates: the
// row-tiled kernel at every column width (one CTA per SM) and the
// weight-stationary kernel (128-column tiles) with 1-4 CTAs resident per SM,
// each with a K split of 1-8 and every CTA (and cluster) resident at once
// (cudaOccupancyMaxActiveClusters).  A candidate's time is the bytes streamed
// by the busiest SM - per CTA its weight columns plus, at half weight, its box
// of A rows read from L2 - at one SM's share of the HBM bandwidth, credited 1.5x
// (1.6x) when two (three or more) independent load pipelines share the SM,
// plus 0.4 us per cluster split for the reduction.  (Measured on GB300 over the
// projection shapes of the layer loop against forced sweeps of every
// configuration: the pick is the fastest or within a few percent of it.)
// Loader warps for a ring of `stages`.  The kernels take up to four (each
// owning the stages s = j mod n), but on GB300 more loaders measured no faster
// and a few percent slower at the layer-loop shapes (and ring depths that are
// multiples of four are common), so one warp issues every stage.
int loaders_for(int stages) {
  (void)stages;
  return 1;
}

struct GemmPick {
  int kernel;  // 1 row-tiled, 2 weight-stationary, 5 two-SM pair tiles
  int bn, splits, stages;
};

GemmPick pick_small_m(int MT, int M, const int* N, int nseg, int ktiles, int nsm) {
  GemmPick best{1, 128, 1, 0};
  double tbest = 1e30;
  const int np = std::max(16, (M + 15) & ~15);
  int ws_tmem = 32;
  while (ws_tmem < np) ws_tmem *= 2;
  // kernel 1: resident = 1; kernel 2: resident CTAs per SM and ring depth given
  auto consider = [&](int kernel, int bn, int s, int resident, int stages, double a_rows) {
    const long long ctas = (long long)rt_tiles(N, nseg, bn) * s;
    if (ctas > (long long)nsm * resident) return;
    int smem;
    if (kernel == 1) {
      int tmem = 32;
      while (tmem < MT * bn) tmem *= 2;
      smem = std::max(rt_smem_bytes(MT, bn, stages), 233472 / (512 / tmem + 1) - 1024 + 16);
    } else {
      smem = std::max(ws_smem_bytes(np, stages), 233472 / (512 / ws_tmem + 1) - 1024 + 16);
    }
    if (s > 1) {
      // every cluster must be resident at once (a cluster size that does not
      // divide the SMs of a GPC leaves some idle and forces a second wave)
      // (with a tenth of the capacity to spare: a grid that needs every last
      // cluster slot was measured to spill clusters into a second wave)
      const int mc = max_active_clusters(smem, s);
      if (mc <= 0 || (double)(ctas / s) > 0.9 * mc) return;
    }
    const long long per_sm = (ctas + nsm - 1) / nsm;
    const double credit = per_sm >= 3 ? 1.6 : (per_sm == 2 ? 1.5 : 1.0);
    const double kel = (double)ktiles * BK / s;
    const double t = per_sm * (bn + 0.5 * a_rows) * kel * 2.0 / 50e3 / credit + 0.4 * s;
    if (t < tbest * 0.999) {
      tbest = t;
      best = GemmPick{kernel, bn, s, stages};
    }
  };
  for (int s = 1; s <= 8; ++s) {
    if (s > 1 && ktiles < 8 * s) break;
    for (int bn = 16; bn <= 256; bn += 16) {
      if (MT * bn > 512 || rt_max_stages(MT, bn) < 3) continue;
      if (s > 1 && rt_max_stages(MT, bn) * rt_stage_bytes(MT, bn) < BM * (bn + 4) * 4) continue;
      consider(1, bn, s, 1, rt_max_stages(MT, bn), MT * BM);
    }
    // (rings shallower than 3 stages and reductions over more than 4 CTAs were
    // measured slower than the time estimate says; they are not candidates)
    for (int r = 1; r <= 4 && r * ws_tmem <= 512 && s <= 4; ++r) {
      const int budget = 233472 / r - 1024;  // dynamic shared memory per CTA for r per SM
      const int stages = std::min(WS_MAX_STAGES, (budget - 2048) / ws_stage_bytes(np));
      if (stages < 3) break;
      if (s > 1 && stages * ws_stage_bytes(np) < np * RED_PITCH * 4) continue;
      consider(2, BN, s, r, stages, np);
    }
  }
  if (tbest >= 1e30) {
    // more 16-column tiles than SMs even unsplit: widest tiles, several waves
    best = GemmPick{1, 256 / MT, 1, 0};
  }
  return best;
}

int p2_default_stages(int bn);
int p2_max_stages(int bn, int kpack);
int p2_clusters(int bn, int stages, long long pair_tiles, int nsm);

// More than 256 rows (several 256-row groups): the GEMM is bound by how fast
// the SMs' pipelines are fed, which measurements on GB300 put per k-step (64
// K-elements) at about 0.415 us for a two-SM pair tile (256 x 256) and
// 0.43 + 0.0022 (bn - 64) us for a row-tiled CTA (256 x bn), whatever the
// operands' bytes.  Candidates: the two-SM pair kernel (persistent, 256 x bn
// tiles, bn 256/224/192) at waves of its resident clusters x (k-steps x 0.415
// + 2 us), and the row-tiled kernel at every column width, waves of one CTA
// per SM x (k-steps x its step cost + 3 us), with a cluster K split of 2 or 4
// costing another 12 us per wave for the reduction of the 256-row partials.
GemmPick pick_large_m(int M, const int* N, int nseg, int ktiles, int nsm, int K) {
  const int MT = 2, mgroups = (M + 2 * BM - 1) / (2 * BM);
  GemmPick best{1, 256, 1, rt_max_stages(MT, 256)};
  double tbest = 1e30;
  // pair kernel: two k-blocks per stage (one 3D box per operand) when K is
  // whole k-blocks, measured at 0.355 us per k-block against 0.415 with one
  const int kp = (ktiles * BK == K) ? 2 : 1;
  for (int bn = 256; bn >= 192; bn -= 32) {
    const int st = kp == 2 ? p2_max_stages(bn, 2) : p2_default_stages(bn);
    const long long tiles = (long long)mgroups * rt_tiles(N, nseg, bn);
    const int ncl = p2_clusters(bn, st, tiles, nsm);
    const long long waves = (tiles + ncl - 1) / ncl;
    const double t = waves * (ktiles * (kp == 2 ? 0.355 : 0.415) + 2.0);
    if (t < tbest * 0.999) {
      tbest = t;
      best = GemmPick{5, bn, kp, st};  // splits field: k-blocks per stage
    }
  }
  for (int s = 1; s <= 4; s *= 2) {
    if (s > 1 && ktiles < 8 * s) break;
    for (int bn = 64; bn <= 256; bn += 16) {
      if (rt_max_stages(MT, bn) < 3) continue;
      if (s > 1 && rt_max_stages(MT, bn) * rt_stage_bytes(MT, bn) < BM * (bn + 4) * 4) continue;
      const long long ctas = (long long)rt_tiles(N, nseg, bn) * mgroups * s;
      long long waves = (ctas + nsm - 1) / nsm;
      if (s > 1) {
        int tmem = 32;
        while (tmem < MT * bn) tmem *= 2;
        const int smem = std::max(rt_smem_bytes(MT, bn, rt_max_stages(MT, bn)), 233472 / (512 / tmem + 1) - 1024 + 16);
        const int mc = max_active_clusters(smem, s);
        if (mc <= 0) continue;
        waves = (ctas / s + mc - 1) / mc;
      }
      const double step = 0.43 + 0.0022 * (bn - 64);
      const double t = waves * ((double)ktiles / s * step + 3.0 + (s > 1 ? 12.0 : 0.0));
      if (t < tbest * 0.999) {
        tbest = t;
        best = GemmPick{1, bn, s, rt_max_stages(MT, bn)};
      }
    }
  }
  return best;
}


// The automatic choice for M rows (one row group: pick_small_m, else
// pick_large_m), memoised per shape in the context's cache.
GemmPick pick_for(TcGemmCache* cache, int M, const int* N, int nseg, int ktiles, int nsm, int K) {
  const std::array<int, 7> key{M, K, nseg, N[0], nseg > 1 ? N[1] : 0, nseg > 2 ? N[2] : 0, nsm};
  auto it = cache->picks.find(key);
  if (it != cache->picks.end()) return GemmPick{it->second[0], it->second[1], it->second[2], it->second[3]};
  const int MT = M > BM ? 2 : 1;
  const int mgroups = (M + MT * BM - 1) / (MT * BM);
  const GemmPick pk = mgroups > 1 ? pick_large_m(M, N, nseg, ktiles, nsm, K) : pick_small_m(MT, M, N, nseg, ktiles, nsm);
  cache->picks.emplace(key, std::array<int, 4>{pk.kernel, pk.bn, pk.splits, pk.stages});
  return pk;
}

int p2_launch_smem(int bn, int stages, int kpack = 1) {
  return std::max(kpack * p2_smem_bytes(bn, stages) - (kpack - 1) * 2048, 233472 / 2 - 1024 + 16);
}
int p2_max_stages(int bn, int kpack = 1) {
  return std::min(P2_MAX_STAGES, (232448 - 2048) / (kpack * p2_stage_bytes(bn)));
}
// default ring depth: the deepest that fits (measured: depth, not loader
// count, decides; 7 stages at bn = 256 beat 4 stages with four loaders)
int p2_default_stages(int bn) { return p2_max_stages(bn); }

// Two-SM pair kernel: clusters of two CTAs, one CTA per SM.
int p2_clusters(int bn, int stages, long long pair_tiles, int nsm) {
  int mc = max_active_clusters(p2_launch_smem(bn, stages), 2);
  if (mc <= 0) mc = nsm / 2;
  return (int)std::max<long long>(1, std::min<long long>(mc, pair_tiles));
}

// Row pairs per group of the pair kernel's tile walk: about 48 MB of A rows
// (2 x 128 rows x K bf16 per pair), so that a group's rows stay in the 129 MB
// L2 while every weight column block passes them once.  Walking row pairs
// fastest over all of A instead (A re-read from DRAM for every column block)
// read 4.5 GB for a 16384 x 12288 x 4096 launch whose operands hold 234 MB.
int p2_group(int M, int K) {
  const int mpairs = (M + 2 * BM - 1) / (2 * BM);
  const long long pair_bytes = 2LL * BM * K * 2;
  const int g = (int)std::max(1LL, (48LL << 20) / std::max(1LL, pair_bytes));
  return std::max(1, std::min(mpairs, g));
}

cudaError_t launch_p2(const CUtensorMap* a, const CUtensorMap* const* b, const Params& p, int nclusters,
                      cudaStream_t st) {
  static PerDeviceOnce attr;
  {
    const cudaError_t e =
        func_attr_once(attr, (const void*)gemm_p2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * nclusters, 1, 1);
  cfg.blockDim = dim3(P2_THREADS);
  cfg.dynamicSmemBytes = p2_launch_smem(p.bn, p.stages, p.kpack);
  cfg.stream = st;
  // No programmatic dependent launch for this kernel: with it (and the row
  // kernels around it launched the same way) the layer loop of the LLaDA-8B
  // batch-32 workload stalled on GB300 within a few steps, with no bounded
  // wait giving up; launched in plain stream order it did not.  The kernel runs
  // only for more than 256 rows, where a launch gap is small against its work.
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_p2_kernel, *a, *b[0], *b[1], *b[2], p);
}

cudaError_t launch_ws(const CUtensorMap* a, const CUtensorMap* const* b, const Params& p, dim3 grid,
                      cudaStream_t st) {
  static PerDeviceOnce attr;
  {
    const cudaError_t e =
        func_attr_once(attr, (const void*)gemm_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
  }
  // CTAs that share an SM must never ask for more than its 512 TMEM columns
  // between them (a blocked tcgen05.alloc inside a cluster that waits for its
  // peers could wait forever): pad the shared memory so that at most
  // 512 / tmem_cols CTAs fit on one SM (228 KB per SM, 1 KB reserved per CTA)
  const int resident = 512 / p.tmem_cols;
  const int smem = std::max(ws_smem_bytes(p.np, p.stages), 233472 / (resident + 1) - 1024 + 16);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = p.splits;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_ws_kernel, *a, *b[0], *b[1], *b[2], p);
}

// A wait that nothing ever satisfies: one thread initialises an mbarrier with
// one expected arrival, never arrives, and waits for its first phase with the
// same bounded wait as the GEMM kernels, which gives up after the limit and
// records `code` in the error word.
__global__ void stalled_wait_kernel(int* err, int code) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(smem_u32(&bar), 0, err, code, (volatile int*)&abort_flag);
  }
}

}  // namespace tc

cudaError_t tc_debug_stalled_wait(int* err, int code, long long limit_cycles, cudaStream_t st) {
  if (!err || limit_cycles < 1) return cudaErrorInvalidValue;
  const long long lim = limit_cycles, def = tc::TIMEOUT_CYCLES;
  cudaError_t e = cudaMemcpyToSymbolAsync(tc::g_wait_limit_cycles, &lim, sizeof(lim), 0, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  tc::stalled_wait_kernel<<<1, 32, 0, st>>>(err, code);
  e = cudaGetLastError();
  // the default bound again for every later launch on this stream
  const cudaError_t e2 = cudaMemcpyToSymbolAsync(tc::g_wait_limit_cycles, &def, sizeof(def), 0,
                                                 cudaMemcpyHostToDevice, st);
  return e != cudaSuccess ? e : e2;
}

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
                               int K, cudaStream_t st, const TcGemmChoice* force) {
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
  const int nsm = cache->num_sms;
  int kind = force && force->kernel ? force->kernel : 0;
  // columns per tile: 128 for the weight-stationary kernels (the MMA's M side),
  // chosen per launch for the row-tiled kernel (its N side)
  int bn = BN, auto_splits = 0, auto_stages = 0;
  if (kind == 0) {
    if (mgroups == 1) {
      const GemmPick pk = pick_for(cache, M, N, nseg, ktiles, nsm, K);
      kind = pk.kernel;
      bn = pk.bn;
      auto_splits = pk.splits;
      auto_stages = pk.stages;
    } else {
      const GemmPick pk = pick_for(cache, M, N, nseg, ktiles, nsm, K);
      kind = pk.kernel;
      bn = pk.bn;
      auto_splits = pk.splits;
      if (kind == 5) auto_stages = pk.stages;
    }
  } else if (kind == 1 && force->bn) {
    bn = force->bn;
    if (bn < 16 || bn > 256 || (bn & 15) || MT * bn > 512) return cudaErrorInvalidValue;
  } else if (kind == 1) {
    bn = pick_for(cache, M, N, nseg, ktiles, nsm, K).bn;
  }
  const CUtensorMap* mb[3] = {nullptr, nullptr, nullptr};
  int tiles = 0;
  for (int sgi = 0; sgi < 3; ++sgi) {
    p.seg_start[sgi] = sgi < nseg ? tiles : 0x3FFFFFFF;
    if (sgi < nseg) {
      if (((uintptr_t)W[sgi] & 15) || N[sgi] < 1) return cudaErrorInvalidValue;
      p.seg_N[sgi] = N[sgi];
      p.seg_C[sgi] = C[sgi];
      mb[sgi] = get_map(cache, W[sgi], N[sgi], K, ldw[sgi], bn);
      if (!mb[sgi]) return cudaErrorInvalidValue;
      tiles += (N[sgi] + bn - 1) / bn;
    }
  }
  p.seg_start[3] = 0x3FFFFFFF;
  for (int sgi = nseg; sgi < 3; ++sgi) mb[sgi] = mb[0];
  if (kind == 5) {
    // two-SM pair tiles: each CTA's W box is half a tile, read by the pair's MMA
    p.bn = force && force->bn ? force->bn : (auto_stages ? bn : 256);
    if (p.bn < 16 || p.bn > 256 || (p.bn & 15)) return cudaErrorInvalidValue;
    // k-blocks per stage (forced through the split field)
    p.kpack = force && force->kernel == 5 && force->splits ? force->splits : (auto_splits ? auto_splits : 1);
    // the 3D view has no out-of-range fill inside a k-block: whole k-blocks only
    if (p.kpack < 1 || p.kpack > 2 || (p.kpack > 1 && K % BK)) return cudaErrorInvalidValue;
    const int max_stages = p2_max_stages(p.bn, p.kpack);
    const int def_stages = p.kpack == 1 ? p2_default_stages(p.bn) : max_stages;
    p.stages = force && force->stages ? force->stages : (auto_stages ? auto_stages : def_stages);
    if (p.stages < 2 || p.stages > max_stages) return cudaErrorInvalidValue;
    p.splits = 1;
    p.nload = loaders_for(p.stages);
    p.tmem_cols = 32;
    while (p.tmem_cols < 2 * p.bn) p.tmem_cols *= 2;
    p.ntn = rt_tiles(N, nseg, p.bn);
    for (int sgi = 0, t = 0; sgi < 3; ++sgi) {
      p.seg_start[sgi] = sgi < nseg ? t : 0x3FFFFFFF;
      if (sgi < nseg) {
        mb[sgi] = p.kpack == 1 ? get_map(cache, W[sgi], N[sgi], K, ldw[sgi], p.bn / 2)
                               : get_map3(cache, W[sgi], N[sgi], K, ldw[sgi], p.bn / 2, p.kpack);
        if (!mb[sgi]) return cudaErrorInvalidValue;
        t += (N[sgi] + p.bn - 1) / p.bn;
      }
    }
    for (int sgi = nseg; sgi < 3; ++sgi) mb[sgi] = mb[0];
    const long long pair_tiles = (long long)((M + 2 * BM - 1) / (2 * BM)) * p.ntn;
    const int ncl = p2_clusters(p.bn, p.stages, pair_tiles, nsm);
    p.group = p2_group(M, K);
    const CUtensorMap* ma = p.kpack == 1 ? get_map(cache, A, M, K, lda, BM) : get_map3(cache, A, M, K, lda, BM, p.kpack);
    if (!ma) return cudaErrorInvalidValue;
    if (nseg == 1) {
      // split tail: rem tail tiles split S >= 2 ways with rem * S <= ncl, so at
      // most ncl partial tiles and ncl / 2 counted tiles
      if (!cache->tail_ws) {
        const size_t slots = (size_t)std::max(1, nsm / 2);
        cudaError_t e = cudaMalloc(&cache->tail_ws, slots * 2 * BM * 256 * sizeof(float));
        if (e == cudaSuccess) e = cudaMalloc(&cache->tail_cnt, slots * 8 * 32 * sizeof(int));
        if (e == cudaSuccess) e = cudaMemsetAsync(cache->tail_cnt, 0, slots * 8 * 32 * sizeof(int), st);
        if (e != cudaSuccess) return e;
      }
      if (ncl <= std::max(1, nsm / 2)) {
        p.tail_ws = cache->tail_ws;
        p.tail_cnt = cache->tail_cnt;
      }
    }
    return launch_p2(ma, mb, p, ncl, st);
  }
  if (kind != 1 && kind != 2) return cudaErrorInvalidValue;
  if (kind == 2) {
    if (M > 2 * BM) return cudaErrorInvalidValue;
    p.np = std::max(16, (M + 15) & ~15);
    p.tmem_cols = 32;
    while (p.tmem_cols < p.np) p.tmem_cols *= 2;
    int splits = auto_splits ? auto_splits : 1;
    if (force && force->splits) {
      splits = force->splits;
    } else if (!auto_splits) {
      while (splits < 8 && tiles * splits * 2 <= nsm && ktiles >= splits * 2 * 8) splits *= 2;
    }
    int stages = force && force->stages ? force->stages : (auto_stages ? auto_stages : ws_stages_for(p.np, 1, splits));
    if (splits < 1 || splits > 8 || stages < 2 || stages > WS_MAX_STAGES ||
        ws_smem_bytes(p.np, stages) > 232448 ||
        (splits > 1 && stages * ws_stage_bytes(p.np) < p.np * RED_PITCH * 4))
      return cudaErrorInvalidValue;
    p.splits = splits;
    p.stages = stages;
    p.nload = loaders_for(stages);
    const CUtensorMap* ma = get_map(cache, A, M, K, lda, p.np);
    if (!ma) return cudaErrorInvalidValue;
    return launch_ws(ma, mb, p, dim3(tiles, 1, splits), st);
  }
  // row-tiled kernel
  int splits = auto_splits ? auto_splits : 1;
  if (force && force->splits) splits = force->splits;
  if (splits < 1 || splits > 8) return cudaErrorInvalidValue;
  p.bn = bn;
  p.splits = splits;
  // k-blocks per stage: 2 reads each operand with one 3D box per stage (whole
  // k-blocks of K only)
  p.kpack = force && force->kpack ? force->kpack : 1;
  if (p.kpack < 1 || p.kpack > 2 || (p.kpack > 1 && K % BK)) return cudaErrorInvalidValue;
  const int rt_max_st = std::min(RT_MAX_STAGES, (232448 - 2048) / (p.kpack * rt_stage_bytes(MT, bn)));
  p.stages = force && force->stages ? force->stages : rt_max_st;
  if (p.stages < 2 || p.stages > rt_max_st ||
      (splits > 1 && p.kpack * p.stages * rt_stage_bytes(MT, bn) < BM * (bn + 4) * 4))
    return cudaErrorInvalidValue;
  p.tmem_cols = 32;
  while (p.tmem_cols < MT * bn) p.tmem_cols *= 2;
  p.nload = loaders_for(p.stages);
  if (p.kpack > 1)
    for (int sgi = 0; sgi < nseg; ++sgi) {
      mb[sgi] = get_map3(cache, W[sgi], N[sgi], K, ldw[sgi], bn, p.kpack);
      if (!mb[sgi]) return cudaErrorInvalidValue;
    }
  for (int sgi = nseg; sgi < 3; ++sgi) mb[sgi] = mb[0];
  const CUtensorMap* ma = p.kpack > 1 ? get_map3(cache, A, M, K, lda, BM, p.kpack) : get_map(cache, A, M, K, lda, BM);
  if (!ma) return cudaErrorInvalidValue;
  const dim3 grid(tiles, mgroups, splits);
  return MT == 2 ? launch_rt<2>(ma, mb, p, grid, st) : launch_rt<1>(ma, mb, p, grid, st);
}

cudaError_t tc_gemm_bf16_swiglu(TcGemmCache* cache, const void* A, int lda, const void* Wg, const void* Wu, int ldw,
                                int F, void* act, int ld_act, int M, const int* m_dev, int K, cudaStream_t st,
                                const TcGemmChoice* force) {
  using namespace tc;
  if (M <= 0 || F <= 0) return cudaSuccess;
  if (!A || !Wg || !Wu || !act || ld_act < F || !tc_gemm_supported(K, lda, ldw)) return cudaErrorInvalidValue;
  if (((uintptr_t)A | (uintptr_t)Wg | (uintptr_t)Wu) & 15) return cudaErrorInvalidValue;
  int* err = tc_error_word(cache);
  if (!err) return cudaErrorMemoryAllocation;
  if (cache->num_sms <= 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&cache->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (cache->num_sms <= 0) return cudaErrorNoDevice;
  }
  const int nsm = cache->num_sms;
  const int MT = M > BM ? 2 : 1;
  const int mgroups = (M + MT * BM - 1) / (MT * BM);
  const int ktiles = (K + BK - 1) / BK;
  const int Ns[2] = {F, F};
  GemmPick pk{1, 0, 1, 0};
  if (force && force->kernel) {
    if (force->kernel != 1 && force->kernel != 5) return cudaErrorNotSupported;
    pk.kernel = force->kernel;
    pk.bn = force->bn;
    pk.splits = force->splits ? force->splits : (force->kernel == 5 ? 0 : 1);
    pk.stages = force->stages;
  } else {
    pk = pick_for(cache, M, Ns, 2, ktiles, nsm, K);
    // the row-tiled and the two-SM pair kernels fuse the activation
    if (pk.kernel != 1 && pk.kernel != 5) return cudaErrorNotSupported;
  }
  if (pk.kernel == 5) {
    // two-SM pair tiles in SwiGLU mode: rank 0 of a pair reads gate rows, rank
    // 1 up rows of the same bn/2 output columns, so the M = 256 accumulator
    // holds both and the epilogue writes the bf16 activation
    Params p{};
    p.M = M;
    p.K = K;
    p.m_dev = m_dev;
    p.ldc = 0;
    p.ktiles = ktiles;
    p.err = err;
    p.nseg = 2;
    p.seg_start[0] = 0;
    p.seg_start[1] = p.seg_start[2] = p.seg_start[3] = 0x3FFFFFFF;
    p.seg_N[0] = p.seg_N[1] = F;
    p.act = (__nv_bfloat16*)act;
    p.ld_act = ld_act;
    p.bn = pk.bn ? pk.bn : 256;
    if (p.bn < 32 || p.bn > 256 || (p.bn & 31)) return cudaErrorInvalidValue;
    p.kpack = pk.splits ? pk.splits : 1;
    if (p.kpack < 1 || p.kpack > 2 || (p.kpack > 1 && K % BK)) return cudaErrorInvalidValue;
    const int max_stages = p2_max_stages(p.bn, p.kpack);
    p.stages = pk.stages ? pk.stages : (p.kpack == 1 ? p2_default_stages(p.bn) : max_stages);
    if (p.stages < 2 || p.stages > max_stages) return cudaErrorInvalidValue;
    p.splits = 1;
    p.nload = loaders_for(p.stages);
    p.tmem_cols = 32;
    while (p.tmem_cols < 2 * p.bn) p.tmem_cols *= 2;
    p.ntn = (F + p.bn / 2 - 1) / (p.bn / 2);
    const CUtensorMap* mb[3];
    mb[0] = p.kpack == 1 ? get_map(cache, Wg, F, K, ldw, p.bn / 2) : get_map3(cache, Wg, F, K, ldw, p.bn / 2, p.kpack);
    mb[1] = p.kpack == 1 ? get_map(cache, Wu, F, K, ldw, p.bn / 2) : get_map3(cache, Wu, F, K, ldw, p.bn / 2, p.kpack);
    mb[2] = mb[0];
    const CUtensorMap* ma = p.kpack == 1 ? get_map(cache, A, M, K, lda, BM) : get_map3(cache, A, M, K, lda, BM, p.kpack);
    if (!mb[0] || !mb[1] || !ma) return cudaErrorInvalidValue;
    const long long pair_tiles = (long long)((M + 2 * BM - 1) / (2 * BM)) * p.ntn;
    const int ncl = p2_clusters(p.bn, p.stages, pair_tiles, nsm);
    p.group = p2_group(M, K);
    return launch_p2(ma, mb, p, ncl, st);
  }
  const int bn = pk.bn ? pk.bn : (mgroups == 1 ? pick_for(cache, M, Ns, 2, ktiles, nsm, K).bn : 256);
  if (bn < 16 || bn > 256 || (bn & 15) || MT * bn > 512) return cudaErrorInvalidValue;
  Params p{};
  p.M = M;
  p.K = K;
  p.m_dev = m_dev;
  p.ldc = 0;
  p.ktiles = ktiles;
  p.err = err;
  p.nseg = 2;
  p.seg_start[0] = 0;
  p.seg_start[1] = p.seg_start[2] = p.seg_start[3] = 0x3FFFFFFF;
  p.seg_N[0] = p.seg_N[1] = F;
  p.act = (__nv_bfloat16*)act;
  p.ld_act = ld_act;
  p.bn = bn;
  p.splits = pk.splits;
  p.stages = pk.stages ? pk.stages : rt_max_stages(MT, bn);
  if (p.splits < 1 || p.splits > 8 || p.stages < 2 || p.stages > RT_MAX_STAGES ||
      rt_smem_bytes(MT, bn, p.stages) > 232448 ||
      (p.splits > 1 && p.stages * rt_stage_bytes(MT, bn) < BM * (bn + 4) * 4))
    return cudaErrorInvalidValue;
  p.tmem_cols = 32;
  while (p.tmem_cols < MT * bn) p.tmem_cols *= 2;
  p.nload = loaders_for(p.stages);
  const CUtensorMap* mb[3];
  mb[0] = get_map(cache, Wg, F, K, ldw, bn / 2);
  mb[1] = get_map(cache, Wu, F, K, ldw, bn / 2);
  mb[2] = mb[0];
  const CUtensorMap* ma = get_map(cache, A, M, K, lda, BM);
  if (!mb[0] || !mb[1] || !ma) return cudaErrorInvalidValue;
  const dim3 grid((F + bn / 2 - 1) / (bn / 2), mgroups, p.splits);
  return MT == 2 ? launch_rt<2>(ma, mb, p, grid, st) : launch_rt<1>(ma, mb, p, grid, st);
}

cudaError_t tc_gemm_bf16_qkv_rope(TcGemmCache* cache, const void* A, int lda, const void* const* W, const int* N,
                                  int M, int K, const TcQkvRope& q, cudaStream_t st) {
  using namespace tc;
  if (M <= 0) return cudaSuccess;
  if (!A || !q.rows || !q.rope || !q.q_out || !q.kv_layer || !tc_gemm_supported(K, lda, K)) return cudaErrorInvalidValue;
  if (((uintptr_t)A | (uintptr_t)q.q_out | (uintptr_t)q.kv_layer) & 15) return cudaErrorInvalidValue;
  // tiles of whole heads (256 columns), rotary pairs in 16-column chunks
  constexpr int PBN = 256;
  if (q.dh < 32 || q.dh % 32 || PBN % q.dh || q.kvdim % 8 || N[1] != q.kvdim || N[2] != q.kvdim) return cudaErrorNotSupported;
  for (int sgi = 0; sgi < 3; ++sgi)
    if (N[sgi] % PBN || ((uintptr_t)W[sgi] & 15)) return cudaErrorNotSupported;
  int* err = tc_error_word(cache);
  if (!err) return cudaErrorMemoryAllocation;
  if (cache->num_sms <= 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&cache->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (cache->num_sms <= 0) return cudaErrorNoDevice;
  }
  const int nsm = cache->num_sms;
  const int ktiles = (K + BK - 1) / BK;
  const GemmPick pk = pick_for(cache, M, N, 3, ktiles, nsm, K);
  if (pk.kernel != 5) return cudaErrorNotSupported;  // the pair kernel carries the mode
  Params p{};
  p.M = M;
  p.K = K;
  p.m_dev = nullptr;
  p.ldc = 0;
  p.ktiles = ktiles;
  p.err = err;
  p.nseg = 3;
  p.bn = PBN;
  p.kpack = (ktiles * BK == K) ? 2 : 1;
  p.stages = p.kpack == 1 ? p2_default_stages(p.bn) : p2_max_stages(p.bn, p.kpack);
  p.splits = 1;
  p.nload = loaders_for(p.stages);
  p.tmem_cols = 512;
  const CUtensorMap* mb[3];
  for (int sgi = 0, t = 0; sgi < 3; ++sgi) {
    p.seg_start[sgi] = t;
    p.seg_N[sgi] = N[sgi];
    p.seg_C[sgi] = nullptr;
    mb[sgi] = p.kpack == 1 ? get_map(cache, W[sgi], N[sgi], K, K, p.bn / 2)
                           : get_map3(cache, W[sgi], N[sgi], K, K, p.bn / 2, p.kpack);
    if (!mb[sgi]) return cudaErrorInvalidValue;
    t += N[sgi] / p.bn;
  }
  p.seg_start[3] = 0x3FFFFFFF;
  p.ntn = (N[0] + N[1] + N[2]) / p.bn;
  p.q_out = (__nv_bfloat16*)q.q_out;
  p.qkv_rows = q.rows;
  p.qkv_write_kv = q.write_kv;
  p.rope = q.rope;
  p.kv_layer = (__nv_bfloat16*)q.kv_layer;
  p.kv_seq_stride = (long long)q.kv_seq_stride;
  p.kvdim = q.kvdim;
  p.dh = q.dh;
  const long long pair_tiles = (long long)((M + 2 * BM - 1) / (2 * BM)) * p.ntn;
  const int ncl = p2_clusters(p.bn, p.stages, pair_tiles, nsm);
  p.group = p2_group(M, K);
  const CUtensorMap* ma = p.kpack == 1 ? get_map(cache, A, M, K, lda, BM) : get_map3(cache, A, M, K, lda, BM, p.kpack);
  if (!ma) return cudaErrorInvalidValue;
  return launch_p2(ma, mb, p, ncl, st);
}

cudaError_t tc_gemm_bf16(TcGemmCache* cache, const void* A, int lda, const void* W, int ldw, float* C, int ldc,
                         int M, const int* m_dev, int N, int K, cudaStream_t st, const TcGemmChoice* force) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  return tc_gemm_bf16_multi(cache, A, lda, 1, &W, &ldw, &N, &C, ldc, M, m_dev, K, st, force);
}

cudaError_t tc_gemm_choice(TcGemmCache* cache, int M, int nseg, const int* N, int K, int* out) {
  using namespace tc;
  if (M <= 0 || nseg < 1 || nseg > 3 || K < 1 || !out) return cudaErrorInvalidValue;
  if (cache->num_sms <= 0) {
    int dev = 0;
    cache->num_sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&cache->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cache->num_sms <= 0) {
      cache->num_sms = 0;
      cudaGetLastError();
      return cudaErrorNoDevice;
    }
  }
  const int ktiles = (K + BK - 1) / BK;
  const GemmPick pk = tc::pick_for(cache, M, N, nseg, ktiles, cache->num_sms, K);
  out[0] = pk.kernel;
  out[1] = pk.bn;
  out[2] = pk.splits;
  out[3] = pk.stages;
  return cudaSuccess;
}

cudaError_t tc_gemm_reset_after_timeout(TcGemmCache* c, cudaStream_t st) {
  if (!c->tail_cnt) return cudaSuccess;
  const size_t slots = (size_t)std::max(1, c->num_sms / 2);
  return cudaMemsetAsync(c->tail_cnt, 0, slots * 8 * 32 * sizeof(int), st);
}

void tc_gemm_cache_clear(TcGemmCache* c) {
  c->maps.clear();
  if (c->err) cudaFree(c->err);
  c->err = nullptr;
  if (c->tail_ws) cudaFree(c->tail_ws);
  if (c->tail_cnt) cudaFree(c->tail_cnt);
  c->tail_ws = nullptr;
  c->tail_cnt = nullptr;
}

}  // namespace polestar
