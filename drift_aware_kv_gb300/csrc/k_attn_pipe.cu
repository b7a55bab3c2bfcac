// bf16 row attention + KL drift on the tensor cores, pipelined per warp.
//
// Same computation as the rest of the row-attention family (Eq. 3 attention
// over all N keys of the row's sequence; Eq. 4 KL drift against the previous
// scores for tracked rows, in the cancellation-free form
//   KL = sum_j p_j d_j - log1p( sum_j q~_j expm1(d_j) / sum_j q~_j ) ),
// organised for small row counts and long key ranges alike:
//
//   * CTA = one work item (up to 48 rows of ONE sequence, given as at most two
//     row ranges: pieces of the sequence's active block and of its window +
//     proxy rows) x one query head x one key range.  Warps 0..2 compute 16 rows
//     each, warp 3 loads; two CTAs share an SM.
//   * The loader warp streams 64-key K/V tiles with TMA (128-byte swizzled
//     boxes of the [batch*N, 2*kvdim] cache view) into a ring of shared-memory
//     stages guarded by mbarriers: a compute warp waits only for the tile it
//     needs and releases it when done, so warps never wait for each other.
//   * S = Q K^T and O += P V run on mma.sync m16n8k16 (fp32 accumulation) with
//     ldmatrix reads that undo the swizzle; online softmax in log2 units.
//   * Rows under drift tracking either compute their KL terms here (they fetch
//     their previous scores for the tile with cp.async into a per-warp
//     shared-memory tile when the tile starts, so the fetch overlaps the wait
//     for K/V and the S = Q K^T products), or, in deferred mode (the layer
//     loop), only write their new scores and log-sum-exp for the drift pass.
//   * Key ranges of one (item, head) form a thread-block cluster; their partial
//     results meet in distributed shared memory and every CTA of the cluster
//     finishes a slice of the rows (ranks in fixed order: deterministic).  No
//     global workspace and no second kernel.
// Every mbarrier wait is bounded; a timeout records an error code, abandons the
// remaining tiles and still reaches the cluster barriers.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"

namespace polestar {
namespace ap {

constexpr int TK = 64;            // keys per tile
constexpr int CW = ATT_ITEM_ROWS / 16;  // compute warps, 16 rows each
constexpr int THREADS = (CW + 1) * 32;
constexpr int MAX_STAGES = 4;
constexpr long long TIMEOUT_CYCLES = 4000000000LL;  // ~2 s

template <int DH>
__host__ __device__ constexpr int tile_bytes() {
  return 2 * TK * DH * 2;  // K + V, bf16
}
constexpr int PREV_PITCH = 72;   // floats per row of a warp's previous-score tile (spreads banks)
// Per-row partials of a key range: max (log2 units), sum, KL numerator,
// q-mass, expm1 sum, then DH outputs; the pitch keeps rows 16-byte aligned and
// holds a previous-score row, which shares the space during the tile loop.
template <int DH>
__host__ __device__ constexpr int part_pitch() {
  return ((5 + DH + 3) / 4) * 4 < PREV_PITCH ? PREV_PITCH : ((5 + DH + 3) / 4) * 4;
}
// aligned ring | barriers, abort flag, previous-score row pointers | partials
// (key splits) or per-warp previous-score tiles
template <int DH>
__host__ __device__ constexpr int smem_bytes(int stages, bool split) {
  return 1024 + stages * tile_bytes<DH>() + 1024 +
         (split ? ATT_ITEM_ROWS * part_pitch<DH>() * 4 : CW * 16 * PREV_PITCH * 4);
}

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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
// Bounded wait; on timeout records `code` and raises the CTA's abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err, int code,
                                          volatile int* abort_flag) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > TIMEOUT_CYCLES) {
      if (err) atomicExch(err, code);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}
// One K/V tile of a head in a single copy: the 4D view {64 columns, row,
// 64-column block within the K (or V) half, K/V} of the cache (see kv_map4)
// lands as [K/V][block][row][64] swizzled boxes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4a(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4a_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// e^x - 1 for the KL drift term.  For |x| < 1/8 the Taylor series of e^x - 1
// through x^6 (the remainder is below |x| 8e-10); elsewhere 2^(x log2 e) - 1,
// where |e^x - 1| > 0.11 so the subtraction costs at most a few bits.
__device__ __forceinline__ float expm1_drift(float x) {
  float t = fmaf(x, 1.f / 720.f, 1.f / 120.f);
  t = fmaf(x, t, 1.f / 24.f);
  t = fmaf(x, t, 1.f / 6.f);
  t = fmaf(x, t, 0.5f);
  t = fmaf(x, t, 1.f);
  const float big = ex2f(x * 1.4426950408889634f) - 1.f;
  return fabsf(x) < 0.125f ? x * t : big;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *(const uint32_t*)&v;
}
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_remote(const float* local, uint32_t rank) {
  uint32_t a = su32(local), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// Shared-memory byte address of element (row, col) of one K or V tile (TK rows
// of DH bf16 as DH/64 boxes of TK x 64, 128-byte swizzle: 16-byte chunk c of
// row r at chunk c ^ (r & 7)); col is a multiple of 8.
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int col) {
  const int box = col >> 6, chunk = (col & 63) >> 3;
  return base + box * (TK * 128) + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// row of the step row space behind local row lr of a work item
__device__ __forceinline__ int item_row(const int4& wk, int lr) { return lr < wk.y ? wk.x + lr : wk.z + (lr - wk.y); }

template <int DH>
__global__ void __launch_bounds__(THREADS, 2) attn_pipe_kernel(const __grid_constant__ CUtensorMap tm_kv, AttnArgs p) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  constexpr int TB = tile_bytes<DH>();
  constexpr int PF = part_pitch<DH>();
  const int STAGES = p.stages;
  uint64_t* full = (uint64_t*)(sm + STAGES * TB);
  uint64_t* empty = full + MAX_STAGES;
  volatile int* abort_flag = (volatile int*)(empty + MAX_STAGES);
  const float** ptab_all = (const float**)(sm + STAGES * TB + 128);  // [CW][16] previous-score rows
  float* part = (float*)(sm + STAGES * TB + 1024);  // [ATT_ITEM_ROWS][PF] with key splits

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int split = blockIdx.z, nsplit = gridDim.z;
  const int kvh = h / (p.H / p.Hkv);
  const int ntiles_all = (p.N + TK - 1) / TK;
  const int tbeg = split * ntiles_all / nsplit, tend = (split + 1) * ntiles_all / nsplit;
  const int ntl = tend - tbeg;
  // K/V rows, queries and (for callers that build them on the device) the work
  // list and row table come from the preceding kernels: nothing of them is read
  // before the dependency wait
  pdl_launch_dependents();
  pdl_wait();
  const int4 wk = p.work[blockIdx.x];  // {rowA, nA, rowB, nB}
  const int nrows = wk.y + wk.w;
  const int nwl = (nrows + 15) >> 4;   // compute warps with rows

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(su32(&full[s]), 1);
      mbar_init(su32(&empty[s]), nwl);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  const int seq = p.rows[wk.x].x;

  if (warp == CW) {
    // ---------------- loader: K then V boxes of each tile
    if (lane == 0) {
      for (int i = 0; i < ntl; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES && !mbar_wait(su32(&empty[s]), ((i / STAGES) - 1) & 1, p.err, 11, abort_flag)) break;
        const uint32_t fb = su32(&full[s]);
        mbar_expect_tx(fb, TB);
        const uint32_t dst = su32(sm + s * TB);
        const int y = seq * p.N + (tbeg + i) * TK;
        tma_load_4d(dst, &tm_kv, 0, y, kvh * (DH / 64), 0, fb);  // K then V, DH/64 boxes each
      }
    }
  } else if (warp < nwl) {
    // ---------------- compute warp: rows 16*warp .. 16*warp+15 of the item
    const int qr = lane >> 2, qc = lane & 3;  // fragment row / column group
    const int rl0 = warp * 16 + qr, rl1 = rl0 + 8;
    int rows[2];
    bool live[2], outp[2];
    float* prev[2] = {nullptr, nullptr};
    float* prev_lse[2] = {nullptr, nullptr};
    // where a tracked row's new scores / log-sum-exp go: the deferred-drift
    // buffers when the drift pass measures it, else over the previous ones
    float* sdst[2] = {nullptr, nullptr};
    float* ldst[2] = {nullptr, nullptr};
    float shift[2] = {0.f, 0.f};
    const bool deferred = p.measure && (p.proxy_new != nullptr || p.active_new != nullptr);
    const bool inl = p.measure && !deferred;  // KL terms computed here
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int rl = i ? rl1 : rl0;
      rows[i] = rl < nrows ? item_row(wk, rl) : item_row(wk, 0);
      int4 m = make_int4(0, 0, ROW_NONE, 0);
      if (rl < nrows) m = p.rows[rows[i]];
      live[i] = m.z != ROW_NONE && (m.z != ROW_OTHER || p.other_live);
      outp[i] = live[i] && m.z != ROW_PROXY;
      if (live[i] && m.z == ROW_PROXY && p.proxy_prev) {
        const size_t idx = ((size_t)seq * p.K + m.w) * p.H + h;
        prev[i] = p.proxy_prev + idx * p.N;
        prev_lse[i] = p.proxy_prev_lse + idx;
        sdst[i] = deferred ? p.proxy_new + idx * p.N : prev[i];
        ldst[i] = deferred ? p.proxy_new_lse + idx : prev_lse[i];
      } else if (live[i] && m.z == ROW_ACTIVE && p.active_prev) {
        const size_t idx = ((size_t)seq * p.B + m.w) * p.H + h;
        prev[i] = p.active_prev + idx * p.N;
        prev_lse[i] = p.active_prev_lse + idx;
        sdst[i] = deferred ? p.active_new + idx * p.N : prev[i];
        ldst[i] = deferred ? p.active_new_lse + idx : prev_lse[i];
      }
      if (prev[i] && inl) shift[i] = *prev_lse[i] * 1.4426950408889634f;  // log2 units
    }
    const bool put = p.store || deferred;  // tracked rows write their scores
    const bool warp_tracked = __any_sync(0xffffffffu, prev[0] != nullptr || prev[1] != nullptr);
    // previous scores of this warp's tracked rows come in per tile through
    // shared memory: row pointers (null = not tracked) and the tile buffer
    const float** ptab = ptab_all + warp * 16;
    float* pbuf = part + warp * 16 * (nsplit > 1 ? PF : PREV_PITCH);
    const bool fetch = warp_tracked && inl;
    const bool vec = (p.N & 3) == 0 && (((uintptr_t)p.active_prev | (uintptr_t)p.proxy_prev) & 15) == 0;
    if (fetch) {
      if (qc == 0) {
        ptab[qr] = prev[0];
        ptab[qr + 8] = prev[1];
      }
      __syncwarp();
    }

    // Q fragments (A operand) straight from global memory
    constexpr int KT = DH / 16;
    uint32_t qa[KT][4];
    {
      const __nv_bfloat16* q0 = (const __nv_bfloat16*)p.q + (size_t)rows[0] * p.ldq + h * DH;
      const __nv_bfloat16* q1 = (const __nv_bfloat16*)p.q + (size_t)rows[1] * p.ldq + h * DH;
#pragma unroll
      for (int kt = 0; kt < KT; ++kt) {
        const int c = kt * 16 + qc * 2;
        qa[kt][0] = live[0] ? *(const uint32_t*)(q0 + c) : 0u;
        qa[kt][1] = live[1] ? *(const uint32_t*)(q1 + c) : 0u;
        qa[kt][2] = live[0] ? *(const uint32_t*)(q0 + c + 8) : 0u;
        qa[kt][3] = live[1] ? *(const uint32_t*)(q1 + c + 8) : 0u;
      }
    }

    constexpr int NT = DH / 8;  // output n-tiles
    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float mrun[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
    float asum[2] = {0.f, 0.f}, sqs[2] = {0.f, 0.f}, esum[2] = {0.f, 0.f};
    const float sl2 = p.scale * 1.4426950408889634f;
    const int mi = lane >> 3, ri = lane & 7;

    for (int i = 0; i < ntl; ++i) {
      const int s = i % STAGES;
      const int j0 = (tbeg + i) * TK;
      if (fetch) {
        // this tile's previous scores: 16 rows x 64 keys
        if (vec) {
          const int c = (lane & 15) * 4;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int r = (lane >> 4) + 2 * k;
            const float* src = ptab[r];
            if (src && j0 + c < p.N) cp_async16(su32(pbuf + r * PREV_PITCH + c), src + j0 + c);
          }
        } else {
          for (int r = 0; r < 16; ++r) {
            const float* src = ptab[r];
            if (!src) continue;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int c = hh * 32 + lane;
              if (j0 + c < p.N) cp_async4(su32(pbuf + r * PREV_PITCH + c), src + j0 + c);
            }
          }
        }
        cp_async_commit();
      }
      if (!mbar_wait(su32(&full[s]), (i / STAGES) & 1, p.err, 12, abort_flag)) break;
      const uint32_t kb = su32(sm + s * TB), vb = kb + TB / 2;
      // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
      float sc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int kt = 0; kt < KT; kt += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4a(b0, b1, b2, b3, swz(kb, nt * 8 + ri, kt * 16 + (mi & 1) * 8 + (mi >> 1) * 16));
          mma16816(sc[nt], qa[kt], b0, b1);
          mma16816(sc[nt], qa[kt + 1], b2, b3);
        }
      }
      const bool fullt = (j0 + TK <= p.N);
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = sc[nt][e] * sl2;
          if (!fullt && j0 + nt * 8 + qc * 2 + (e & 1) >= p.N) v = -INFINITY;
          sc[nt][e] = v;
          tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
        }
      }
      if (fetch) {
        cp_async_wait_all();
        __syncwarp();
      }
      float corr[2];
#pragma unroll
      for (int ii = 0; ii < 2; ++ii) {
        tmax[ii] = fmaxf(tmax[ii], __shfl_xor_sync(0xffffffffu, tmax[ii], 1));
        tmax[ii] = fmaxf(tmax[ii], __shfl_xor_sync(0xffffffffu, tmax[ii], 2));
        const float mnew = fmaxf(mrun[ii], tmax[ii]);
        corr[ii] = ex2f(mrun[ii] - mnew);
        mrun[ii] = mnew;
        lsum[ii] *= corr[ii];
        asum[ii] *= corr[ii];
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        acc[nt][0] *= corr[0];
        acc[nt][1] *= corr[0];
        acc[nt][2] *= corr[1];
        acc[nt][3] *= corr[1];
      }
      uint32_t pa[4][4];  // P as A fragments: 4 k-steps of 16 keys
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pv[e] = ex2f(sc[nt][e] - mrun[e >> 1]);  // exp2(-inf) = 0 for masked keys
          lsum[e >> 1] += pv[e];
        }
        if (warp_tracked) {
          const int j = j0 + nt * 8 + qc * 2;
#pragma unroll
          for (int ii = 0; ii < 2; ++ii) {
            if (!prev[ii] || j >= p.N) continue;
            const float s0 = sc[nt][2 * ii] * 0.6931471805599453f, s1 = sc[nt][2 * ii + 1] * 0.6931471805599453f;
            if (inl) {
              // Eq. 4 terms against the previous scores sp (natural-log units):
              // d = s - sp, q~ = exp(sp - lse_prev)
              const float2 sp = *(const float2*)(pbuf + (qr + 8 * ii) * PREV_PITCH + nt * 8 + qc * 2);
              const float d0 = s0 - sp.x, q0 = ex2f(fmaf(sp.x, 1.4426950408889634f, -shift[ii]));
              asum[ii] = fmaf(pv[2 * ii], d0, asum[ii]);
              sqs[ii] += q0;
              esum[ii] = fmaf(q0, expm1_drift(d0), esum[ii]);
              if (j + 1 < p.N) {
                const float d1 = s1 - sp.y, q1 = ex2f(fmaf(sp.y, 1.4426950408889634f, -shift[ii]));
                asum[ii] = fmaf(pv[2 * ii + 1], d1, asum[ii]);
                sqs[ii] += q1;
                esum[ii] = fmaf(q1, expm1_drift(d1), esum[ii]);
              }
            }
            if (put) {
              float* dst = sdst[ii] + j;
              if (j + 1 < p.N && (((uintptr_t)dst) & 7) == 0) {
                *(float2*)dst = make_float2(s0, s1);
              } else {
                dst[0] = s0;
                if (j + 1 < p.N) dst[1] = s1;
              }
            }
          }
        }
        const int kt = nt >> 1;
        if ((nt & 1) == 0) {
          pa[kt][0] = pack2(pv[0], pv[1]);
          pa[kt][1] = pack2(pv[2], pv[3]);
        } else {
          pa[kt][2] = pack2(pv[0], pv[1]);
          pa[kt][3] = pack2(pv[2], pv[3]);
        }
      }
      // O += P V
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4a_t(b0, b1, b2, b3, swz(vb, kt * 16 + (mi & 1) * 8 + ri, (nt + (mi >> 1)) * 8));
          mma16816(acc[nt], pa[kt], b0, b1);
          mma16816(acc[nt + 1], pa[kt], b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(su32(&empty[s]));
    }
    // row sums across the 4 threads sharing a row
#pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        lsum[ii] += __shfl_xor_sync(0xffffffffu, lsum[ii], o);
        asum[ii] += __shfl_xor_sync(0xffffffffu, asum[ii], o);
        sqs[ii] += __shfl_xor_sync(0xffffffffu, sqs[ii], o);
        esum[ii] += __shfl_xor_sync(0xffffffffu, esum[ii], o);
      }
    }
    if (nsplit > 1) {
      // this key range's partial results, finished below by the cluster
#pragma unroll
      for (int ii = 0; ii < 2; ++ii) {
        const int rl = ii ? rl1 : rl0;
        if (rl >= nrows) continue;
        float* pp = part + (size_t)rl * PF;
        if (qc == 0) {
          pp[0] = mrun[ii];
          pp[1] = lsum[ii];
          pp[2] = asum[ii];
          pp[3] = sqs[ii];
          pp[4] = esum[ii];
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          pp[5 + nt * 8 + qc * 2] = acc[nt][2 * ii];
          pp[5 + nt * 8 + qc * 2 + 1] = acc[nt][2 * ii + 1];
        }
      }
    } else {
#pragma unroll
      for (int ii = 0; ii < 2; ++ii) {
        if (outp[ii]) {
          __nv_bfloat16* o = (__nv_bfloat16*)p.out + (size_t)rows[ii] * p.ldo + h * DH;
          const float inv = 1.f / lsum[ii];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            *(uint32_t*)(o + nt * 8 + qc * 2) = pack2(acc[nt][2 * ii] * inv, acc[nt][2 * ii + 1] * inv);
        }
        if (prev[ii] && qc == 0) {
          if (inl)
            p.kl_out[(size_t)rows[ii] * p.H + h] =
                asum[ii] / lsum[ii] - kl_log_mass(esum[ii] / sqs[ii], mrun[ii] * 0.6931471805599453f + logf(lsum[ii]),
                                                  shift[ii] * 0.6931471805599453f);
          if (put) *ldst[ii] = mrun[ii] * 0.6931471805599453f + logf(lsum[ii]);
        }
      }
    }
  }

  if (nsplit > 1) {
    // ---------------- cluster combine: CTA `rank` finishes rows [r0, r1) of the
    // item from every key range's partials (ranks in order)
    cl_sync();
    const int rank = (int)cl_rank();
    const int r0 = rank * nrows / nsplit, r1 = (rank + 1) * nrows / nsplit;
    constexpr int NV = DH / 32;
    for (int rl = r0 + warp; rl < r1; rl += CW + 1) {
      const int r = item_row(wk, rl);
      const int4 m = p.rows[r];
      if (m.z == ROW_NONE || (m.z == ROW_OTHER && !p.other_live)) continue;
      const float* base = part + (size_t)rl * PF;
      float M = -INFINITY;
      for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ld_remote(base, (uint32_t)s));
      float l = 0.f, a = 0.f, sq = 0.f, e = 0.f;
      float acc[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) acc[i] = 0.f;
      for (int s = 0; s < nsplit; ++s) {
        const float w = ex2f(ld_remote(base, (uint32_t)s) - M);  // partial maxima are in log2 units
        l += ld_remote(base + 1, (uint32_t)s) * w;
        a += ld_remote(base + 2, (uint32_t)s) * w;
        sq += ld_remote(base + 3, (uint32_t)s);
        e += ld_remote(base + 4, (uint32_t)s);
#pragma unroll
        for (int i = 0; i < NV; ++i) acc[i] += ld_remote(base + 5 + lane + 32 * i, (uint32_t)s) * w;
      }
      if (m.z != ROW_PROXY) {
        __nv_bfloat16* o = (__nv_bfloat16*)p.out + (size_t)r * p.ldo + h * DH;
        const float inv = 1.f / l;
#pragma unroll
        for (int i = 0; i < NV; ++i) o[lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
      }
      const bool deferred = p.measure && (p.proxy_new != nullptr || p.active_new != nullptr);
      float* prev_lse = nullptr;
      float* lse_dst = nullptr;
      if (m.z == ROW_PROXY && p.proxy_prev) {
        const size_t idx = ((size_t)seq * p.K + m.w) * p.H + h;
        prev_lse = p.proxy_prev_lse + idx;
        lse_dst = deferred ? p.proxy_new_lse + idx : prev_lse;
      } else if (m.z == ROW_ACTIVE && p.active_prev) {
        const size_t idx = ((size_t)seq * p.B + m.w) * p.H + h;
        prev_lse = p.active_prev_lse + idx;
        lse_dst = deferred ? p.active_new_lse + idx : prev_lse;
      }
      if (prev_lse && lane == 0) {
        if (p.measure && !deferred)
          p.kl_out[(size_t)r * p.H + h] = a / l - kl_log_mass(e / sq, M * 0.6931471805599453f + logf(l), *prev_lse);
        if (p.store || deferred) *lse_dst = M * 0.6931471805599453f + logf(l);
      }
    }
    cl_sync();  // no CTA leaves while another still reads its partials
  }
  if (*abort_flag && warp == CW && lane == 0) {
    // let in-flight bulk copies land before the CTA's shared memory is released
    const long long t0 = clock64();
    while (clock64() - t0 < 20000000LL) {
    }
  }
}
// 4D tensor map of one layer's K/V cache ([batch*N rows][2 * kvdim] bf16, K
// then V of each row) viewed as {64 columns, row, 64-column block of the K or
// V half, K/V}: a box {64, TK, dh / 64, 2} at (0, row, head * dh / 64, 0) is one
// head's K and V for TK keys, as 128-byte-swizzled [TK][64] boxes in the order
// K block 0, K block 1, .., V block 0, ..  (cached per buffer and shape).
const CUtensorMap* kv_map(const void* base, int rows, int kvdim, int dh) {
  static std::map<std::tuple<const void*, int, int, int>, CUtensorMap> cache;
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_tuple(base, rows, kvdim, dh);
  auto it = cache.find(key);
  if (it != cache.end()) return &it->second;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  }
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  const cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)(kvdim / 64), 2};
  const cuuint64_t strides[3] = {(cuuint64_t)kvdim * 4, 128, (cuuint64_t)kvdim * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)TK, (cuuint32_t)(dh / 64), 2};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return nullptr;
  return &cache.emplace(key, m).first->second;
}

template <int DH>
cudaError_t launch(const AttnArgs& a, int batch, cudaStream_t st) {
  if (a.kvdim % 64) return cudaErrorInvalidValue;
  const CUtensorMap* map = kv_map(a.kv_layer, batch * a.N, a.kvdim, DH);
  if (!map) return cudaErrorInvalidValue;
  const bool split = a.splits > 1;
  const int smem = smem_bytes<DH>(a.stages, split);
  static PerDeviceOnce attr;
  {
    const cudaError_t e =
        func_attr_once(attr, (const void*)attn_pipe_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.n_work, a.H, a.splits);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = a.splits;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attn_pipe_kernel<DH>, *map, a);
}

}  // namespace ap

int attention_pipe_config(int n_work, int H, int N, int dh, int num_sms, int* stages) {
  const int tiles = (N + ap::TK - 1) / ap::TK;
  int s = 1;
  // key splits (at most 8, the portable cluster size) while the grid stays
  // within one wave of two CTAs per SM and every split keeps at least two tiles
  while (s < 8 && (long long)n_work * H * (s + 1) <= 2LL * num_sms && tiles >= 2 * (s + 1)) ++s;
  // ring depth: two CTAs per SM must fit in shared memory (a split also keeps
  // its partials there)
  const int per_cta = 233472 / 2 - 1024;
  int st = std::min(ap::MAX_STAGES, (tiles + s - 1) / s);
  while (st > 2 && (dh == 128 ? ap::smem_bytes<128>(st, s > 1) : ap::smem_bytes<64>(st, s > 1)) > per_cta) --st;
  *stages = std::max(2, st);
  return s;
}

cudaError_t launch_attention_pipe(const AttnArgs& a, int batch, cudaStream_t st) {
  if (a.dh == 128) return ap::launch<128>(a, batch, st);
  if (a.dh == 64) return ap::launch<64>(a, batch, st);
  return cudaErrorInvalidValue;
}

}  // namespace polestar
