// bf16 row attention on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators), for work items of up to 128 rows of one sequence.
//
// Same computation as the rest of the row-attention family (Eq. 3 attention
// over all N keys of the row's sequence), organised flash-attention style with
// every matrix product on tcgen05.  The KL drift of tracked rows (Eq. 4) is not
// computed here: a tracked row's scores and log-sum-exp are written out (to the
// deferred-drift buffers when the launch measures drift, which the drift pass
// then compares with the previous ones; over the previous ones when it only
// stores them), so the softmax threads do the same work for every row.
//
//   * CTA = one work item (<= 128 rows, given as at most two row ranges of one
//     sequence) x one query head; the item's Q rows are the MMA's M side
//     (TMEM lane = row); keys come in tiles of 64.  Two CTAs share an SM (256
//     TMEM columns and under half the shared memory each), so one SM runs
//     sixteen softmax warps.
//   * warp 0 streams K and V tiles with TMA (128-byte swizzled 64 x 64 boxes
//     of the [batch*N, 2*kvdim] cache view) into a two-stage ring whose K and
//     V halves have barriers of their own (K runs a tile ahead: K_j is free
//     once S_j is done, V_j only after P_j V_j);
//     warp 1 issues S_j = Q K_j^T into one of two TMEM score buffers and
//     O += P_{j-1} V_{j-1} into the TMEM output, taking P straight from TMEM
//     (the A operand), so the tensor cores compute tile j's scores while the
//     softmax warps work on tile j-1;
//   * warps 2-9 (a warp pair per TMEM lane quarter, each thread half of its
//     row's keys and output columns) read the row's scores from TMEM, keep the
//     running maximum (log2 units; the pair exchanges tile maxima through
//     shared memory) and sum, and write P (bf16 pairs) back over the first half
//     of the same score buffer; the running maximum is raised lazily (only when
//     a tile's maximum exceeds it by more than 8, i.e. p <= 2^8), and then the
//     TMEM output row is rescaled before the next P V;
//   * V is the second product's B operand read N-major (dh contiguous) from
//     the swizzled boxes, so no transposition is needed.
// Every mbarrier wait is bounded; a timeout records an error code and the
// CTA's roles fall through to the final barrier.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"

namespace polestar {
namespace at {

constexpr int ROWS = 128;   // rows per work item (MMA M)
constexpr int TK = 64;      // keys per tile (MMA N of S, K of P V)
constexpr int DH = 128;     // head dim
constexpr int SOFT_WARPS = 8;                 // two warps per TMEM lane quarter, each half of a tile's keys
constexpr int THREADS = (2 + SOFT_WARPS) * 32;
constexpr int STAGES = 2;
constexpr int QBOX = 64 * ROWS * 2;           // 64 columns x 128 rows (Q)
constexpr int KBOX = 64 * TK * 2;             // 64 columns x 64 keys (K, V)
constexpr int Q_OFF = 0;                      // 2 boxes (dh 0-63, 64-127)
constexpr int RING_OFF = 2 * QBOX;            // STAGES x (K: 2 boxes, V: 2 boxes)
constexpr int STAGE_BYTES = 4 * KBOX;
constexpr int O_COL = 2 * TK;                 // TMEM: S/P buffers at 0 and TK, O after
constexpr int TMEM_COLS = O_COL + DH;         // 256
constexpr int CTL_OFF = RING_OFF + STAGES * STAGE_BYTES;
constexpr int XCH_OFF = CTL_OFF + 256;          // [2 tile parities][2 halves][ROWS] partial maxima, then [2][ROWS] sums
constexpr int SMEM_BYTES = XCH_OFF + 6 * ROWS * 4 + 1024;  // + alignment
constexpr long long TIMEOUT_CYCLES = 4000000000LL;  // ~2 s
static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs per SM");

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
// UMMA shared-memory descriptor, 128-byte swizzle: K-major (lbo unused) or
// N-major (lbo = bytes between 64-element groups along N); sbo = bytes between
// 8-row groups.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// kind::f16, bf16 x bf16 -> fp32, M = 128, N = n; B N-major when bmn
__host__ __device__ constexpr uint32_t idesc(int n, bool bmn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((bmn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// D (TMEM) += A (TMEM, M = 128 lanes x K = 16 bf16 in 8 columns) * B (shared memory)
__device__ __forceinline__ void umma_ta(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 columns of a row without waiting (tcgen05_wait_ld() makes them usable)
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tcgen05_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st32_nw(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16_nw(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *(const uint32_t*)&v;
}
// byte offset of 16-byte chunk c (columns 8c..8c+7) of row r in a 128-row x
// 64-column swizzled box
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }
__device__ __forceinline__ int item_row(const int4& wk, int lr) { return lr < wk.y ? wk.x + lr : wk.z + (lr - wk.y); }

__global__ void __launch_bounds__(THREADS, 2) attn_tc_kernel(const __grid_constant__ CUtensorMap tm_kv, AttnArgs p) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  // K and V of a stage have barriers of their own: K_j is free once S_j is
  // done, long before P_j V_j has read V_j, so the next K tiles stream in while
  // the softmax still works on earlier tiles
  uint64_t* k_full = (uint64_t*)(sm + CTL_OFF);
  uint64_t* k_empty = k_full + STAGES;
  uint64_t* v_full = k_empty + STAGES;
  uint64_t* v_empty = v_full + STAGES;
  uint64_t* s_full = v_empty + STAGES;   // [2]
  uint64_t* p_full = s_full + 2;         // [2]
  uint64_t* pv_done = p_full + 2;        // [2]: P V of tiles j with j % 2 == b
  uint64_t* q_full = pv_done + 2;
  uint32_t* tmem_slot = (uint32_t*)(q_full + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int kvh = h / (p.H / p.Hkv);
  const int ntl = (p.N + TK - 1) / TK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(su32(&k_full[s]), 1);
      mbar_init(su32(&k_empty[s]), 1);
      mbar_init(su32(&v_full[s]), 1);
      mbar_init(su32(&v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(su32(&s_full[b]), 1);
      mbar_init(su32(&p_full[b]), SOFT_WARPS);
      mbar_init(su32(&pv_done[b]), 1);
    }
    mbar_init(su32(q_full), SOFT_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  // K/V rows, queries and (for callers that build them on the device) the work
  // list and row table come from the preceding kernels: read after the wait
  pdl_launch_dependents();
  pdl_wait();
  const int4 wk = p.work[blockIdx.x];  // {rowA, nA, rowB, nB}
  const int nrows = wk.y + wk.w;
  const int seq = p.rows[wk.x].x;

  if (warp == 0) {
    // ---------------- loader: K then V boxes of each 64-key tile
    if (lane == 0) {
      // K runs one tile ahead of V: K_{i+1}, then V_i
      auto load = [&](int j, int w) -> bool {
        const int s = j % STAGES;
        uint64_t* empty = w ? v_empty : k_empty;
        uint64_t* full = w ? v_full : k_full;
        if (j >= STAGES && !mbar_wait(su32(&empty[s]), ((j / STAGES) - 1) & 1, p.err, 21, abort_flag)) return false;
        mbar_expect_tx(su32(&full[s]), STAGE_BYTES / 2);
        const uint32_t dst = su32(sm + RING_OFF + s * STAGE_BYTES + w * (STAGE_BYTES / 2));
        tma_load_4d(dst, &tm_kv, 0, seq * p.N + j * TK, kvh * (DH / 64), w, su32(&full[s]));  // two 64-column boxes
        return true;
      };
      bool go = ntl > 0 && load(0, 0);
      for (int i = 0; i < ntl && go; ++i) {
        if (i + 1 < ntl) go = load(i + 1, 0);
        go = go && load(i, 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t q = su32(sm + Q_OFF);
      bool live = mbar_wait(su32(q_full), 0, p.err, 22, abort_flag);
      auto issue_pv = [&](int t) -> bool {
        if (!mbar_wait(su32(&p_full[t & 1]), (t >> 1) & 1, p.err, 23, abort_flag)) return false;
        if (!mbar_wait(su32(&v_full[t % STAGES]), (t / STAGES) & 1, p.err, 29, abort_flag)) return false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t v = su32(sm + RING_OFF + (t % STAGES) * STAGE_BYTES + 2 * KBOX);
        const uint32_t pt = tmem + (t & 1) * TK;  // P_t: bf16 pairs in the first TK/2 columns of S_t's buffer
#pragma unroll
        for (int kk = 0; kk < TK / 16; ++kk)
          umma_ta(tmem + O_COL, pt + kk * 8, sdesc(v + kk * 16 * 128, KBOX, 1024), idesc(DH, true),
                  (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit(su32(&pv_done[t & 1]));
        umma_commit(su32(&v_empty[t % STAGES]));
        return true;
      };
      for (int j = 0; j < ntl && live; ++j) {
        const int s = j % STAGES, b = j & 1;
        if (!mbar_wait(su32(&k_full[s]), (j / STAGES) & 1, p.err, 24, abort_flag)) break;
        // score buffer b holds P_{j-2} until P_{j-2} V_{j-2} has read it; that
        // product was issued before this one and the products run in order,
        // and the softmax has read S_{j-2} once it signalled P_{j-2}
        if (j >= 2 && !mbar_wait(su32(&p_full[b]), ((j - 2) >> 1) & 1, p.err, 25, abort_flag)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t kt = su32(sm + RING_OFF + s * STAGE_BYTES);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk)
          umma(tmem + b * TK, sdesc(q + (kk >> 2) * QBOX + (kk & 3) * 32, 16, 1024),
               sdesc(kt + (kk >> 2) * KBOX + (kk & 3) * 32, 16, 1024), idesc(TK, false), kk > 0 ? 1u : 0u);
        umma_commit(su32(&s_full[b]));
        umma_commit(su32(&k_empty[s]));
        if (j >= 1 && !issue_pv(j - 1)) live = false;
      }
      if (live && ntl > 0) issue_pv(ntl - 1);
    }
  } else {
    // ---------------- softmax / epilogue: row r = TMEM lane; the warp pair of
    // a lane quarter splits each tile's 64 keys (half = 0: keys 0-31, 1: 32-63)
    // and the output's 128 columns
    const int qd = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = qd * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
    float* xmax = (float*)(sm + XCH_OFF);  // [2][2][ROWS]
    float* xsum = xmax + 4 * ROWS;         // [2][ROWS]
    const uint32_t pair_bar = 1 + qd;      // named barrier of the warp pair (64 threads)
    const bool has = r < nrows;
    const int row = has ? item_row(wk, r) : item_row(wk, 0);
    int4 m = make_int4(0, 0, ROW_NONE, 0);
    if (has) m = p.rows[row];
    const bool live = m.z != ROW_NONE && (m.z != ROW_OTHER || p.other_live);
    const bool outp = live && m.z != ROW_PROXY;
    // tracked rows write their scores (natural-log units) and log-sum-exp: to
    // the deferred-drift buffers when the launch measures drift (the drift pass
    // compares them with the previous ones), else over the previous ones
    const bool defer = p.measure != 0;
    float* sdst = nullptr;
    float* ldst = nullptr;
    if (live && m.z == ROW_PROXY && p.proxy_prev) {
      const size_t idx = ((size_t)seq * p.K + m.w) * p.H + h;
      sdst = (defer ? p.proxy_new : p.proxy_prev) + idx * p.N;
      ldst = (defer ? p.proxy_new_lse : p.proxy_prev_lse) + idx;
    } else if (live && m.z == ROW_ACTIVE && p.active_prev) {
      const size_t idx = ((size_t)seq * p.B + m.w) * p.H + h;
      sdst = (defer ? p.active_new : p.active_prev) + idx * p.N;
      ldst = (defer ? p.active_new_lse : p.active_prev_lse) + idx;
    }
    if (!defer && !p.store) sdst = ldst = nullptr;
    const bool vec_sc = (p.N & 3) == 0 && (((uintptr_t)sdst) & 15) == 0;

    // 16-byte row accesses when the strides and bases allow them
    const bool vec_io = ((p.ldq | p.ldo) & 7) == 0 && ((((uintptr_t)p.q) | ((uintptr_t)p.out)) & 15) == 0;
    // this half's 64 Q columns of the row into the swizzled A-operand tile
    // (zeros for padding rows)
    {
      const __nv_bfloat16* qrow = (const __nv_bfloat16*)p.q + (size_t)row * p.ldq + h * DH;
#pragma unroll
      for (int cc = 0; cc < DH / 16; ++cc) {
        const int c = half * (DH / 16) + cc;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (live) {
          if (vec_io) {
            v = *(const uint4*)(qrow + c * 8);
          } else {
            uint16_t e[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) e[k] = ((const uint16_t*)qrow)[c * 8 + k];
            v = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16), e[4] | ((uint32_t)e[5] << 16),
                           e[6] | ((uint32_t)e[7] << 16));
          }
        }
        *(uint4*)(sm + Q_OFF + (c >> 3) * QBOX + swz(r, c & 7)) = v;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(su32(q_full));
    }

    const float sl2 = p.scale * 1.4426950408889634f;
    float mrun = -INFINITY, l = 0.f;
    bool ok = true;
    // a warp pair whose 32 rows all lie past the item's rows (items of fewer
    // than 128 rows) only keeps pace with the tiles: its lanes' P and O are
    // never read back, so it leaves the issue slots to the warps with rows
    const bool wdead = !__any_sync(0xffffffffu, has);
    for (int j = 0; j < ntl; ++j) {
      const int b = j & 1, j0 = j * TK + half * 32;
      // a failed wait anywhere is carried to the partner as a NaN maximum, and
      // the pair leaves together after the exchange (never alone: the pair's
      // named barrier would otherwise wait for a warp that left)
      ok = ok && mbar_wait(su32(&s_full[b]), (j >> 1) & 1, p.err, 26, abort_flag);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (wdead) {
        if (!ok) break;  // a dead pair exchanges nothing: each warp leaves on its own
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&p_full[b]));
        continue;
      }
      // this half's 32 scores of the row, pass 1: their maximum (raw scores,
      // keys past N at -inf) over eight independent chains
      uint32_t sv[32];
      float pmax = -INFINITY;
      if (ok) {
        tmem_ld32_nw(tl + b * TK + half * 32, sv);
        tcgen05_wait_ld();
        float mx8[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) mx8[c] = -INFINITY;
        if (j0 + 32 <= p.N) {
#pragma unroll
          for (int i = 0; i < 32; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sv[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (j0 + i >= p.N) sv[i] = __float_as_uint(-INFINITY);
            mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sv[i]));
          }
        }
        pmax = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                     fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      } else {
        pmax = __int_as_float(0x7fc00000);  // NaN: this warp gave up
      }
      xmax[(b * 2 + half) * ROWS + r] = pmax;
      asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
      const float omax = xmax[(b * 2 + (half ^ 1)) * ROWS + r];
      if (__any_sync(0xffffffffu, pmax != pmax || omax != omax)) {  // either warp gave up
        ok = false;
        break;
      }
      const float mx = sl2 * fmaxf(pmax, omax);  // log2 units; both halves compute the same value
      // raise the running maximum only when it grows by more than 8 (p <= 2^8)
      const bool raise = mx > mrun + 8.f;
      const float mnew = raise ? mx : mrun;
      const float corr = raise ? ex2f(mrun - mnew) : 1.f;  // exp2(-inf) = 0 on the first tile
      l *= corr;
      // a raised maximum rescales the output, which must then hold P_{j-1} V_{j-1};
      // each half rescales its 64 output columns
      const bool rescale = j >= 1 && __any_sync(0xffffffffu, raise);
      if (rescale) {
        const int t = j - 1;
        ok = mbar_wait(su32(&pv_done[t & 1]), (t >> 1) & 1, p.err, 27, abort_flag);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (ok) {
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t v[32];
            tmem_ld32_nw(tl + O_COL + half * 64 + c * 32, v);
            tcgen05_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * corr);
            tmem_st32_nw(tl + O_COL + half * 64 + c * 32, v);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
      }
      mrun = mnew;
      if (ok) {
        // pass 2: this half's probabilities as bf16 pairs (P, written over the
        // score buffer), the running sum over four chains, a tracked row's scores
        uint32_t pk[16];
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          float pv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            pv[e] = ex2f(fmaf(__uint_as_float(sv[g * 4 + e]), sl2, -mrun));  // exp2(-inf) = 0 past N
            l4[e] += pv[e];
          }
          pk[2 * g] = pack2(pv[0], pv[1]);
          pk[2 * g + 1] = pack2(pv[2], pv[3]);
          if (sdst) {
            const int jj = j0 + g * 4;
            float sn[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) sn[e] = __uint_as_float(sv[g * 4 + e]) * p.scale;
            if (vec_sc && jj + 3 < p.N) {
              *(float4*)(sdst + jj) = make_float4(sn[0], sn[1], sn[2], sn[3]);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (jj + e < p.N) sdst[jj + e] = sn[e];
            }
          }
        }
        l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        // keys 32 half .. 32 half + 31 as bf16 pairs: columns 16 half .. 16 half + 15
        // of the score buffer (this half's scores are all in registers by now; the
        // partner writes the other 16 columns from its own registers)
        tmem_st16_nw(tl + b * TK + half * 16, pk);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(su32(&p_full[b]));
      }
    }
    // ---------------- epilogue: O / l (each half its 64 columns), log-sum-exp
    if (ok && ntl > 0) {
      ok = mbar_wait(su32(&pv_done[(ntl - 1) & 1]), ((ntl - 1) >> 1) & 1, p.err, 28, abort_flag);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    }
    if (!wdead) {
      // the row's sum is the two halves' sums (same running maximum)
      xsum[half * ROWS + r] = ok ? l : __int_as_float(0x7fc00000);
      asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
      const float lo = xsum[(half ^ 1) * ROWS + r];
      if (lo != lo) ok = false;
      l += lo;
    }
    if (ok && !wdead) {
      const float inv = 1.f / l;
      __nv_bfloat16* o = (__nv_bfloat16*)p.out + (size_t)row * p.ldo + h * DH;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t ov[32];
        tmem_ld32_nw(tl + O_COL + half * 64 + c * 32, ov);
        tcgen05_wait_ld();
        if (outp) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t* v = ov + g * 8;
            const uint4 w = make_uint4(pack2(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                                       pack2(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                                       pack2(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                                       pack2(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
            const int col = half * 64 + c * 32 + g * 8;
            if (vec_io) {
              *(uint4*)(o + col) = w;
            } else {
              const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                ((uint16_t*)o)[col + 2 * k] = (uint16_t)(ww[k] & 0xFFFF);
                ((uint16_t*)o)[col + 2 * k + 1] = (uint16_t)(ww[k] >> 16);
              }
            }
          }
        }
      }
      if (ldst && half == 0) *ldst = mrun * 0.6931471805599453f + logf(l);
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
  }
}
// 4D tensor map of one layer's K/V cache ([batch*N rows][2 * kvdim] bf16, K
// then V of each row) viewed as {64 columns, row, 64-column block of the K or
// V half, K/V}: a box {64, TK, dh / 64, 1} at (0, row, head * dh / 64, w) is one
// head's K (w = 0) or V (w = 1) for TK keys, as 128-byte-swizzled [TK][64]
// boxes, one per 64-column block (cached per buffer and shape).
const CUtensorMap* kv_map_tiles(const void* base, int rows, int kvdim, int dh) {
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
  const cuuint32_t box[4] = {64, (cuuint32_t)TK, (cuuint32_t)(dh / 64), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return nullptr;
  return &cache.emplace(key, m).first->second;
}

}  // namespace at

cudaError_t launch_attention_tc(const AttnArgs& a, int batch, cudaStream_t st) {
  if (a.dh != at::DH || (a.kvdim % 64)) return cudaErrorInvalidValue;
  // drift is measured by the deferred pass only
  if (a.measure && ((a.proxy_prev && (!a.proxy_new || !a.proxy_new_lse)) ||
                    (a.active_prev && (!a.active_new || !a.active_new_lse))))
    return cudaErrorInvalidValue;
  const CUtensorMap* map = at::kv_map_tiles(a.kv_layer, batch * a.N, a.kvdim, at::DH);
  if (!map) return cudaErrorInvalidValue;
  static PerDeviceOnce attr;
  {
    const cudaError_t e = func_attr_once(attr, (const void*)at::attn_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, at::SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.n_work, a.H, 1);
  cfg.blockDim = dim3(at::THREADS);
  cfg.dynamicSmemBytes = at::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute att[1];
  att[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  att[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = att;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, at::attn_tc_kernel, *map, a);
}

}  // namespace polestar
