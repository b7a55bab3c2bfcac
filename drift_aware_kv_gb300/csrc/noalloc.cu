// Row attention + KL drift without any device allocation.
//
// Some callers cannot let a library allocate device memory: a host application
// that owns every device allocation through its own pool or memory cap (where a
// stray cudaMalloc breaks its accounting or fails), or a latency-critical
// serving loop in which cudaMalloc / cudaFree may synchronise the whole device.
// For them, polestar_attention_noalloc runs the same bf16 tensor-core attention
// kernels as the rest of the library, but every piece of scratch it needs (the
// row table and the work list; key-split partial results stay in distributed
// shared memory) lives in the fixed-size file-scope device arrays below.  Those arrays exist on every GPU
// that loads the library, for as long as the library stays loaded.
#include <mutex>

#include "../../include/polestar.h"
#include "kernels.h"

namespace polestar {
namespace {

constexpr int kMaxRows = 256;                               // rows per call
constexpr int kMaxWork = (kMaxRows + ATT_ITEM_ROWS - 1) / ATT_ITEM_ROWS;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int4 g_scratch_rows[kMaxRows];
static __device__ __align__(256) int4 g_scratch_work[kMaxWork];

struct DeviceScratch {
  bool ready = false;
  int4* rows = nullptr;
  int4* work = nullptr;
};
DeviceScratch g_dev[kMaxDevices];
std::mutex g_mu;

// Resolve the device addresses of the scratch arrays for the current device
// (host code cannot use the array names as device pointers).
polestar_status resolve(int dev, DeviceScratch** out) {
  if (dev < 0 || dev >= kMaxDevices) return POLESTAR_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceScratch& s = g_dev[dev];
  if (!s.ready) {
    if (cudaGetSymbolAddress((void**)&s.rows, g_scratch_rows) != cudaSuccess) return POLESTAR_ERR_CUDA;
    if (cudaGetSymbolAddress((void**)&s.work, g_scratch_work) != cudaSuccess) return POLESTAR_ERR_CUDA;
    s.ready = true;
  }
  *out = &s;
  return POLESTAR_OK;
}

// Row table (tracked rows carry their history, the rest only produce output)
// and work list (near-equal items of the row range [0, R), as attention_items
// builds them), written on the device from the caller's flags.
__global__ void fill_tables_kernel(const uint8_t* __restrict__ tracked, int R, int n_work, int4* rows,
                                   int4* work) {
  for (int r = threadIdx.x; r < R; r += blockDim.x)
    rows[r] = make_int4(0, 0, (tracked && tracked[r]) ? ROW_ACTIVE : ROW_OTHER, r);
  for (int i = threadIdx.x; i < n_work; i += blockDim.x) {
    const int lo = i * R / n_work, hi = (i + 1) * R / n_work;
    work[i] = make_int4(lo, hi - lo, 0, 0);
  }
}

}  // namespace
}  // namespace polestar

using namespace polestar;

extern "C" polestar_status polestar_attention_noalloc(const void* q, const void* kv, int32_t N, int32_t H,
                                                      int32_t Hkv, int32_t head_dim, int32_t R,
                                                      const uint8_t* tracked, float* prev, float* prev_lse,
                                                      int32_t measure, int32_t store, void* out, float* kl,
                                                      void* stream) {
  if (!q || !kv || !out || R < 1 || N < 1 || H < 1 || Hkv < 1 || H % Hkv) return POLESTAR_ERR_INVALID_ARG;
  if (R > kMaxRows) return POLESTAR_ERR_INVALID_ARG;  // the static row table holds kMaxRows rows
  if (head_dim != 64 && head_dim != 128) return POLESTAR_ERR_UNSUPPORTED;
  if (tracked && (!prev || !prev_lse || (measure && !kl))) return POLESTAR_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return POLESTAR_ERR_CUDA;
  DeviceScratch* s = nullptr;
  const polestar_status st0 = resolve(dev, &s);
  if (st0 != POLESTAR_OK) return st0;
  cudaStream_t st = (cudaStream_t)stream;
  const int item_rows =
      attention_item_rows(true, head_dim, (R + ATT_TC_ROWS - 1) / ATT_TC_ROWS, H, tracked != nullptr && measure != 0);
  const int n_work = (R + item_rows - 1) / item_rows;
  fill_tables_kernel<<<1, 256, 0, st>>>(tracked, R, n_work, s->rows, s->work);
  AttnArgs a{};
  a.q = q;
  a.ldq = H * head_dim;
  a.rows = s->rows;
  a.R = R;
  a.kv_layer = kv;
  a.kv_seq_stride = 0;
  a.kvdim = Hkv * head_dim;
  a.N = N;
  a.H = H;
  a.Hkv = Hkv;
  a.dh = head_dim;
  a.K = 1;
  a.B = R;
  a.scale = 1.f / sqrtf((float)head_dim);
  a.out = out;
  a.ldo = H * head_dim;
  a.other_live = 1;
  a.active_prev = tracked ? prev : nullptr;
  a.active_prev_lse = tracked ? prev_lse : nullptr;
  a.measure = measure;
  a.store = store;
  a.kl_out = kl;
  a.work = s->work;
  a.n_work = n_work;
  a.item_rows = item_rows;
  a.batch = 1;
  if (launch_row_attention<__nv_bfloat16>(a, st) != cudaSuccess) return POLESTAR_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? POLESTAR_OK : POLESTAR_ERR_CUDA;
}
