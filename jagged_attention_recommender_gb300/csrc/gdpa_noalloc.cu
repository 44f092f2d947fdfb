// gdpa_noalloc.cu -- gdpa_fwd_noalloc: the forward pass for callers that
// must not allocate memory.
//
// Some callers cannot call cudaMalloc, or any allocator, where they run
// attention: a serving process that carves all device memory into a fixed
// arena up front and forbids allocation on its request path (an allocation
// there can fail or stall the whole device), or a framework hook that must
// not go around its caching allocator.  gdpa_fwd keeps its work list in a
// library-owned device buffer that it grows with cudaMalloc; this entry point
// keeps the work list in one fixed file-scope device array instead and plans
// into fixed host arrays, so it never allocates.  The price is a hard size
// limit and one scratch area per GPU shared by every call.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gdpa_internal.h"

namespace gdpa {
namespace {

constexpr int64_t kNaMaxItems = 261632;  // work items (query tiles x heads) per call
constexpr int kNaMaxCtas = 2047;         // persistent CTAs (SMs) the work list can describe
constexpr int kNaMaxBatch = 65536;       // sequences per call
constexpr size_t kNaItemBytes = (size_t)kNaMaxItems * sizeof(gdpa_work_item_t);
constexpr size_t kNaScratchBytes = kNaItemBytes + (size_t)(kNaMaxCtas + 1) * sizeof(int32_t);  // 4 MiB
static_assert(kNaScratchBytes == (size_t)4 << 20, "scratch is 4 MiB");

// Work list of the most recent call (items grouped by CTA, then cta_begin).
// A device holds these 4 MiB from the moment the driver loads this module
// onto it (at the first call there, under lazy module loading) until the
// process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaScratchBytes];

// Host-side staging and planner arrays: static storage, shared by every call.
constexpr int kNaBuckets = 1 << 16;  // counting-sort cursors; costlier batches sort in place
struct NoAllocHost {
  int32_t offsets[2 * (kNaMaxBatch + 1)];
  gdpa_work_item_t items[kNaMaxItems];
  int64_t cost[kNaMaxItems];
  uint32_t order[kNaMaxItems];
  int32_t owner[kNaMaxItems];
  uint64_t keys[kNaMaxItems];
  uint32_t bucket[kNaBuckets];
  int64_t load[2048];
  int32_t tree[4096];
  int32_t count[2048];
  unsigned char upload[kNaScratchBytes];
};
static NoAllocHost g_host;
static std::mutex g_mu;
static void* g_dev_scratch[64];

// The library's planner (plan_items_into, the same routine gdpa_fwd uses)
// over the fixed arrays; the work list lands in the upload image: items at
// offset 0, cta_begin at kNaItemBytes.
gdpa_status_t na_plan(const int32_t* qo, const int32_t* ko, int B, int H, int window_blocks, int rows_per_item,
                      int num_ctas, int64_t* n_out) {
  const PlanStorage st{g_host.items, g_host.cost, g_host.order, g_host.owner, g_host.keys, g_host.bucket,
                       g_host.load,  g_host.tree, g_host.count, kNaMaxItems,  kNaBuckets,   2048};
  gdpa_work_item_t* out_items = reinterpret_cast<gdpa_work_item_t*>(g_host.upload);
  int32_t* cta_begin = reinterpret_cast<int32_t*>(g_host.upload + kNaItemBytes);
  return plan_items_into(qo, ko, B, H, window_blocks, rows_per_item, num_ctas, st, out_items, cta_begin, nullptr,
                         n_out);
}

}  // namespace
}  // namespace gdpa

using namespace gdpa;

extern "C" gdpa_status_t gdpa_fwd_noalloc(const void* q, const void* k, const void* v, const int32_t* q_offsets,
                                          const int32_t* kv_offsets, int B, int H, int D, int act,
                                          int window_blocks, float scale, void* out, void* stream) {
  gdpa_status_t st = validate_shape(B, H, D, act, window_blocks);
  if (st != GDPA_OK) return st;
  if (B == 0) return GDPA_OK;
  if (B > kNaMaxBatch) return GDPA_ERR_NO_MEMORY;
  if (!q_offsets || !kv_offsets) return GDPA_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return GDPA_ERR_CUDA;
  if (device < 0 || device >= 64) return GDPA_ERR_UNSUPPORTED;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0)
    return GDPA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_scratch[device]) {  // once per device: the array's device address
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return GDPA_ERR_CUDA;
    g_dev_scratch[device] = ptr;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t ob = ((size_t)B + 1) * sizeof(int32_t);
  int32_t* hq = g_host.offsets;
  int32_t* hk = g_host.offsets + B + 1;
  if (cudaMemcpyAsync(hq, q_offsets, ob, cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (cudaMemcpyAsync(hk, kv_offsets, ob, cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDPA_ERR_CUDA;
  int64_t Tq = 0, Tkv = 0;
  if ((st = validate_offsets(hq, hk, B, window_blocks, &Tq, &Tkv)) != GDPA_OK) return st;
  if (Tq > 0 && (!q || !out || (reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)))
    return GDPA_ERR_INVALID_ARG;
  if (Tkv > 0 && (!k || !v || (reinterpret_cast<uintptr_t>(k) & 15) || (reinterpret_cast<uintptr_t>(v) & 15)))
    return GDPA_ERR_INVALID_ARG;
  if (Tq >= (int64_t)1 << 31 || Tkv >= (int64_t)1 << 31) return GDPA_ERR_UNSUPPORTED;
  if (Tq == 0) return GDPA_OK;
  const int rpi = choose_rows_per_item(hq, B, D, window_blocks);
  const int64_t n_est = count_plan_items(hq, B, H, rpi);
  if (n_est > kNaMaxItems) return GDPA_ERR_NO_MEMORY;
  const int num_ctas = (int)std::min<int64_t>(std::min<int64_t>(n_est, sms), kNaMaxCtas);
  int64_t n = 0;
  if ((st = na_plan(hq, hk, B, H, window_blocks, rpi, num_ctas, &n)) != GDPA_OK) return st;
  unsigned char* dev = static_cast<unsigned char*>(g_dev_scratch[device]);
  // The whole region the launch reads is rewritten here; nothing needs zeroing.
  if (cudaMemcpyAsync(dev, g_host.upload, (size_t)n * sizeof(gdpa_work_item_t), cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaMemcpyAsync(dev + kNaItemBytes, g_host.upload + kNaItemBytes, (size_t)(num_ctas + 1) * sizeof(int32_t),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return GDPA_ERR_CUDA;
  LaunchArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.q_off = q_offsets;
  a.kv_off = kv_offsets;
  a.items = reinterpret_cast<const gdpa_work_item_t*>(dev);
  a.cta_begin = reinterpret_cast<const int32_t*>(dev + kNaItemBytes);
  a.num_ctas = num_ctas;
  a.rows_per_item = rpi;
  a.kv_tile = choose_kv_tile(hq, hk, B, window_blocks, rpi);
  a.Tq = Tq;
  a.Tkv = Tkv;
  a.H = H;
  a.D = D;
  a.act = act;
  a.window_blocks = window_blocks;
  a.scale = scale;
  a.stream = stream;
  return launch_forward(a);
}
