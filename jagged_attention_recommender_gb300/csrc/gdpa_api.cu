// gdpa_api.cu -- the C ABI of libgdpa (declared in include/gdpa.h): argument
// validation, planning, library-owned buffers, launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "gdpa_internal.h"

struct gdpa_plan {
  int B, H, D, act, window_blocks;
  int num_ctas;
  int rows_per_item, kv_tile;
  int device;
  int64_t n_items, Tq, Tkv;
  void* d_buf;  // work items followed by cta_begin
  const gdpa_work_item_t* d_items;
  const int32_t* d_cta_begin;
};

namespace gdpa {

bool fault_injected(const char* what) {
  const char* e = std::getenv("GDPA_FAULT_INJECT");
  return e && std::strcmp(e, what) == 0;
}

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 8;                        // gdpa_fwd_host pipeline depth
constexpr double kChunkBytes = 64.0 * (1 << 20);     // target bytes in + out per chunk

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdpa_status_t num_sms(int* device, int* sms) {
  if (cudaGetDevice(device) != cudaSuccess) return GDPA_ERR_CUDA;
  if (*device < 0 || *device >= kMaxDevices) return GDPA_ERR_UNSUPPORTED;
  static int cache[kMaxDevices] = {};
  if (cache[*device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *device) != cudaSuccess || n <= 0)
      return GDPA_ERR_CUDA;
    cache[*device] = n;
  }
  *sms = cache[*device];
  return GDPA_OK;
}

// Grow-only device / pinned-host buffer.
struct Buf {
  void* p = nullptr;
  size_t cap = 0;
  bool pinned = false;
  gdpa_status_t ensure(size_t bytes) {
    if (fault_injected("alloc")) return GDPA_ERR_NO_MEMORY;  // failure-path tests
    if (bytes <= cap) return GDPA_OK;
    size_t want = bytes + bytes / 4 + 256;
    void* np = nullptr;
    cudaError_t e = pinned ? cudaMallocHost(&np, want) : cudaMalloc(&np, want);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GDPA_ERR_NO_MEMORY;
    }
    release();
    p = np;
    cap = want;
    return GDPA_OK;
  }
  void release() {
    if (p) pinned ? cudaFreeHost(p) : cudaFree(p);
    p = nullptr;
    cap = 0;
  }
};

// The planner's working arrays, kept from call to call (grow-only), so that
// planning a batch allocates and first-touches nothing in the steady state.
struct PlanScratch {
  std::vector<gdpa_work_item_t> items;
  std::vector<int64_t> cost, load;
  std::vector<uint32_t> order, bucket;
  std::vector<int32_t> owner, tree, count;
  std::vector<uint64_t> keys;
  gdpa_status_t ensure(int64_t n, int leaves, int ctas) {
    try {
      if ((int64_t)items.size() < n) {
        items.resize((size_t)n);
        cost.resize((size_t)n);
        order.resize((size_t)n);
        owner.resize((size_t)n);
        keys.resize((size_t)n);
        bucket.resize((size_t)(4 * n + 1026));
      }
      if ((int)load.size() < leaves) {
        load.resize((size_t)leaves);
        tree.resize(2 * (size_t)leaves);
      }
      if ((int)count.size() < ctas) count.resize((size_t)ctas);
    } catch (const std::bad_alloc&) {
      return GDPA_ERR_NO_MEMORY;
    }
    return GDPA_OK;
  }
  PlanStorage storage() {
    return PlanStorage{items.data(), cost.data(),  order.data(), owner.data(), keys.data(), bucket.data(),
                       load.data(),  tree.data(),  count.data(), (int64_t)items.size(), (int64_t)bucket.size(),
                       (int)load.size()};
  }
};

// Per-device state behind gdpa_fwd / gdpa_fwd_host.
struct DeviceCtx {
  std::mutex mu;
  PlanScratch plan;
  // Work lists go up through two slots used in turn, each a pinned staging
  // buffer and a device buffer, on the upload stream s_up: the list of the
  // next launch is copied while the current one runs, and the launch stream
  // only waits for its own list (up_done).  stage_free[b]: slot b's staging
  // buffer may be overwritten; work_free[b]: no launch reads d_work[b] any more.
  Buf h_stage[2] = {{nullptr, 0, true}, {nullptr, 0, true}};
  Buf d_work[2];
  int slot = 0;  // the slot the next plan takes
  int cur = 0;   // the slot of the last plan (read by the launch that follows it)
  cudaStream_t s_up = nullptr;
  cudaEvent_t up_done[2] = {};
  Buf h_off{nullptr, 0, true};    // gdpa_fwd: device offsets read back
  Buf d_io;                       // gdpa_fwd_host: q, k, v, out, offsets, work lists
  Buf h_io{nullptr, 0, true};     // gdpa_fwd_host: pinned offsets + work lists
  cudaEvent_t stage_free[2] = {};
  cudaEvent_t work_free[2] = {};
  bool events_ok = false;
  // gdpa_bwd: device work lists + scratch, pinned staging, and their events
  Buf d_bwd;
  Buf h_bwd{nullptr, 0, true};
  cudaEvent_t bwd_stage_free = nullptr, bwd_free = nullptr;
  // gdpa_fwd_host pipeline: copy-in and copy-out streams, per-chunk events
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_meta = nullptr, ev_in[kMaxChunks] = {}, ev_done[kMaxChunks] = {};
  bool host_path_ok = false;
  gdpa_status_t init_host_path() {
    if (host_path_ok) return GDPA_OK;
    if (cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking) != cudaSuccess) return GDPA_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking) != cudaSuccess) return GDPA_ERR_CUDA;
    if (cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming) != cudaSuccess) return GDPA_ERR_CUDA;
    if (cudaEventCreateWithFlags(&ev_meta, cudaEventDisableTiming) != cudaSuccess) return GDPA_ERR_CUDA;
    for (int i = 0; i < kMaxChunks; ++i)
      if (cudaEventCreateWithFlags(&ev_in[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&ev_done[i], cudaEventDisableTiming) != cudaSuccess)
        return GDPA_ERR_CUDA;
    host_path_ok = true;
    return GDPA_OK;
  }
  gdpa_status_t init() {
    if (events_ok) return GDPA_OK;
    if (cudaStreamCreateWithFlags(&s_up, cudaStreamNonBlocking) != cudaSuccess) return GDPA_ERR_CUDA;
    for (int b = 0; b < 2; ++b) {
      if (cudaEventCreateWithFlags(&stage_free[b], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&work_free[b], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&up_done[b], cudaEventDisableTiming) != cudaSuccess)
        return GDPA_ERR_CUDA;
      if (cudaEventRecord(stage_free[b], 0) != cudaSuccess || cudaEventRecord(work_free[b], 0) != cudaSuccess)
        return GDPA_ERR_CUDA;
    }
    if (cudaEventCreateWithFlags(&bwd_stage_free, cudaEventDisableTiming) != cudaSuccess) return GDPA_ERR_CUDA;
    if (cudaEventCreateWithFlags(&bwd_free, cudaEventDisableTiming) != cudaSuccess) return GDPA_ERR_CUDA;
    if (cudaEventRecord(bwd_stage_free, 0) != cudaSuccess || cudaEventRecord(bwd_free, 0) != cudaSuccess)
      return GDPA_ERR_CUDA;
    events_ok = true;
    return GDPA_OK;
  }
};

DeviceCtx& ctx(int device) {
  static DeviceCtx ctxs[kMaxDevices];
  return ctxs[device];
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Plans on the host into the next slot's pinned staging buffer and uploads
// the work list into that slot's device buffer on the upload stream (both
// guarded by events against the launch that used the slot two calls ago);
// `stream` waits for the copy.  The launch that follows reads slot c.cur.
// `single_tile`: one 128-row query tile and 128-key tiles per item whatever
// the shapes (the MXFP8 kernel's item kind).
// `extra` (optional): an int32 array uploaded after the work list (the
// MXFP8 V layout's sequence columns), at work_extra().
gdpa_status_t plan_and_upload(DeviceCtx& c, const int32_t* h_q_off, const int32_t* h_kv_off, int B, int H,
                              int D, int window_blocks, int sms, cudaStream_t stream, int* num_ctas, int* rows_per_item,
                              int* kv_tile, int64_t* n_items, bool single_tile = false, bool pair64 = false,
                              const std::vector<int32_t>* extra = nullptr) {
  const int rpi = single_tile ? kBlockM : pair64 ? 2 * kBlockM : choose_rows_per_item(h_q_off, B, D, window_blocks);
  *rows_per_item = rpi;
  *kv_tile = single_tile ? kBlockN : pair64 ? kBlockN / 2 : choose_kv_tile(h_q_off, h_kv_off, B, window_blocks, rpi);
  const int64_t n = count_plan_items(h_q_off, B, H, rpi);
  *n_items = n;
  if (n == 0) {
    *num_ctas = 0;
    return GDPA_OK;
  }
  const int ctas = (int)(n < sms ? n : sms);
  int leaves = 1;
  while (leaves < ctas) leaves <<= 1;
  gdpa_status_t st;
  if ((st = c.plan.ensure(n, leaves, ctas)) != GDPA_OK) return st;
  const size_t items_bytes = (size_t)n * sizeof(gdpa_work_item_t);
  const size_t list_bytes = align_up(items_bytes, 16) + ((size_t)ctas + 1) * sizeof(int32_t);
  const size_t total = extra ? align_up(list_bytes, 16) + extra->size() * sizeof(int32_t) : list_bytes;
  const int b = c.slot;
  // A stream being captured into a graph keeps the copy on itself.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return GDPA_ERR_CUDA;
  cudaStream_t us = cs == cudaStreamCaptureStatusNone ? c.s_up : stream;
  if (cudaStreamWaitEvent(us, c.work_free[b], 0) != cudaSuccess) return GDPA_ERR_CUDA;
  if (c.d_work[b].cap < total) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GDPA_ERR_CUDA;  // old buffer may be in use
    if ((st = c.d_work[b].ensure(total)) != GDPA_OK) return st;
  }
  if (cudaEventSynchronize(c.stage_free[b]) != cudaSuccess) return GDPA_ERR_CUDA;
  if ((st = c.h_stage[b].ensure(total)) != GDPA_OK) return st;
  // the plan lands in the pinned staging buffer directly: items, then cta_begin
  char* h = static_cast<char*>(c.h_stage[b].p);
  int64_t got = 0;
  st = plan_items_into(h_q_off, h_kv_off, B, H, window_blocks, rpi, ctas, c.plan.storage(),
                       reinterpret_cast<gdpa_work_item_t*>(h), reinterpret_cast<int32_t*>(h + align_up(items_bytes, 16)),
                       nullptr, &got);
  if (st != GDPA_OK) return st;
  if (got != n) return GDPA_ERR_INVALID_ARG;
  if (extra && !extra->empty())
    std::memcpy(h + align_up(list_bytes, 16), extra->data(), extra->size() * sizeof(int32_t));
  if (cudaMemcpyAsync(c.d_work[b].p, h, total, cudaMemcpyHostToDevice, us) != cudaSuccess) return GDPA_ERR_CUDA;
  if (cudaEventRecord(c.stage_free[b], us) != cudaSuccess) return GDPA_ERR_CUDA;
  if (us != stream) {
    if (cudaEventRecord(c.up_done[b], us) != cudaSuccess) return GDPA_ERR_CUDA;
    if (cudaStreamWaitEvent(stream, c.up_done[b], 0) != cudaSuccess) return GDPA_ERR_CUDA;
  }
  c.cur = b;
  c.slot = b ^ 1;
  *num_ctas = ctas;
  return GDPA_OK;
}

// Device address of the `extra` array plan_and_upload placed after a work
// list of n_items items over num_ctas CTAs.
const int32_t* work_extra(const DeviceCtx& c, int64_t n_items, int num_ctas) {
  const size_t list_bytes = align_up((size_t)n_items * sizeof(gdpa_work_item_t), 16) + ((size_t)num_ctas + 1) * 4;
  return reinterpret_cast<const int32_t*>(static_cast<const char*>(c.d_work[c.cur].p) + align_up(list_bytes, 16));
}

gdpa_status_t launch_with_ctx(DeviceCtx& c, const void* q, const void* k, const void* v, void* out,
                              const int32_t* d_q_off, const int32_t* d_kv_off, int64_t Tq, int64_t Tkv, int H, int D,
                              int act, int window_blocks, float scale, int num_ctas, int rows_per_item,
                              int kv_tile, int64_t n_items, cudaStream_t stream, float* lse = nullptr,
                              const void* q_sf = nullptr, const void* k_sf = nullptr, const void* vt_sf = nullptr,
                              int64_t VT = -1) {
  LaunchArgs a;
  a.lse = lse;
  a.q_sf = q_sf;
  a.k_sf = k_sf;
  if (VT >= 0) {  // all three inputs in MXFP8 (gdpa_fwd_mxfp8): the sequence columns follow the work list
    a.vt_sf = vt_sf;
    a.vt_col = work_extra(c, n_items, num_ctas);
    a.VT = VT;
  }
  a.rows_per_item = rows_per_item;
  a.kv_tile = kv_tile;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.q_off = d_q_off;
  a.kv_off = d_kv_off;
  a.items = static_cast<const gdpa_work_item_t*>(c.d_work[c.cur].p);
  a.cta_begin = reinterpret_cast<const int32_t*>(static_cast<const char*>(c.d_work[c.cur].p) +
                                                 align_up((size_t)n_items * sizeof(gdpa_work_item_t), 16));
  a.num_ctas = num_ctas;
  a.Tq = Tq;
  a.Tkv = Tkv;
  a.H = H;
  a.D = D;
  a.act = act;
  a.window_blocks = window_blocks;
  a.scale = scale;
  a.stream = stream;
  gdpa_status_t st = launch_forward(a);
  if (st != GDPA_OK) return st;
  return cudaEventRecord(c.work_free[c.cur], stream) == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}


gdpa_status_t check_tensors(const void* q, const void* k, const void* v, const void* out, int64_t Tq, int64_t Tkv) {
  if (Tq > 0 && (!q || !out || !aligned16(q) || !aligned16(out))) return GDPA_ERR_INVALID_ARG;
  if (Tkv > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return GDPA_ERR_INVALID_ARG;
  if (Tq >= (int64_t)1 << 31 || Tkv >= (int64_t)1 << 31) return GDPA_ERR_UNSUPPORTED;
  return GDPA_OK;
}

}  // namespace
}  // namespace gdpa

using namespace gdpa;

extern "C" gdpa_status_t gdpa_fwd(const void* q, const void* k, const void* v, const int32_t* q_offsets,
                                  const int32_t* kv_offsets, int B, int H, int D, int act, int window_blocks,
                                  float scale, void* out, void* stream) {
  gdpa_status_t st = validate_shape(B, H, D, act, window_blocks);
  if (st != GDPA_OK) return st;
  if (B == 0) return GDPA_OK;
  if (!q_offsets || !kv_offsets) return GDPA_ERR_INVALID_ARG;
  int device = 0, sms = 0;
  if ((st = num_sms(&device, &sms)) != GDPA_OK) return st;
  DeviceCtx& c = ctx(device);
  std::lock_guard<std::mutex> lock(c.mu);
  if ((st = c.init()) != GDPA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::vector<int32_t> off(2 * ((size_t)B + 1));
  const size_t ob = ((size_t)B + 1) * sizeof(int32_t);
  if ((st = c.h_off.ensure(2 * ob)) != GDPA_OK) return st;
  int32_t* h = static_cast<int32_t*>(c.h_off.p);
  if (cudaMemcpyAsync(h, q_offsets, ob, cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (cudaMemcpyAsync(h + B + 1, kv_offsets, ob, cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDPA_ERR_CUDA;
  std::memcpy(off.data(), h, 2 * ob);
  const int32_t* hq = off.data();
  const int32_t* hk = off.data() + B + 1;
  int64_t Tq = 0, Tkv = 0;
  if ((st = validate_offsets(hq, hk, B, window_blocks, &Tq, &Tkv)) != GDPA_OK) return st;
  if ((st = check_tensors(q, k, v, out, Tq, Tkv)) != GDPA_OK) return st;
  if (Tq == 0) return GDPA_OK;
  int num_ctas = 0;
  int rpi = 0, kvt = 0;
  int64_t n_items = 0;
  if ((st = plan_and_upload(c, hq, hk, B, H, D, window_blocks, sms, s, &num_ctas, &rpi, &kvt, &n_items)) != GDPA_OK)
    return st;
  return launch_with_ctx(c, q, k, v, out, q_offsets, kv_offsets, Tq, Tkv, H, D, act, window_blocks, scale, num_ctas,
                         rpi, kvt, n_items, s);
}

extern "C" gdpa_status_t gdpa_fwd_async(const void* q, const void* k, const void* v, const int32_t* h_q_offsets,
                                        const int32_t* h_kv_offsets, const int32_t* q_offsets,
                                        const int32_t* kv_offsets, int B, int H, int D, int act, int window_blocks,
                                        float scale, void* out, void* stream) {
  gdpa_status_t st = validate_shape(B, H, D, act, window_blocks);
  if (st != GDPA_OK) return st;
  if (B == 0) return GDPA_OK;
  int64_t Tq = 0, Tkv = 0;
  if ((st = validate_offsets(h_q_offsets, h_kv_offsets, B, window_blocks, &Tq, &Tkv)) != GDPA_OK) return st;
  if ((st = check_tensors(q, k, v, out, Tq, Tkv)) != GDPA_OK) return st;
  if (Tq == 0) return GDPA_OK;
  if (!q_offsets || !kv_offsets) return GDPA_ERR_INVALID_ARG;
  int device = 0, sms = 0;
  if ((st = num_sms(&device, &sms)) != GDPA_OK) return st;
  DeviceCtx& c = ctx(device);
  std::lock_guard<std::mutex> lock(c.mu);
  if ((st = c.init()) != GDPA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int num_ctas = 0;
  int rpi = 0, kvt = 0;
  int64_t n_items = 0;
  if ((st = plan_and_upload(c, h_q_offsets, h_kv_offsets, B, H, D, window_blocks, sms, s, &num_ctas, &rpi,
                            &kvt, &n_items)) != GDPA_OK)
    return st;
  return launch_with_ctx(c, q, k, v, out, q_offsets, kv_offsets, Tq, Tkv, H, D, act, window_blocks, scale, num_ctas,
                         rpi, kvt, n_items, s);
}

namespace gdpa {
namespace {

// gdpa_fwd_async with an optional logsumexp output and the internal window
// code (> 0: block window, < 0: sliding window of -window tokens).
// With q_sf set, q and k are MXFP8 codes with those scale words (full
// attention, D = 128, single-tile items).
gdpa_status_t fwd_async_impl(const void* q, const void* k, const void* v, const int32_t* h_q_offsets,
                             const int32_t* h_kv_offsets, const int32_t* q_offsets, const int32_t* kv_offsets, int B,
                             int H, int D, int act, int window, float scale, void* out, float* lse, void* stream,
                             const void* q_sf = nullptr, const void* k_sf = nullptr) {
  int64_t Tq = 0, Tkv = 0;
  gdpa_status_t st;
  if ((st = validate_offsets(h_q_offsets, h_kv_offsets, B, window, &Tq, &Tkv)) != GDPA_OK) return st;
  if ((st = check_tensors(q, k, v, out, Tq, Tkv)) != GDPA_OK) return st;
  if (Tq == 0) return GDPA_OK;
  if (!q_offsets || !kv_offsets) return GDPA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return GDPA_ERR_INVALID_ARG;
  int device = 0, sms = 0;
  if ((st = num_sms(&device, &sms)) != GDPA_OK) return st;
  DeviceCtx& c = ctx(device);
  std::lock_guard<std::mutex> lock(c.mu);
  if ((st = c.init()) != GDPA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int num_ctas = 0;
  int rpi = 0, kvt = 0;
  int64_t n_items = 0;
  if ((st = plan_and_upload(c, h_q_offsets, h_kv_offsets, B, H, D, window, sms, s, &num_ctas, &rpi, &kvt,
                            &n_items, q_sf != nullptr)) != GDPA_OK)
    return st;
  return launch_with_ctx(c, q, k, v, out, q_offsets, kv_offsets, Tq, Tkv, H, D, act, window, scale, num_ctas, rpi,
                         kvt, n_items, s, act == GDPA_ACT_SOFTMAX ? lse : nullptr, q_sf, k_sf);
}

}  // namespace
}  // namespace gdpa

extern "C" gdpa_status_t gdpa_fwd_lse(const void* q, const void* k, const void* v, const int32_t* h_q_offsets,
                                      const int32_t* h_kv_offsets, const int32_t* q_offsets, const int32_t* kv_offsets,
                                      int B, int H, int D, int act, int window_blocks, float scale, void* out,
                                      float* lse, void* stream) {
  gdpa_status_t st = validate_shape(B, H, D, act, window_blocks);
  if (st != GDPA_OK) return st;
  if (B == 0) return GDPA_OK;
  if (act == GDPA_ACT_SOFTMAX && !lse) return GDPA_ERR_INVALID_ARG;
  return fwd_async_impl(q, k, v, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act, window_blocks,
                        scale, out, lse, stream);
}

extern "C" gdpa_status_t gdpa_fwd_sliding(const void* q, const void* k, const void* v, const int32_t* h_q_offsets,
                                          const int32_t* h_kv_offsets, const int32_t* q_offsets,
                                          const int32_t* kv_offsets, int B, int H, int D, int act, int window_tokens,
                                          float scale, void* out, float* lse, void* stream) {
  if (window_tokens < 1) return GDPA_ERR_INVALID_ARG;
  gdpa_status_t st = validate_shape(B, H, D, act, 1);  // as a window: softmax only
  if (st != GDPA_OK) return st;
  if (B == 0) return GDPA_OK;
  return fwd_async_impl(q, k, v, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act, -window_tokens,
                        scale, out, lse, stream);
}

extern "C" gdpa_status_t gdpa_fwd_mx(const void* q8, const void* q_sf, const void* k8, const void* k_sf,
                                     const void* v, const int32_t* h_q_offsets, const int32_t* h_kv_offsets,
                                     const int32_t* q_offsets, const int32_t* kv_offsets, int B, int H, int D, int act,
                                     float scale, void* out, float* lse, void* stream) {
  gdpa_status_t st = validate_shape(B, H, D, act, 0);
  if (st != GDPA_OK) return st;
  if (D != 128) return GDPA_ERR_UNSUPPORTED;
  if (B == 0) return GDPA_OK;
  const bool any_q = h_q_offsets && h_q_offsets[B] > 0, any_kv = h_kv_offsets && h_kv_offsets[B] > 0;
  if (any_q && (!q_sf || (reinterpret_cast<uintptr_t>(q_sf) & 3u) != 0)) return GDPA_ERR_INVALID_ARG;
  if (any_kv && (!k_sf || (reinterpret_cast<uintptr_t>(k_sf) & 3u) != 0)) return GDPA_ERR_INVALID_ARG;
  // with no keys k_sf is never read
  return fwd_async_impl(q8, k8, v, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act, 0, scale, out, lse,
                        stream, q_sf, k_sf ? k_sf : q_sf);
}

extern "C" gdpa_status_t gdpa_fwd_mxfp8(const void* q8, const void* q_sf, const void* k8, const void* k_sf,
                                        const void* vt8, const void* vt_sf, const int32_t* h_q_offsets,
                                        const int32_t* h_kv_offsets, const int32_t* q_offsets,
                                        const int32_t* kv_offsets, int B, int H, int D, int act, float scale,
                                        void* out, float* lse, void* stream) {
  gdpa_status_t st = validate_shape(B, H, D, act, 0);
  if (st != GDPA_OK) return st;
  if (D != 128 || act != GDPA_ACT_SOFTMAX) return GDPA_ERR_UNSUPPORTED;
  if (B == 0) return GDPA_OK;
  int64_t Tq = 0, Tkv = 0;
  if ((st = validate_offsets(h_q_offsets, h_kv_offsets, B, 0, &Tq, &Tkv)) != GDPA_OK) return st;
  if (Tq > 0 && (!q8 || !out || !aligned16(q8) || !aligned16(out))) return GDPA_ERR_INVALID_ARG;
  if (Tq > 0 && (!q_sf || (reinterpret_cast<uintptr_t>(q_sf) & 3u) != 0)) return GDPA_ERR_INVALID_ARG;
  if (Tkv > 0 && (!k8 || !vt8 || !vt_sf || !k_sf || !aligned16(k8) || !aligned16(vt8) ||
                  (reinterpret_cast<uintptr_t>(k_sf) & 3u) != 0))
    return GDPA_ERR_INVALID_ARG;
  if (Tq >= (int64_t)1 << 31 || Tkv >= (int64_t)1 << 31) return GDPA_ERR_UNSUPPORTED;
  if (Tq == 0) return GDPA_OK;
  if (!q_offsets || !kv_offsets) return GDPA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return GDPA_ERR_INVALID_ARG;
  // the key-major V layout: sequence b from column 32 * sum_{b' < b} ceil(Lkv_b' / 32)
  std::vector<int32_t> vt_col;
  try {
    vt_col.resize((size_t)B + 1);
  } catch (const std::bad_alloc&) {
    return GDPA_ERR_NO_MEMORY;
  }
  int64_t col = 0;
  for (int b = 0; b < B; ++b) {
    vt_col[b] = static_cast<int32_t>(col);
    col += 32 * (((int64_t)h_kv_offsets[b + 1] - h_kv_offsets[b] + 31) / 32);
    if (col >= ((int64_t)1 << 31)) return GDPA_ERR_UNSUPPORTED;
  }
  vt_col[B] = static_cast<int32_t>(col);
  int device = 0, sms = 0;
  if ((st = num_sms(&device, &sms)) != GDPA_OK) return st;
  DeviceCtx& c = ctx(device);
  std::lock_guard<std::mutex> lock(c.mu);
  if ((st = c.init()) != GDPA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int num_ctas = 0, rpi = 0, kvt = 0;
  int64_t n_items = 0;
  if ((st = plan_and_upload(c, h_q_offsets, h_kv_offsets, B, H, D, 0, sms, s, &num_ctas, &rpi, &kvt, &n_items,
                            false, true, &vt_col)) != GDPA_OK)
    return st;
  // with no keys nothing of k or v is read
  return launch_with_ctx(c, q8, Tkv > 0 ? k8 : q8, Tkv > 0 ? vt8 : q8, out, q_offsets, kv_offsets, Tq, Tkv, H, D,
                         act, 0, scale, num_ctas, rpi, kvt, n_items, s, lse, q_sf, k_sf ? k_sf : q_sf, vt_sf, col);
}

namespace gdpa {
namespace {

// The backward with the internal window code (0 full, > 0 block window,
// < 0 sliding window of -window tokens); shape already validated.
gdpa_status_t bwd_impl(const void* q, const void* k, const void* v, const void* out, const void* dout,
                       const float* lse, const int32_t* h_q_offsets, const int32_t* h_kv_offsets,
                       const int32_t* q_offsets, const int32_t* kv_offsets, int B, int H, int D, int act, int window,
                       float scale, void* dq, void* dk, void* dv, void* stream) {
  gdpa_status_t st;
  if (B == 0) return GDPA_OK;
  int64_t Tq = 0, Tkv = 0;
  if ((st = validate_offsets(h_q_offsets, h_kv_offsets, B, window, &Tq, &Tkv)) != GDPA_OK) return st;
  if (Tq >= (int64_t)1 << 31 || Tkv >= (int64_t)1 << 31) return GDPA_ERR_UNSUPPORTED;
  if (Tq > 0 && (!q || !dq || !aligned16(q) || !aligned16(dq))) return GDPA_ERR_INVALID_ARG;
  if (Tq > 0 && Tkv > 0 && (!out || !dout || !aligned16(out) || !aligned16(dout))) return GDPA_ERR_INVALID_ARG;
  if (Tq > 0 && Tkv > 0 && act == GDPA_ACT_SOFTMAX && (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0))
    return GDPA_ERR_INVALID_ARG;
  if (Tkv > 0 && (!k || !v || !dk || !dv || !aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv)))
    return GDPA_ERR_INVALID_ARG;
  if (!q_offsets || !kv_offsets) return GDPA_ERR_INVALID_ARG;
  if (Tq == 0 && Tkv == 0) return GDPA_OK;
  int device = 0, sms = 0;
  if ((st = num_sms(&device, &sms)) != GDPA_OK) return st;
  DeviceCtx& c = ctx(device);
  std::lock_guard<std::mutex> lock(c.mu);
  if ((st = c.init()) != GDPA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::vector<int32_t> dq_items, kv_items;
  try {
    plan_backward(h_q_offsets, h_kv_offsets, B, H, dq_items, kv_items);
  } catch (const std::bad_alloc&) {
    return GDPA_ERR_NO_MEMORY;
  }
  const size_t dq_bytes = dq_items.size() * sizeof(int32_t), kv_bytes = kv_items.size() * sizeof(int32_t);
  const size_t lists = align_up(dq_bytes, 16) + align_up(kv_bytes, 16);
  const size_t scratch = (size_t)Tq * H * 2 * sizeof(float);
  const size_t total = lists + scratch + 16;
  // the device buffer may still be read by an earlier backward on another stream
  if (cudaStreamWaitEvent(s, c.bwd_free, 0) != cudaSuccess) return GDPA_ERR_CUDA;
  if (c.d_bwd.cap < total) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GDPA_ERR_CUDA;
    if ((st = c.d_bwd.ensure(total)) != GDPA_OK) return st;
  }
  if (cudaEventSynchronize(c.bwd_stage_free) != cudaSuccess) return GDPA_ERR_CUDA;
  if ((st = c.h_bwd.ensure(lists + 16)) != GDPA_OK) return st;
  char* h = static_cast<char*>(c.h_bwd.p);
  if (dq_bytes) std::memcpy(h, dq_items.data(), dq_bytes);
  if (kv_bytes) std::memcpy(h + align_up(dq_bytes, 16), kv_items.data(), kv_bytes);
  char* d = static_cast<char*>(c.d_bwd.p);
  if (lists && cudaMemcpyAsync(d, h, lists, cudaMemcpyHostToDevice, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (cudaEventRecord(c.bwd_stage_free, s) != cudaSuccess) return GDPA_ERR_CUDA;
  BwdLaunchArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.q_off = q_offsets;
  a.kv_off = kv_offsets;
  a.dq_items = d;
  a.n_dq = (int64_t)(dq_items.size() / 4);
  a.kv_items = d + align_up(dq_bytes, 16);
  a.n_kv = (int64_t)(kv_items.size() / 4);
  a.scratch = reinterpret_cast<float*>(d + lists);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.Tq = Tq;
  a.Tkv = Tkv;
  a.H = H;
  a.D = D;
  a.act = act;
  a.window = window;
  a.scale = scale;
  a.stream = stream;
  if ((st = launch_backward(a)) != GDPA_OK) return st;
  return cudaEventRecord(c.bwd_free, s) == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

}  // namespace
}  // namespace gdpa

extern "C" gdpa_status_t gdpa_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                  const float* lse, const int32_t* h_q_offsets, const int32_t* h_kv_offsets,
                                  const int32_t* q_offsets, const int32_t* kv_offsets, int B, int H, int D, int act,
                                  int window_blocks, float scale, void* dq, void* dk, void* dv, void* stream) {
  gdpa_status_t st = validate_shape(B, H, D, act, window_blocks);
  if (st != GDPA_OK) return st;
  return bwd_impl(q, k, v, out, dout, lse, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act,
                  window_blocks, scale, dq, dk, dv, stream);
}

extern "C" gdpa_status_t gdpa_bwd_sliding(const void* q, const void* k, const void* v, const void* out,
                                          const void* dout, const float* lse, const int32_t* h_q_offsets,
                                          const int32_t* h_kv_offsets, const int32_t* q_offsets,
                                          const int32_t* kv_offsets, int B, int H, int D, int act, int window_tokens,
                                          float scale, void* dq, void* dk, void* dv, void* stream) {
  if (window_tokens < 1) return GDPA_ERR_INVALID_ARG;
  gdpa_status_t st = validate_shape(B, H, D, act, 1);  // as a window: softmax only
  if (st != GDPA_OK) return st;
  return bwd_impl(q, k, v, out, dout, lse, h_q_offsets, h_kv_offsets, q_offsets, kv_offsets, B, H, D, act,
                  -window_tokens, scale, dq, dk, dv, stream);
}

// The plan of gdpa_plan_create (window_blocks >= 0) and gdpa_plan_create_sliding
// (window_blocks = -window_tokens); the caller has validated the shape.
static gdpa_status_t plan_create_impl(const int32_t* h_q_offsets, const int32_t* h_kv_offsets, int B, int H, int D,
                                      int act, int window_blocks, gdpa_plan_t** plan) {
  gdpa_status_t st;
  int64_t Tq = 0, Tkv = 0;
  if ((st = validate_offsets(h_q_offsets, h_kv_offsets, B, window_blocks, &Tq, &Tkv)) != GDPA_OK) return st;
  if (Tq >= (int64_t)1 << 31 || Tkv >= (int64_t)1 << 31) return GDPA_ERR_UNSUPPORTED;
  int device = 0, sms = 0;
  if ((st = num_sms(&device, &sms)) != GDPA_OK) return st;
  gdpa_plan* P = new (std::nothrow) gdpa_plan();
  if (!P) return GDPA_ERR_NO_MEMORY;
  P->B = B;
  P->H = H;
  P->D = D;
  P->act = act;
  P->window_blocks = window_blocks;
  P->device = device;
  P->Tq = Tq;
  P->Tkv = Tkv;
  P->d_buf = nullptr;
  P->d_items = nullptr;
  P->d_cta_begin = nullptr;
  P->rows_per_item = choose_rows_per_item(h_q_offsets, B, D, window_blocks);
  P->kv_tile = choose_kv_tile(h_q_offsets, h_kv_offsets, B, window_blocks, P->rows_per_item);
  const int64_t n = B > 0 ? count_plan_items(h_q_offsets, B, H, P->rows_per_item) : 0;
  P->n_items = n;
  P->num_ctas = (int)(n < sms ? n : sms);
  if (n > 0) {
    std::vector<gdpa_work_item_t> items;
    std::vector<int32_t> cta_begin;
    try {
      st = plan_items(h_q_offsets, h_kv_offsets, B, H, window_blocks, P->rows_per_item, P->num_ctas, items,
                      cta_begin,
                      nullptr);
    } catch (const std::bad_alloc&) {
      st = GDPA_ERR_NO_MEMORY;
    }
    if (st != GDPA_OK) {
      delete P;
      return st;
    }
    const size_t items_bytes = align_up(items.size() * sizeof(gdpa_work_item_t), 16);
    const size_t total = items_bytes + cta_begin.size() * sizeof(int32_t);
    if (cudaMalloc(&P->d_buf, total) != cudaSuccess) {
      cudaGetLastError();
      delete P;
      return GDPA_ERR_NO_MEMORY;
    }
    if (cudaMemcpy(P->d_buf, items.data(), items.size() * sizeof(gdpa_work_item_t), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemcpy(static_cast<char*>(P->d_buf) + items_bytes, cta_begin.data(), cta_begin.size() * sizeof(int32_t),
                   cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaFree(P->d_buf);
      delete P;
      return GDPA_ERR_CUDA;
    }
    P->d_items = static_cast<const gdpa_work_item_t*>(P->d_buf);
    P->d_cta_begin = reinterpret_cast<const int32_t*>(static_cast<char*>(P->d_buf) + items_bytes);
  }
  *plan = P;
  return GDPA_OK;
}

extern "C" gdpa_status_t gdpa_plan_create(const int32_t* h_q_offsets, const int32_t* h_kv_offsets, int B, int H,
                                          int D, int act, int window_blocks, gdpa_plan_t** plan) {
  if (!plan) return GDPA_ERR_INVALID_ARG;
  *plan = nullptr;
  const gdpa_status_t st = validate_shape(B, H, D, act, window_blocks);
  if (st != GDPA_OK) return st;
  return plan_create_impl(h_q_offsets, h_kv_offsets, B, H, D, act, window_blocks, plan);
}

extern "C" gdpa_status_t gdpa_plan_create_sliding(const int32_t* h_q_offsets, const int32_t* h_kv_offsets, int B,
                                                  int H, int D, int act, int window_tokens, gdpa_plan_t** plan) {
  if (!plan) return GDPA_ERR_INVALID_ARG;
  *plan = nullptr;
  if (window_tokens < 1) return GDPA_ERR_INVALID_ARG;
  const gdpa_status_t st = validate_shape(B, H, D, act, 1);  // as a window: softmax only
  if (st != GDPA_OK) return st;
  return plan_create_impl(h_q_offsets, h_kv_offsets, B, H, D, act, -window_tokens, plan);
}

extern "C" gdpa_status_t gdpa_fwd_planned(const gdpa_plan_t* plan, const void* q, const void* k, const void* v,
                                          const int32_t* q_offsets, const int32_t* kv_offsets, float scale, void* out,
                                          void* stream) {
  if (!plan) return GDPA_ERR_INVALID_ARG;
  gdpa_status_t st = check_tensors(q, k, v, out, plan->Tq, plan->Tkv);
  if (st != GDPA_OK) return st;
  if (plan->n_items == 0) return GDPA_OK;
  if (!q_offsets || !kv_offsets) return GDPA_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return GDPA_ERR_CUDA;
  if (device != plan->device) return GDPA_ERR_INVALID_ARG;
  LaunchArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.q_off = q_offsets;
  a.kv_off = kv_offsets;
  a.items = plan->d_items;
  a.cta_begin = plan->d_cta_begin;
  a.num_ctas = plan->num_ctas;
  a.rows_per_item = plan->rows_per_item;
  a.kv_tile = plan->kv_tile;
  a.Tq = plan->Tq;
  a.Tkv = plan->Tkv;
  a.H = plan->H;
  a.D = plan->D;
  a.act = plan->act;
  a.window_blocks = plan->window_blocks;
  a.scale = scale;
  a.stream = stream;
  return launch_forward(a);
}

extern "C" void gdpa_plan_destroy(gdpa_plan_t* plan) {
  if (!plan) return;
  if (plan->d_buf) cudaFree(plan->d_buf);  // cudaFree waits for work that may still read it
  delete plan;
}

extern "C" int64_t gdpa_plan_num_items(const gdpa_plan_t* plan) { return plan ? plan->n_items : -1; }
extern "C" int gdpa_plan_num_ctas(const gdpa_plan_t* plan) { return plan ? plan->num_ctas : -1; }

// End-to-end call with host buffers.  The batch is cut into up to 8 chunks of
// whole sequences (~64 MB of input + output each); chunk i's inputs stream in
// on a copy stream while chunk i-1 computes on `stream` and chunk i-2's
// output streams back on a second copy stream.  Planning of each chunk runs
// on the host while the copies are in flight.
extern "C" gdpa_status_t gdpa_fwd_host(const void* h_q, const void* h_k, const void* h_v, const int32_t* h_q_offsets,
                                       const int32_t* h_kv_offsets, int B, int H, int D, int act, int window_blocks,
                                       float scale, void* h_out, void* stream) {
  gdpa_status_t st = validate_shape(B, H, D, act, window_blocks);
  if (st != GDPA_OK) return st;
  int64_t Tq = 0, Tkv = 0;
  if ((st = validate_offsets(h_q_offsets, h_kv_offsets, B, window_blocks, &Tq, &Tkv)) != GDPA_OK) return st;
  if (Tq > 0 && (!h_q || !h_out)) return GDPA_ERR_INVALID_ARG;
  if (Tkv > 0 && (!h_k || !h_v)) return GDPA_ERR_INVALID_ARG;
  if (Tq >= (int64_t)1 << 31 || Tkv >= (int64_t)1 << 31) return GDPA_ERR_UNSUPPORTED;
  if (Tq == 0) return GDPA_OK;
  int device = 0, sms = 0;
  if ((st = num_sms(&device, &sms)) != GDPA_OK) return st;
  DeviceCtx& c = ctx(device);
  std::lock_guard<std::mutex> lock(c.mu);
  if ((st = c.init()) != GDPA_OK || (st = c.init_host_path()) != GDPA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t row = (size_t)H * D * 2;
  const int32_t* qo = h_q_offsets;
  const int32_t* ko = h_kv_offsets;

  // chunk boundaries (sequence indices), balanced by bytes moved
  const double total = (double)(2 * Tq + 2 * Tkv) * (double)row;
  int C = (int)std::min<double>(kMaxChunks, std::max(1.0, std::floor(total / kChunkBytes)));
  if (C > B) C = B;
  int cut[kMaxChunks + 1];
  cut[0] = 0;
  cut[C] = B;
  {
    int b = 0;
    double acc = 0.0;
    for (int i = 1; i < C; ++i) {
      const double goal = total * i / C;
      while (b < B - (C - i) && (acc < goal || b < cut[i - 1] + 1)) {
        acc += (double)(2 * (qo[b + 1] - qo[b]) + 2 * (ko[b + 1] - ko[b])) * (double)row;
        ++b;
      }
      cut[i] = b;
    }
  }
  // per-chunk sizes of the rebased offsets and work lists
  int64_t n_items[kMaxChunks];
  int ctas[kMaxChunks];
  int rpi[kMaxChunks], kvt[kMaxChunks];
  size_t off_at[kMaxChunks], work_at[kMaxChunks], item_bytes[kMaxChunks];
  size_t meta = 0;
  for (int i = 0; i < C; ++i) {
    const int nb = cut[i + 1] - cut[i];
    // rows per item depend only on the lengths, which rebasing keeps
    std::vector<int32_t> tmp(nb + 1);
    for (int b = 0; b <= nb; ++b) tmp[b] = qo[cut[i] + b] - qo[cut[i]];
    rpi[i] = choose_rows_per_item(tmp.data(), nb, D, window_blocks);
    {
      std::vector<int32_t> tmpk(nb + 1);
      for (int b = 0; b <= nb; ++b) tmpk[b] = ko[cut[i] + b] - ko[cut[i]];
      kvt[i] = choose_kv_tile(tmp.data(), tmpk.data(), nb, window_blocks, rpi[i]);
    }
    const int64_t n = count_plan_items(tmp.data(), nb, H, rpi[i]);
    n_items[i] = n;
    ctas[i] = (int)(n < sms ? n : sms);
    off_at[i] = meta;
    meta += align_up(2 * ((size_t)nb + 1) * sizeof(int32_t), 256);
    work_at[i] = meta;
    item_bytes[i] = align_up((size_t)n * sizeof(gdpa_work_item_t), 16);
    meta += align_up(item_bytes[i] + ((size_t)ctas[i] + 1) * sizeof(int32_t), 256);
  }
  const size_t bq = align_up((size_t)Tq * row, 256), bkv = align_up((size_t)Tkv * row, 256);
  const size_t need = 2 * bq + 2 * bkv + meta;
  if (c.d_io.cap < need) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GDPA_ERR_CUDA;
    if ((st = c.d_io.ensure(need)) != GDPA_OK) return st;
  }
  if ((st = c.h_io.ensure(meta)) != GDPA_OK) return st;
  char* base = static_cast<char*>(c.d_io.p);
  char* dq = base;
  char* dout = base + bq;
  char* dk = base + 2 * bq;
  char* dv = base + 2 * bq + bkv;
  char* dmeta = base + 2 * bq + 2 * bkv;
  char* hmeta = static_cast<char*>(c.h_io.p);

  // All copies in run in order on one copy stream: chunk 0's inputs, then
  // every chunk's offsets and work list in one piece, then the other chunks'
  // inputs; chunk i computes as soon as its inputs are in and copies out on a
  // second copy stream, so the host link carries inputs and outputs at once.
  // (A work list uploaded later on the compute stream would queue behind all
  // the input copies on the same copy engine and hold every kernel back.)
  if (cudaEventRecord(c.ev_start, s) != cudaSuccess || cudaStreamWaitEvent(c.s_in, c.ev_start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(c.s_out, c.ev_start, 0) != cudaSuccess)
    return GDPA_ERR_CUDA;
  auto copy_in = [&](int i) -> gdpa_status_t {
    const size_t q0 = (size_t)qo[cut[i]] * row, q1 = (size_t)qo[cut[i + 1]] * row;
    const size_t k0 = (size_t)ko[cut[i]] * row, k1 = (size_t)ko[cut[i + 1]] * row;
    if (q1 > q0 &&
        cudaMemcpyAsync(dq + q0, static_cast<const char*>(h_q) + q0, q1 - q0, cudaMemcpyHostToDevice, c.s_in) !=
            cudaSuccess)
      return GDPA_ERR_CUDA;
    if (k1 > k0) {
      if (cudaMemcpyAsync(dk + k0, static_cast<const char*>(h_k) + k0, k1 - k0, cudaMemcpyHostToDevice, c.s_in) !=
              cudaSuccess ||
          cudaMemcpyAsync(dv + k0, static_cast<const char*>(h_v) + k0, k1 - k0, cudaMemcpyHostToDevice, c.s_in) !=
              cudaSuccess)
        return GDPA_ERR_CUDA;
    }
    return cudaEventRecord(c.ev_in[i], c.s_in) == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
  };
  if ((st = copy_in(0)) != GDPA_OK) return st;
  // plan every chunk on the host while chunk 0 travels
  std::vector<gdpa_work_item_t> items;
  std::vector<int32_t> cta_begin;
  for (int i = 0; i < C; ++i) {
    const int b0 = cut[i], nb = cut[i + 1] - cut[i];
    int32_t* hqo = reinterpret_cast<int32_t*>(hmeta + off_at[i]);
    int32_t* hko = hqo + nb + 1;
    for (int b = 0; b <= nb; ++b) {
      hqo[b] = qo[b0 + b] - qo[b0];
      hko[b] = ko[b0 + b] - ko[b0];
    }
    if (n_items[i] > 0) {
      try {
        st = plan_items(hqo, hko, nb, H, window_blocks, rpi[i], ctas[i], items, cta_begin, nullptr);
      } catch (const std::bad_alloc&) {
        st = GDPA_ERR_NO_MEMORY;
      }
      if (st != GDPA_OK) return st;
      std::memcpy(hmeta + work_at[i], items.data(), items.size() * sizeof(gdpa_work_item_t));
      std::memcpy(hmeta + work_at[i] + item_bytes[i], cta_begin.data(), cta_begin.size() * sizeof(int32_t));
    }
  }
  if (cudaMemcpyAsync(dmeta, hmeta, meta, cudaMemcpyHostToDevice, c.s_in) != cudaSuccess ||
      cudaEventRecord(c.ev_meta, c.s_in) != cudaSuccess || cudaStreamWaitEvent(s, c.ev_meta, 0) != cudaSuccess)
    return GDPA_ERR_CUDA;
  for (int i = 1; i < C; ++i)
    if ((st = copy_in(i)) != GDPA_OK) return st;
  for (int i = 0; i < C; ++i) {
    const int b0 = cut[i], nb = cut[i + 1] - cut[i];
    const int32_t* hqo = reinterpret_cast<const int32_t*>(hmeta + off_at[i]);
    const int64_t Tq_i = hqo[nb], Tkv_i = hqo[2 * nb + 1];
    if (cudaStreamWaitEvent(s, c.ev_in[i], 0) != cudaSuccess) return GDPA_ERR_CUDA;
    if (n_items[i] > 0) {
      LaunchArgs a;
      a.q = dq + (size_t)qo[b0] * row;
      a.k = dk + (size_t)ko[b0] * row;
      a.v = dv + (size_t)ko[b0] * row;
      a.out = dout + (size_t)qo[b0] * row;
      a.q_off = reinterpret_cast<const int32_t*>(dmeta + off_at[i]);
      a.kv_off = a.q_off + nb + 1;
      a.items = reinterpret_cast<const gdpa_work_item_t*>(dmeta + work_at[i]);
      a.cta_begin = reinterpret_cast<const int32_t*>(dmeta + work_at[i] + item_bytes[i]);
      a.num_ctas = ctas[i];
      a.rows_per_item = rpi[i];
      a.kv_tile = kvt[i];
      a.Tq = Tq_i;
      a.Tkv = Tkv_i;
      a.H = H;
      a.D = D;
      a.act = act;
      a.window_blocks = window_blocks;
      a.scale = scale;
      a.stream = s;
      if ((st = launch_forward(a)) != GDPA_OK) return st;
    }
    if (cudaEventRecord(c.ev_done[i], s) != cudaSuccess || cudaStreamWaitEvent(c.s_out, c.ev_done[i], 0) != cudaSuccess)
      return GDPA_ERR_CUDA;
    if (Tq_i > 0 && cudaMemcpyAsync(static_cast<char*>(h_out) + (size_t)qo[b0] * row, dout + (size_t)qo[b0] * row,
                                    (size_t)Tq_i * row, cudaMemcpyDeviceToHost, c.s_out) != cudaSuccess)
      return GDPA_ERR_CUDA;
  }
  if (cudaStreamSynchronize(c.s_out) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return GDPA_ERR_CUDA;
  return GDPA_OK;
}

extern "C" gdpa_status_t gdpa_set_act_route(int route) {
  if (route != GDPA_ROUTE_SFU && route != GDPA_ROUTE_ALU) return GDPA_ERR_INVALID_ARG;
  set_act_route(route);
  return GDPA_OK;
}

extern "C" int gdpa_get_act_route(void) { return act_route(); }

extern "C" gdpa_status_t gdpa_act_eval(int act, const float* x, float* y, int64_t n, void* stream) {
  if (act != GDPA_ACT_SOFTMAX && act != GDPA_ACT_GELU_TANH && act != GDPA_ACT_SILU) return GDPA_ERR_INVALID_ARG;
  if (n < 0 || (n > 0 && (!x || !y))) return GDPA_ERR_INVALID_ARG;
  return launch_act_eval(act, x, y, n, stream);
}

extern "C" gdpa_status_t gdpa_device_status(void* stream) { return read_and_clear_device_status(stream); }

extern "C" gdpa_status_t gdpa_wait_selftest(int timeout_ms, void* stream) {
  if (timeout_ms < 1 || timeout_ms > 10000) return GDPA_ERR_INVALID_ARG;
  return launch_wait_selftest(timeout_ms, stream);
}

extern "C" const char* gdpa_status_string(int status) {
  switch (status) {
    case GDPA_OK: return "GDPA_OK";
    case GDPA_ERR_INVALID_ARG: return "GDPA_ERR_INVALID_ARG";
    case GDPA_ERR_UNSUPPORTED: return "GDPA_ERR_UNSUPPORTED";
    case GDPA_ERR_CUDA: return "GDPA_ERR_CUDA";
    case GDPA_ERR_DEVICE_TIMEOUT: return "GDPA_ERR_DEVICE_TIMEOUT";
    case GDPA_ERR_NO_MEMORY: return "GDPA_ERR_NO_MEMORY";
    default: return "GDPA_ERR_UNKNOWN";
  }
}

extern "C" const char* gdpa_version(void) { return "gdpa 0.1 sm_103a"; }
