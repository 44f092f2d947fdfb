// gdpa_api.cu -- the C ABI of libgdpa (declared in include/gdpa.h): argument
// validation, planning, library-owned buffers, launches.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "gdpa_internal.h"

struct gdpa_plan {
  int B, H, D, act, window_blocks;
  int num_ctas;
  int device;
  int64_t n_items, Tq, Tkv;
  void* d_buf;  // work items followed by cta_begin
  const gdpa_work_item_t* d_items;
  const int32_t* d_cta_begin;
};

namespace gdpa {
namespace {

constexpr int kMaxDevices = 64;

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

// Per-device state behind gdpa_fwd / gdpa_fwd_host.
struct DeviceCtx {
  std::mutex mu;
  Buf h_stage{nullptr, 0, true};  // pinned: offsets in, work list out
  Buf d_work;                     // device work list + cta_begin
  Buf d_io;                       // gdpa_fwd_host: q, k, v, out, offsets
  cudaEvent_t stage_free = nullptr;  // host staging buffer may be overwritten
  cudaEvent_t work_free = nullptr;   // device buffers no longer read by an earlier launch
  bool events_ok = false;
  gdpa_status_t init() {
    if (events_ok) return GDPA_OK;
    if (cudaEventCreateWithFlags(&stage_free, cudaEventDisableTiming) != cudaSuccess) return GDPA_ERR_CUDA;
    if (cudaEventCreateWithFlags(&work_free, cudaEventDisableTiming) != cudaSuccess) return GDPA_ERR_CUDA;
    if (cudaEventRecord(stage_free, 0) != cudaSuccess || cudaEventRecord(work_free, 0) != cudaSuccess)
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

// Plans on the host and uploads the work list through the pinned staging
// buffer into c.d_work (both guarded by events against earlier calls).
gdpa_status_t plan_and_upload(DeviceCtx& c, const int32_t* h_q_off, const int32_t* h_kv_off, int B, int H,
                              int window_blocks, int sms, cudaStream_t stream, int* num_ctas) {
  std::vector<gdpa_work_item_t> items;
  std::vector<int32_t> cta_begin;
  int64_t n = 0;
  for (int b = 0; b < B; ++b) n += (int64_t)((h_q_off[b + 1] - h_q_off[b] + kBlockM - 1) / kBlockM) * H;
  if (n == 0) {
    *num_ctas = 0;
    return GDPA_OK;
  }
  const int ctas = (int)(n < sms ? n : sms);
  gdpa_status_t st;
  try {
    st = plan_items(h_q_off, h_kv_off, B, H, window_blocks, ctas, items, cta_begin, nullptr);
  } catch (const std::bad_alloc&) {
    return GDPA_ERR_NO_MEMORY;
  }
  if (st != GDPA_OK) return st;
  const size_t items_bytes = items.size() * sizeof(gdpa_work_item_t);
  const size_t total = align_up(items_bytes, 16) + cta_begin.size() * sizeof(int32_t);
  if (cudaStreamWaitEvent(stream, c.work_free, 0) != cudaSuccess) return GDPA_ERR_CUDA;
  if (c.d_work.cap < total) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GDPA_ERR_CUDA;  // old buffer may be in use
    if ((st = c.d_work.ensure(total)) != GDPA_OK) return st;
  }
  if (cudaEventSynchronize(c.stage_free) != cudaSuccess) return GDPA_ERR_CUDA;
  if ((st = c.h_stage.ensure(total)) != GDPA_OK) return st;
  char* h = static_cast<char*>(c.h_stage.p);
  std::memcpy(h, items.data(), items_bytes);
  std::memcpy(h + align_up(items_bytes, 16), cta_begin.data(), cta_begin.size() * sizeof(int32_t));
  if (cudaMemcpyAsync(c.d_work.p, h, total, cudaMemcpyHostToDevice, stream) != cudaSuccess) return GDPA_ERR_CUDA;
  if (cudaEventRecord(c.stage_free, stream) != cudaSuccess) return GDPA_ERR_CUDA;
  *num_ctas = ctas;
  return GDPA_OK;
}

gdpa_status_t launch_with_ctx(DeviceCtx& c, const void* q, const void* k, const void* v, void* out,
                              const int32_t* d_q_off, const int32_t* d_kv_off, int64_t Tq, int64_t Tkv, int H, int D,
                              int act, int window_blocks, float scale, int num_ctas, int64_t n_items,
                              cudaStream_t stream) {
  LaunchArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.q_off = d_q_off;
  a.kv_off = d_kv_off;
  a.items = static_cast<const gdpa_work_item_t*>(c.d_work.p);
  a.cta_begin = reinterpret_cast<const int32_t*>(static_cast<const char*>(c.d_work.p) +
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
  return cudaEventRecord(c.work_free, stream) == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

int64_t count_items(const int32_t* h_q_off, int B, int H) {
  int64_t n = 0;
  for (int b = 0; b < B; ++b) n += (int64_t)((h_q_off[b + 1] - h_q_off[b] + kBlockM - 1) / kBlockM) * H;
  return n;
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
  if (cudaEventSynchronize(c.stage_free) != cudaSuccess) return GDPA_ERR_CUDA;
  if ((st = c.h_stage.ensure(2 * ob)) != GDPA_OK) return st;
  int32_t* h = static_cast<int32_t*>(c.h_stage.p);
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
  if ((st = plan_and_upload(c, hq, hk, B, H, window_blocks, sms, s, &num_ctas)) != GDPA_OK) return st;
  return launch_with_ctx(c, q, k, v, out, q_offsets, kv_offsets, Tq, Tkv, H, D, act, window_blocks, scale, num_ctas,
                         count_items(hq, B, H), s);
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
  if ((st = plan_and_upload(c, h_q_offsets, h_kv_offsets, B, H, window_blocks, sms, s, &num_ctas)) != GDPA_OK)
    return st;
  return launch_with_ctx(c, q, k, v, out, q_offsets, kv_offsets, Tq, Tkv, H, D, act, window_blocks, scale, num_ctas,
                         count_items(h_q_offsets, B, H), s);
}

extern "C" gdpa_status_t gdpa_plan_create(const int32_t* h_q_offsets, const int32_t* h_kv_offsets, int B, int H,
                                          int D, int act, int window_blocks, gdpa_plan_t** plan) {
  if (!plan) return GDPA_ERR_INVALID_ARG;
  *plan = nullptr;
  gdpa_status_t st = validate_shape(B, H, D, act, window_blocks);
  if (st != GDPA_OK) return st;
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
  const int64_t n = B > 0 ? count_items(h_q_offsets, B, H) : 0;
  P->n_items = n;
  P->num_ctas = (int)(n < sms ? n : sms);
  if (n > 0) {
    std::vector<gdpa_work_item_t> items;
    std::vector<int32_t> cta_begin;
    try {
      st = plan_items(h_q_offsets, h_kv_offsets, B, H, window_blocks, P->num_ctas, items, cta_begin, nullptr);
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
  if ((st = c.init()) != GDPA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t row = (size_t)H * D * 2;
  const size_t bq = align_up((size_t)Tq * row, 256), bkv = align_up((size_t)Tkv * row, 256);
  const size_t boff = align_up(((size_t)B + 1) * sizeof(int32_t), 256);
  const size_t total = 2 * bq + 2 * bkv + 2 * boff;
  if (c.d_io.cap < total) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GDPA_ERR_CUDA;
    if ((st = c.d_io.ensure(total)) != GDPA_OK) return st;
  }
  char* base = static_cast<char*>(c.d_io.p);
  void* dq = base;
  void* dout = base + bq;
  void* dk = base + 2 * bq;
  void* dv = base + 2 * bq + bkv;
  int32_t* dqo = reinterpret_cast<int32_t*>(base + 2 * bq + 2 * bkv);
  int32_t* dko = reinterpret_cast<int32_t*>(base + 2 * bq + 2 * bkv + boff);
  if (cudaStreamWaitEvent(s, c.work_free, 0) != cudaSuccess) return GDPA_ERR_CUDA;
  if (cudaMemcpyAsync(dq, h_q, (size_t)Tq * row, cudaMemcpyHostToDevice, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (Tkv > 0) {
    if (cudaMemcpyAsync(dk, h_k, (size_t)Tkv * row, cudaMemcpyHostToDevice, s) != cudaSuccess) return GDPA_ERR_CUDA;
    if (cudaMemcpyAsync(dv, h_v, (size_t)Tkv * row, cudaMemcpyHostToDevice, s) != cudaSuccess) return GDPA_ERR_CUDA;
  }
  const size_t ob = ((size_t)B + 1) * sizeof(int32_t);
  if (cudaMemcpyAsync(dqo, h_q_offsets, ob, cudaMemcpyHostToDevice, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (cudaMemcpyAsync(dko, h_kv_offsets, ob, cudaMemcpyHostToDevice, s) != cudaSuccess) return GDPA_ERR_CUDA;
  int num_ctas = 0;
  if ((st = plan_and_upload(c, h_q_offsets, h_kv_offsets, B, H, window_blocks, sms, s, &num_ctas)) != GDPA_OK)
    return st;
  if ((st = launch_with_ctx(c, dq, dk, dv, dout, dqo, dko, Tq, Tkv, H, D, act, window_blocks, scale, num_ctas,
                            count_items(h_q_offsets, B, H), s)) != GDPA_OK)
    return st;
  if (cudaMemcpyAsync(h_out, dout, (size_t)Tq * row, cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDPA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDPA_ERR_CUDA;
  return GDPA_OK;
}

extern "C" gdpa_status_t gdpa_act_eval(int act, const float* x, float* y, int64_t n, void* stream) {
  if (act != GDPA_ACT_SOFTMAX && act != GDPA_ACT_GELU_TANH) return GDPA_ERR_INVALID_ARG;
  if (n < 0 || (n > 0 && (!x || !y))) return GDPA_ERR_INVALID_ARG;
  return launch_act_eval(act, x, y, n, stream);
}

extern "C" gdpa_status_t gdpa_device_status(void* stream) { return read_and_clear_device_status(stream); }

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
