// gdpa_bwd.cu -- backward kernel instantiations and their launcher.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gdpa_bwd.cuh"
#include "gdpa_internal.h"

namespace gdpa {

// Defined in gdpa_kernels.cu (shared with the forward launcher).
gdpa_status_t encode_rows_2d(CUtensorMap* m, const void* base, int64_t rows, int H, int D, int box_rows);
int* device_status_word(int device);
unsigned long long bounded_wait_ns();

namespace {

constexpr int kMaxDevices = 64;

// Persistent: one CTA per SM (or per item, if fewer), each taking every
// grid-th item of the list.
template <typename Kernel>
gdpa_status_t launch_bwd_kernel(Kernel kernel, int smem, BwdParams& prm, int64_t n_items, cudaStream_t stream,
                                int device, bool* attr_done, std::mutex* mu) {
  if (n_items <= 0) return GDPA_OK;
  if (n_items > 0x7fffffffLL) return GDPA_ERR_UNSUPPORTED;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0)
    return GDPA_ERR_CUDA;
  prm.n_items = static_cast<int>(n_items);
  const int64_t grid = n_items < sms ? n_items : sms;
  {
    std::lock_guard<std::mutex> lock(*mu);
    if (!attr_done[device]) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return GDPA_ERR_CUDA;
      attr_done[device] = true;
    }
  }
  kernel<<<static_cast<unsigned>(grid), BwdCfg<128>::THREADS, smem, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

template <int D, int ACT>
gdpa_status_t launch_bwd_d(const BwdLaunchArgs& a, BwdParams& prm, cudaStream_t s, int device) {
  using C = BwdCfg<D>;
  static std::mutex mu;
  static bool dq_done[kMaxDevices] = {}, kv_done[kMaxDevices] = {};
  if (ACT == kActSoftmax && a.Tq > 0 && a.Tkv > 0) {
    const int64_t rows = a.Tq * a.H;
    gdpa_bwd_prep_kernel<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(a.out), static_cast<const __nv_bfloat16*>(a.dout), a.lse, a.scratch,
        a.scratch + rows, rows);
    if (cudaGetLastError() != cudaSuccess) return GDPA_ERR_CUDA;
  }
  prm.items = static_cast<const int4*>(a.dq_items);
  gdpa_status_t st = launch_bwd_kernel(gdpa_bwd_dq_kernel<D, ACT>, C::SMEM_BYTES, prm, a.n_dq, s, device, dq_done, &mu);
  if (st != GDPA_OK) return st;
  prm.items = static_cast<const int4*>(a.kv_items);
  return launch_bwd_kernel(gdpa_bwd_dkdv_kernel<D, ACT>, C::SMEM_BYTES, prm, a.n_kv, s, device, kv_done, &mu);
}

}  // namespace

gdpa_status_t launch_backward(const BwdLaunchArgs& a) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return GDPA_ERR_CUDA;
  if (device < 0 || device >= kMaxDevices) return GDPA_ERR_UNSUPPORTED;
  if (a.n_dq <= 0 && a.n_kv <= 0) return GDPA_OK;
  int* status = device_status_word(device);
  if (!status) return GDPA_ERR_CUDA;
  BwdParams prm;
  // An empty side is never loaded (its items return before any copy); any
  // valid address will do for its tensor map.
  const void* qb = a.Tq > 0 ? a.q : a.k;
  const void* dob = a.Tq > 0 ? a.dout : a.k;
  const void* kb = a.Tkv > 0 ? a.k : a.q;
  const void* vb = a.Tkv > 0 ? a.v : a.q;
  const int64_t qr = a.Tq > 0 ? a.Tq : a.Tkv, kr = a.Tkv > 0 ? a.Tkv : a.Tq;
  gdpa_status_t st;
  // boxes of 64 rows: a streamed tile is one box, a resident 128-row tile two
  constexpr int box = BwdCfg<128>::BN;
  if ((st = encode_rows_2d(&prm.tm_q, qb, qr, a.H, a.D, box)) != GDPA_OK) return st;
  if ((st = encode_rows_2d(&prm.tm_do, dob, qr, a.H, a.D, box)) != GDPA_OK) return st;
  if ((st = encode_rows_2d(&prm.tm_k, kb, kr, a.H, a.D, box)) != GDPA_OK) return st;
  if ((st = encode_rows_2d(&prm.tm_v, vb, kr, a.H, a.D, box)) != GDPA_OK) return st;
  prm.q_off = a.q_off;
  prm.kv_off = a.kv_off;
  prm.lse2 = a.scratch;
  prm.dvec = a.scratch + a.Tq * a.H;
  prm.dq = static_cast<__nv_bfloat16*>(a.dq);
  prm.dk = static_cast<__nv_bfloat16*>(a.dk);
  prm.dv = static_cast<__nv_bfloat16*>(a.dv);
  prm.status = status;
  prm.timeout_ns = bounded_wait_ns();
  prm.H = a.H;
  prm.window = a.window;
  prm.score_scale = a.act == GDPA_ACT_SOFTMAX ? a.scale * 1.4426950408889634f : a.scale;
  prm.scale = a.scale;
  const uintptr_t al = reinterpret_cast<uintptr_t>(a.dq) | reinterpret_cast<uintptr_t>(a.dk) |
                       reinterpret_cast<uintptr_t>(a.dv);
  prm.align32 = (al & 31u) == 0 ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(a.stream);
  const bool gelu = a.act != GDPA_ACT_SOFTMAX;  // the ALU activations
  alu_act_consts(a.act == GDPA_ACT_SILU, a.scale, prm.act_a, prm.act_c);
  prm.act_sfu = act_route() == GDPA_ROUTE_SFU ? 1 : 0;
  if (a.D == 128)
    return gelu ? launch_bwd_d<128, kActGelu>(a, prm, s, device) : launch_bwd_d<128, kActSoftmax>(a, prm, s, device);
  if (a.D == 64)
    return gelu ? launch_bwd_d<64, kActGelu>(a, prm, s, device) : launch_bwd_d<64, kActSoftmax>(a, prm, s, device);
  return GDPA_ERR_UNSUPPORTED;
}

}  // namespace gdpa
