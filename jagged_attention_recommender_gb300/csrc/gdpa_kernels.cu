// gdpa_kernels.cu -- kernel instantiations and launchers: TMA tensor-map
// encoding, the device status word, the activation evaluation kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "gdpa_fwd_kernel.cuh"
#include "gdpa_fwd_pair.cuh"
#include "gdpa_fwd_mxp.cuh"
#include "gdpa_fwd_pair64.cuh"
#include "gdpa_internal.h"

namespace gdpa {

namespace {
std::atomic<int> g_act_route{GDPA_ROUTE_SFU};
}  // namespace

int act_route() { return g_act_route.load(std::memory_order_relaxed); }
void set_act_route(int route) { g_act_route.store(route, std::memory_order_relaxed); }


// Device status word: bits set by kernels whose bounded waits ran out.
__device__ int g_device_status;

namespace {

constexpr int kMaxDevices = 64;

// Claim counters of the kernels that take their items at run time: one pair
// per launch, in turn from a fixed array (zero at load; the last CTA of each
// launch sets its pair back to zero), so that launches in flight at the same
// time on different streams use different pairs unless more than
// kClaimSlots of them are.
constexpr int kClaimSlots = 1024;
__device__ int g_claim_ctr[2 * kClaimSlots];

int* claim_counter(int device) {
  static std::mutex mu;
  static int* base[kMaxDevices] = {};
  static unsigned next[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (!base[device]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_claim_ctr) != cudaSuccess) return nullptr;
    base[device] = static_cast<int*>(a);
  }
  return base[device] + 2 * (next[device]++ % kClaimSlots);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 2-D view of a [rows, H, D] bf16 tensor as [rows, H*D]; boxes of
// `box_rows` rows x 64 columns (128 bytes, the swizzle width).  Rows past the
// end read as zero.
gdpa_status_t encode_rows(CUtensorMap* m, const void* base, int64_t rows, int H, int D, int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return GDPA_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * D, static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * D * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GDPA_OK : GDPA_ERR_CUDA;
}

// 2-D view of a [rows, H, 128] byte tensor (e4m3 codes) as [rows, H*128];
// boxes of `box_rows` rows x 128 bytes (the swizzle width).
gdpa_status_t encode_rows_u8(CUtensorMap* m, const void* base, int64_t rows, int H, int D, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return GDPA_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * D, static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * D};
  cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GDPA_OK : GDPA_ERR_CUDA;
}

// Key-major e4m3 V: 2-D [H*D rows, VT columns] bytes; boxes of 128 rows x
// 128 columns (the swizzle width).  Columns past VT read as zero.
gdpa_status_t encode_vt_u8(CUtensorMap* m, const void* base, int64_t VT, int H, int D) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return GDPA_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(VT), static_cast<cuuint64_t>(H) * D};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(VT)};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GDPA_OK : GDPA_ERR_CUDA;
}

int* status_ptr(int device) {
  static std::mutex mu;
  static int* ptrs[kMaxDevices] = {};
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    ptrs[device] = static_cast<int*>(p);
  }
  return ptrs[device];
}

unsigned long long wait_timeout_ns() {
  static unsigned long long ns = [] {
    const char* e = std::getenv("GDPA_WAIT_TIMEOUT_MS");
    long long ms = e ? std::atoll(e) : 0;
    if (ms <= 0) ms = 4000;
    return static_cast<unsigned long long>(ms) * 1000000ull;
  }();
  return ns;
}

// `min_regs`: a kernel that moves registers between its warpgroups needs at
// least this many registers a thread at launch, or its register increase
// would wait forever; such a build is refused instead of launched.
template <typename Kernel>
gdpa_status_t launch_k(Kernel kernel, int threads, int smem, int min_regs, const FwdParams& prm, int grid,
                       cudaStream_t stream, int device, bool* attr_done, std::mutex* mu) {
  {
    std::lock_guard<std::mutex> lock(*mu);
    if (!attr_done[device]) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return GDPA_ERR_CUDA;
      if (fa.numRegs < min_regs || fa.maxThreadsPerBlock < threads) return GDPA_ERR_UNSUPPORTED;
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return GDPA_ERR_CUDA;
      attr_done[device] = true;
    }
  }
  kernel<<<grid, threads, smem, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

// Two query tiles per work item, 64-key K/V tiles with the scores
// double-buffered (block windows, short key ranges).
template <int D, int ACT, bool WIN>
gdpa_status_t launch_pair64(const FwdParams& prm, int grid, cudaStream_t stream, int device) {
  using C = Pair64Cfg<D, WIN>;
  static std::mutex mu;
  static bool attr_done[kMaxDevices] = {};
  return launch_k(gdpa_fwd_pair64_kernel<D, ACT, WIN>, C::THREADS, C::SMEM_BYTES, C::MIN_LAUNCH_REGS, prm, grid,
                  stream, device, attr_done, &mu);
}

// One query tile per work item; MODE: full attention, block window or key
// split (at most 32 queries, the key range split over the four warps).
template <int D, int ACT, int MODE>
gdpa_status_t launch_t(const FwdParams& prm, int grid, cudaStream_t stream, int device) {
  using C = FwdCfg<D, MODE>;
  static std::mutex mu;
  static bool attr_done[kMaxDevices] = {};
  return launch_k(gdpa_fwd_kernel<D, ACT, MODE>, C::THREADS, C::SMEM_BYTES, C::MIN_LAUNCH_REGS, prm, grid, stream,
                  device, attr_done, &mu);
}

template <int D>
gdpa_status_t launch_single(int act, int mode, const FwdParams& prm, int grid, cudaStream_t s, int device) {
  const bool gelu = act != GDPA_ACT_SOFTMAX;  // the ALU activations
  switch (mode) {
    case kModeFull:
      return gelu ? launch_t<D, kActGelu, kModeFull>(prm, grid, s, device)
                  : launch_t<D, kActSoftmax, kModeFull>(prm, grid, s, device);
    case kModeWindow:  // softmax only (validated on entry)
      return launch_t<D, kActSoftmax, kModeWindow>(prm, grid, s, device);
    default:
      return GDPA_ERR_INVALID_ARG;
  }
}

// Two query tiles per work item, 128-key K/V tiles (long key ranges).
template <int D, int ACT, bool WIN>
gdpa_status_t launch_pair(const FwdParams& prm, int grid, cudaStream_t stream, int device) {
  using C = PairCfg<D>;
  static std::mutex mu;
  static bool attr_done[kMaxDevices] = {};
  return launch_k(gdpa_fwd_pair_kernel<D, ACT, WIN>, C::THREADS, C::SMEM_BYTES, C::MIN_LAUNCH_REGS, prm, grid, stream,
                  device, attr_done, &mu);
}

// Q, K and V in MXFP8, P rounded to MXFP8 on chip (softmax, D = 128).
gdpa_status_t launch_mxp(const FwdParams& prm, int grid, cudaStream_t stream, int device) {
  static std::mutex mu;
  static bool attr_done[kMaxDevices] = {};
  return launch_k(gdpa_fwd_mxp_kernel, MxpCfg::THREADS, MxpCfg::SMEM_BYTES, MxpCfg::MIN_LAUNCH_REGS, prm, grid, stream,
                  device, attr_done, &mu);
}

// Evaluates the activation exactly as the kernels do: GELU two arguments at
// a time with the packed evaluation of the given sigma route, exp2 on the
// special-function unit.
__global__ void act_eval_kernel(int act, int sfu, const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  for (int64_t i = 2 * (blockIdx.x * (int64_t)blockDim.x + threadIdx.x); i < n;
       i += 2 * (int64_t)gridDim.x * blockDim.x) {
    if (act != kActSoftmax) {
      float a, b, A, C;
      alu_act_consts(act == GDPA_ACT_SILU, 1.0f, A, C);
      act_eval2(act_k(A, C, sfu), x[i], i + 1 < n ? x[i + 1] : 0.0f, a, b);
      y[i] = a;
      if (i + 1 < n) y[i + 1] = b;
    } else {
      y[i] = ptx::ex2_approx(x[i]);
      if (i + 1 < n) y[i + 1] = ptx::ex2_approx(x[i + 1]);
    }
  }
}

// One thread waits, with the forward kernel's bounded wait, on an mbarrier
// that nothing ever arrives on; when the limit runs out it records the
// timeout in the status word exactly as the forward kernel's roles do.
__global__ void wait_selftest_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  ptx::mbar_init(&bar, 1);
  abort_flag = 0;
  ptx::fence_mbar_init();
  if (!ptx::mbar_wait(&bar, 0, limit_ns, &abort_flag)) atomicOr(status, kStatusActivation);
}

}  // namespace

// Shared with the backward launcher (gdpa_bwd.cu).
gdpa_status_t encode_rows_2d(CUtensorMap* m, const void* base, int64_t rows, int H, int D, int box_rows) {
  return encode_rows(m, base, rows, H, D, box_rows);
}
int* device_status_word(int device) { return status_ptr(device); }
unsigned long long bounded_wait_ns() { return wait_timeout_ns(); }

gdpa_status_t launch_wait_selftest(int timeout_ms, void* stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return GDPA_ERR_CUDA;
  int* status = status_ptr(device);
  if (!status) return GDPA_ERR_CUDA;
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      status, static_cast<unsigned long long>(timeout_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

gdpa_status_t launch_forward(const LaunchArgs& a) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return GDPA_ERR_CUDA;
  if (device < 0 || device >= kMaxDevices) return GDPA_ERR_UNSUPPORTED;
  if (a.num_ctas <= 0 || a.Tq <= 0) return GDPA_OK;
  int* status = status_ptr(device);
  if (!status) return GDPA_ERR_CUDA;
  FwdParams prm;
  prm.vt_col = nullptr;
  prm.vt_sf = nullptr;
  prm.vt_blocks = 0;
  const bool key_split = a.rows_per_item == kKeySplitRows;
  const bool mx = a.q_sf != nullptr;
  if (mx && a.vt_col) {  // all three inputs in MXFP8
    if (a.D != 128 || a.rows_per_item != 2 * kBlockM || a.kv_tile != kBlockN / 2 || a.window_blocks != 0 ||
        a.act != GDPA_ACT_SOFTMAX || !a.k_sf || (a.Tkv > 0 && !a.vt_sf) || a.VT >= ((int64_t)1 << 31))
      return GDPA_ERR_INVALID_ARG;
    gdpa_status_t st = encode_rows_u8(&prm.tm_q, a.q, a.Tq, a.H, a.D, kBlockM);
    if (st != GDPA_OK) return st;
    if (a.Tkv > 0) {
      if ((st = encode_rows_u8(&prm.tm_k, a.k, a.Tkv, a.H, a.D, MxpCfg::KB)) != GDPA_OK) return st;
      if ((st = encode_vt_u8(&prm.tm_v, a.v, a.VT, a.H, a.D)) != GDPA_OK) return st;
    } else {  // nothing is loaded; maps over Q's codes keep the descriptors valid
      if ((st = encode_rows_u8(&prm.tm_k, a.q, a.Tq, a.H, a.D, MxpCfg::KB)) != GDPA_OK) return st;
      if ((st = encode_rows_u8(&prm.tm_v, a.q, a.Tq, a.H, a.D, kBlockM)) != GDPA_OK) return st;
    }
    prm.q_sf = static_cast<const uint32_t*>(a.q_sf);
    prm.k_sf = static_cast<const uint32_t*>(a.k_sf);
    prm.vt_col = a.vt_col;
    prm.vt_sf = static_cast<const uint8_t*>(a.vt_sf);
    prm.vt_blocks = static_cast<int>(a.VT / 32);
    prm.items = reinterpret_cast<const int4*>(a.items);
    prm.cta_begin = a.cta_begin;
    prm.q_off = a.q_off;
    prm.kv_off = a.kv_off;
    prm.out = static_cast<__nv_bfloat16*>(a.out);
    prm.status = status;
    prm.timeout_ns = wait_timeout_ns();
    prm.H = a.H;
    prm.window_blocks = 0;
    prm.score_scale = a.scale * 1.4426950408889634f;
    prm.out_align32 = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0 ? 1 : 0;
    prm.lse = a.lse;
    prm.Tq = static_cast<int>(a.Tq);
    prm.Tkv = static_cast<int>(a.Tkv);
    prm.test_skip_arrive = 0;
    alu_act_consts(false, a.scale, prm.act_a, prm.act_c);
    return launch_mxp(prm, a.num_ctas, static_cast<cudaStream_t>(a.stream), device);
  }
  if (mx && (a.D != 128 || a.rows_per_item != kBlockM || a.kv_tile != kBlockN || a.window_blocks != 0 || !a.k_sf))
    return GDPA_ERR_INVALID_ARG;
  gdpa_status_t st = mx ? encode_rows_u8(&prm.tm_q, a.q, a.Tq, a.H, a.D, kBlockM)
                        : encode_rows(&prm.tm_q, a.q, a.Tq, a.H, a.D, key_split ? kKeySplitRows : kBlockM);
  if (st != GDPA_OK) return st;
  // With no keys at all no K/V tile is ever loaded; any valid address will do.
  const void* kb = a.Tkv > 0 ? a.k : a.q;
  const void* vb = a.Tkv > 0 ? a.v : a.q;
  const int64_t kv_rows = a.Tkv > 0 ? a.Tkv : a.Tq;
  if (a.kv_tile != kBlockN && !(a.kv_tile == kBlockN / 2 && a.rows_per_item == 2 * kBlockM)) return GDPA_ERR_INVALID_ARG;
  const int kv_box = a.kv_tile;  // rows of a K/V tile the kernel stages
  if (mx) {
    if (a.Tkv > 0) {
      if ((st = encode_rows_u8(&prm.tm_k, a.k, a.Tkv, a.H, a.D, kv_box)) != GDPA_OK) return st;
      if ((st = encode_rows(&prm.tm_v, a.v, a.Tkv, a.H, a.D, kv_box)) != GDPA_OK) return st;
    } else {  // nothing is loaded; maps over Q's codes keep the descriptors valid
      if ((st = encode_rows_u8(&prm.tm_k, a.q, a.Tq, a.H, a.D, kv_box)) != GDPA_OK) return st;
      if ((st = encode_rows_u8(&prm.tm_v, a.q, a.Tq, a.H, a.D, kv_box)) != GDPA_OK) return st;
    }
  } else {
    if ((st = encode_rows(&prm.tm_k, kb, kv_rows, a.H, a.D, kv_box)) != GDPA_OK) return st;
    if ((st = encode_rows(&prm.tm_v, vb, kv_rows, a.H, a.D, kv_box)) != GDPA_OK) return st;
  }
  prm.q_sf = static_cast<const uint32_t*>(a.q_sf);
  prm.k_sf = static_cast<const uint32_t*>(a.k_sf);
  prm.items = reinterpret_cast<const int4*>(a.items);
  prm.cta_begin = a.cta_begin;
  prm.q_off = a.q_off;
  prm.kv_off = a.kv_off;
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.status = status;
  prm.timeout_ns = wait_timeout_ns();
  prm.H = a.H;
  prm.window_blocks = a.window_blocks;
  prm.score_scale = a.act == GDPA_ACT_SOFTMAX ? a.scale * 1.4426950408889634f : a.scale;
  prm.out_align32 = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0 ? 1 : 0;
  prm.lse = a.lse;
  prm.Tq = static_cast<int>(a.Tq);
  prm.Tkv = static_cast<int>(a.Tkv);
  prm.test_skip_arrive = fault_injected("skip_arrive") ? 1 : 0;
  alu_act_consts(a.act == GDPA_ACT_SILU, a.scale, prm.act_a, prm.act_c);
  prm.act_sfu = act_route() == GDPA_ROUTE_SFU ? 1 : 0;
  prm.item_ctr = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(a.stream);
  const bool win = a.window_blocks != 0;
  // sliding windows (window_blocks < 0) exist only in the 64-key pair kernel
  if (a.window_blocks < 0 && !(a.rows_per_item == 256 && a.kv_tile == kBlockN / 2)) return GDPA_ERR_INVALID_ARG;
  // the pair kernels (256-row items) claim their items at run time
  if (a.rows_per_item == 256 && !mx && !(prm.item_ctr = claim_counter(device))) return GDPA_ERR_CUDA;
  prm.out_tma = 0;
  if (a.rows_per_item == 256 && a.kv_tile == kBlockN / 2) {
    // with windows the 64-key kernel stores whole 128-row output tiles in bulk
    if (win) prm.out_tma = encode_rows(&prm.tm_o, a.out, a.Tq, a.H, a.D, 128) == GDPA_OK ? 1 : 0;
    if (win) {  // softmax only (validated on entry)
      if (a.D == 128) return launch_pair64<128, kActSoftmax, true>(prm, a.num_ctas, s, device);
      if (a.D == 64) return launch_pair64<64, kActSoftmax, true>(prm, a.num_ctas, s, device);
      return GDPA_ERR_UNSUPPORTED;
    }
    if (a.D == 128)
      return a.act != GDPA_ACT_SOFTMAX ? launch_pair64<128, kActGelu, false>(prm, a.num_ctas, s, device)
                                         : launch_pair64<128, kActSoftmax, false>(prm, a.num_ctas, s, device);
    if (a.D == 64)
      return a.act != GDPA_ACT_SOFTMAX ? launch_pair64<64, kActGelu, false>(prm, a.num_ctas, s, device)
                                         : launch_pair64<64, kActSoftmax, false>(prm, a.num_ctas, s, device);
    return GDPA_ERR_UNSUPPORTED;
  }
  if (a.rows_per_item == 256) {
    if (win) return GDPA_ERR_INVALID_ARG;  // windows take 64-key tiles
    if (a.D == 128)
      return a.act != GDPA_ACT_SOFTMAX ? launch_pair<128, kActGelu, false>(prm, a.num_ctas, s, device)
                                         : launch_pair<128, kActSoftmax, false>(prm, a.num_ctas, s, device);
    if (a.D == 64)
      return a.act != GDPA_ACT_SOFTMAX ? launch_pair<64, kActGelu, false>(prm, a.num_ctas, s, device)
                                         : launch_pair<64, kActSoftmax, false>(prm, a.num_ctas, s, device);
    return GDPA_ERR_UNSUPPORTED;
  }
  if (key_split) {
    if (win || a.D != 64) return GDPA_ERR_INVALID_ARG;
    return a.act != GDPA_ACT_SOFTMAX ? launch_t<64, kActGelu, kModeKeySplit>(prm, a.num_ctas, s, device)
                                       : launch_t<64, kActSoftmax, kModeKeySplit>(prm, a.num_ctas, s, device);
  }
  if (a.rows_per_item != kBlockM) return GDPA_ERR_INVALID_ARG;
  if (mx)
    return a.act != GDPA_ACT_SOFTMAX ? launch_t<128, kActGelu, kModeFullMx>(prm, a.num_ctas, s, device)
                                       : launch_t<128, kActSoftmax, kModeFullMx>(prm, a.num_ctas, s, device);
  const int mode = win ? kModeWindow : kModeFull;
  if (a.D == 128) return launch_single<128>(a.act, mode, prm, a.num_ctas, s, device);
  if (a.D == 64) return launch_single<64>(a.act, mode, prm, a.num_ctas, s, device);
  return GDPA_ERR_UNSUPPORTED;
}

gdpa_status_t launch_act_eval(int act, const float* x, float* y, int64_t n, void* stream) {
  if (act != GDPA_ACT_SOFTMAX && act != GDPA_ACT_GELU_TANH && act != GDPA_ACT_SILU) return GDPA_ERR_INVALID_ARG;
  if (n <= 0) return GDPA_OK;
  const int threads = 256;
  const int64_t want = (n + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 4096 ? want : 4096);
  act_eval_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(act, act_route() == GDPA_ROUTE_SFU ? 1 : 0,
                                                                             x, y, n);
  return cudaGetLastError() == cudaSuccess ? GDPA_OK : GDPA_ERR_CUDA;
}

gdpa_status_t read_and_clear_device_status(void* stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return GDPA_ERR_CUDA;
  int* status = status_ptr(device);
  if (!status) return GDPA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDPA_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GDPA_ERR_CUDA;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return GDPA_ERR_CUDA;
    // a wait that ran out outranks a bad plan (which a timeout can follow from)
    return (h & ~kStatusBadPlan) ? GDPA_ERR_DEVICE_TIMEOUT : GDPA_ERR_INVALID_ARG;
  }
  return GDPA_OK;
}

}  // namespace gdpa
