// gdpa_fwd_common.cuh -- what both forward kernels share: the launch
// parameter block, the activation and status codes, and the row store.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "gelu_alu.cuh"
#include "sm103_ptx.cuh"

namespace gdpa {

struct FwdParams {  // CUtensorMap members carry their own 64+ byte alignment
  CUtensorMap tm_q;  // 2-D view [T, H*D] bf16, box 64 x 128, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  const int4* items;         // work items grouped by CTA: {seq, head, q0, kv0}
  const int32_t* cta_begin;  // [gridDim.x + 1]
  const int32_t* q_off;
  const int32_t* kv_off;
  __nv_bfloat16* out;
  int* status;               // device status word (bit set on a wait timeout)
  unsigned long long timeout_ns;
  int H;
  int window_blocks;
  float score_scale;         // softmax: scale * log2(e); GELU: scale
  int out_align32;           // out is 32-byte aligned: 32-byte stores allowed
  float* lse;                // optional [Tq, H]: softmax row logsumexp (natural log) for the backward
  float act_a, act_c;        // ALU activations: folded constants (alu_act_consts)
  int act_sfu;               // ALU activations: 1 = sigma on the special-function unit, 0 = the FMA polynomial
  // MXFP8 Q and K (tm_q, tm_k then view e4m3 codes): per (token, head) one
  // 32-bit word of four E8M0 scales, block b of D in byte b
  const uint32_t* q_sf;
  const uint32_t* k_sf;
  int Tq, Tkv;               // rows of q / out and of k / v: device offsets beyond them are a bad plan
  int test_skip_arrive;      // failure-path test only: one activation warp of CTA 0 skips one arrive
  // MXFP8 V, key-major (tm_v then views the codes [H*D, VT]): first column
  // of each sequence [B+1], E8M0 scales [VT/32, H*D], VT/32
  const int32_t* vt_col;
  const uint8_t* vt_sf;
  int vt_blocks;
};

// kActGelu instantiates the ALU activations (tanh-GELU and SiLU, told apart
// by the constants act_a / act_c the launcher passes).
enum : int { kActSoftmax = 0, kActGelu = 1 };

enum : int { kStatusProducer = 1, kStatusMma = 2, kStatusActivation = 4, kStatusEpilogue = 8, kStatusBadPlan = 16 };

// Rows a work item may touch, from the device offsets of its sequence,
// clipped to the tensors the launch was given: a plan used with offsets it
// was not built from (or offsets past the tensors) can then only read rows
// that exist -- TMA fills the rest with zeros -- and never writes outside
// `out`.  Every role clips the same way; the one decode with FLAG (the Q/K
// producer's) flags the launch with kStatusBadPlan.  Returns {first row,
// rows} for Q/O (rows counted from qs + q0) and K/V.
struct ItemRows {
  int qs, ks, Lq, Lkv;
};
// A sequence's device offsets [qs, qe) and [ks, ke).
struct SeqOffs {
  int qs, qe, ks, ke;
};
__device__ __forceinline__ SeqOffs load_seq_offs(const FwdParams& p, int b) {
  return SeqOffs{__ldg(p.q_off + b), __ldg(p.q_off + b + 1), __ldg(p.kv_off + b), __ldg(p.kv_off + b + 1)};
}
template <bool FLAG = false>
__device__ __forceinline__ ItemRows item_rows_from(const FwdParams& p, const SeqOffs& o) {
  const int qs = o.qs, qe = o.qe, ks = o.ks, ke = o.ke;
  ItemRows r;
  r.qs = qs;
  r.ks = ks;
  r.Lq = min(qe, p.Tq) - qs;
  r.Lkv = min(ke, p.Tkv) - ks;
  if (qs < 0 || ks < 0 || qe > p.Tq || ke > p.Tkv || r.Lq < 0 || r.Lkv < 0) {
    if (FLAG) atomicOr(p.status, kStatusBadPlan);
    r.Lq = max(r.Lq, 0);
    r.Lkv = max(r.Lkv, 0);
    if (qs < 0 || qs > p.Tq) r.Lq = 0;
    if (ks < 0 || ks > p.Tkv) r.Lkv = 0;
  }
  return r;
}
template <bool FLAG = false>
__device__ __forceinline__ ItemRows item_rows(const FwdParams& p, int b) {
  return item_rows_from<FLAG>(p, load_seq_offs(p, b));
}

// Work-item descriptors loaded ahead of their use: the raw item two ahead
// and the sequence offsets of the item one ahead, so that neither of the two
// dependent global loads of a decode sits on a role's critical path.
struct ItemPrefetch {
  int4 raw1, raw2;  // items idx + 1, idx + 2
  SeqOffs offs1;    // offsets of item idx + 1's sequence
};
// Loads for the first item [ibeg] (and starts the pipeline); returns its
// descriptor and offsets through it0 / offs0.
__device__ __forceinline__ ItemPrefetch item_prefetch_start(const FwdParams& p, int ibeg, int iend, int4& it0,
                                                            SeqOffs& offs0) {
  ItemPrefetch f;
  it0 = ibeg < iend ? __ldg(p.items + ibeg) : make_int4(0, 0, 0, 0);
  f.raw1 = ibeg + 1 < iend ? __ldg(p.items + ibeg + 1) : make_int4(0, 0, 0, 0);
  offs0 = load_seq_offs(p, it0.x);
  f.raw2 = ibeg + 2 < iend ? __ldg(p.items + ibeg + 2) : make_int4(0, 0, 0, 0);
  f.offs1 = load_seq_offs(p, f.raw1.x);
  return f;
}
// Moves the pipeline on by one item (call once the current item idx has
// been decoded): item idx + 1 becomes current, and the loads for idx + 2 and
// idx + 3 are issued.
__device__ __forceinline__ void item_prefetch_next(const FwdParams& p, ItemPrefetch& f, int idx, int iend, int4& it,
                                                   SeqOffs& offs) {
  it = f.raw1;
  offs = f.offs1;
  f.raw1 = f.raw2;
  f.offs1 = load_seq_offs(p, f.raw1.x);
  f.raw2 = idx + 3 < iend ? __ldg(p.items + idx + 3) : make_int4(0, 0, 0, 0);
}

// 32 bf16 values (16 packed words) to global memory: two 32-byte stores when
// `v8` (the address is 32-byte aligned), else four 16-byte stores.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&pk)[16], bool v8) {
  if (v8) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(pk[0]), "r"(pk[1]), "r"(pk[2]),
                 "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7])
                 : "memory");
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + 16), "r"(pk[8]), "r"(pk[9]),
                 "r"(pk[10]), "r"(pk[11]), "r"(pk[12]), "r"(pk[13]), "r"(pk[14]), "r"(pk[15])
                 : "memory");
  } else {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  }
}

// Natural-log row logsumexp from the log2-domain running max m and sum l
// (sum_j 2^(x_j - m) = l): ln 2 (m + log2 l); -inf for an empty row.
__device__ __forceinline__ float row_lse(float m, float l) {
  return l > 0.0f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
}

__device__ __forceinline__ void report_failure(const FwdParams& p, volatile int* abort, int bit) {
  *abort = 1;
  atomicOr(p.status, bit);
}

}  // namespace gdpa
