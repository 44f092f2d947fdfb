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
  // Run-time claiming of work items (kernels that take it): [0] the next
  // claim, [1] CTAs finished; the last CTA to finish sets both back to 0.
  int* item_ctr;
  // The output as a 2-D view [Tq, H*D] bf16, box 64 x 128, 128-byte swizzle,
  // for bulk tensor stores of whole 128-row tiles (64-key pair kernel);
  // out_tma = 0: rows are stored by the threads.
  CUtensorMap tm_o;
  int out_tma;
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

// ------------------------------------------------------------------ run-time work claiming
//
// The host plan gives each CTA a list of items (longest-processing-time
// assignment, each list in decreasing cost).  Kernels that claim at run time
// walk those lists interleaved -- claim k is position k / G of list k % G
// (G = gridDim.x), so the claims run through the items in roughly decreasing
// cost -- and each CTA takes the next claim when it is ready for another
// item: a CTA that runs slow (or was given more) hands its remaining items
// to the others, which is greedy list scheduling in longest-first order.
// One thread of the CTA (the claimer) takes the claims, decodes each item and
// publishes it in a ring of shared-memory slots that every role of the CTA
// reads in the same order; a slot is refilled once every reader has
// released it.
constexpr int kRing = 4;

template <typename Item>
struct ItemRing {
  Item slot[kRing];
  int live[kRing];         // 0: the lists are exhausted
  uint64_t full[kRing];    // one arrival: the claimer published the slot
  uint64_t empty[kRing];   // one arrival per reader
};

struct ListClaim {
  int G, lmax;
};

// The longest list (a hole in a shorter one is skipped).
__device__ __forceinline__ ListClaim claim_init(const FwdParams& p) {
  ListClaim L;
  L.G = gridDim.x;
  L.lmax = 0;
  for (int c = 0; c < L.G; ++c) L.lmax = max(L.lmax, __ldg(p.cta_begin + c + 1) - __ldg(p.cta_begin + c));
  return L;
}

// The next item index, or -1 once every list is exhausted.
__device__ __forceinline__ int claim_next(const FwdParams& p, const ListClaim& L) {
  while (true) {
    const int k = atomicAdd(p.item_ctr, 1);
    const int c = k % L.G, j = k / L.G;
    if (j >= L.lmax) return -1;
    const int b0 = __ldg(p.cta_begin + c), b1 = __ldg(p.cta_begin + c + 1);
    if (b0 + j < b1) return b0 + j;
  }
}

// Claimer: waits until slot k % kRing is free, then publishes t (live) or
// the end of the lists.
template <typename Item>
__device__ __forceinline__ bool ring_publish(const FwdParams& p, ItemRing<Item>& R, uint32_t k, const Item& t,
                                             bool live, volatile int* abort) {
  const int r = k % kRing;
  if (!ptx::mbar_wait(&R.empty[r], ((k / kRing) & 1) ^ 1, p.timeout_ns, abort)) return false;
  R.slot[r] = t;
  R.live[r] = live ? 1 : 0;
  ptx::mbar_arrive(&R.full[r]);  // release: the slot's contents are visible to whoever sees the phase
  return true;
}

// Reader: entry k of the sequence.  `mask`: the lanes of the calling warp
// that read together (0 for a single-thread role); lane 0 of them -- or the
// single thread -- releases the slot for the role.  Returns false at the end
// of the lists or on a timeout (ok = false).
template <typename Item>
__device__ __forceinline__ bool ring_read(const FwdParams& p, ItemRing<Item>& R, uint32_t k, Item& t, unsigned mask,
                                          volatile int* abort, bool& ok) {
  const int r = k % kRing;
  ok = ptx::mbar_wait(&R.full[r], (k / kRing) & 1, p.timeout_ns, abort);
  if (mask) ok = __all_sync(mask, ok);
  if (!ok) return false;
  t = R.slot[r];
  const bool live = R.live[r] != 0;
  if (mask) __syncwarp(mask);
  if (!mask || (threadIdx.x & 31) == (__ffs(mask) - 1)) ptx::mbar_arrive(&R.empty[r]);
  return live;
}

// End of a claiming launch (one thread per CTA, after every role is done):
// the last CTA sets the claim counter back for the next launch that uses it.
__device__ __forceinline__ void claim_finish(const FwdParams& p) {
  __threadfence();
  if (atomicAdd(p.item_ctr + 1, 1) == (int)gridDim.x - 1) {
    atomicExch(p.item_ctr, 0);
    atomicExch(p.item_ctr + 1, 0);
  }
}

__device__ __forceinline__ void report_failure(const FwdParams& p, volatile int* abort, int bit) {
  *abort = 1;
  atomicOr(p.status, bit);
}

}  // namespace gdpa
