// gdpa_bwd.cuh -- jagged GDPA backward on sm_103a: dQ, dK and dV.
//
// The gradients of the forward for an upstream gradient dO, per (sequence,
// head), with s_ij = <q_i, k_j>, x_ij = scale s_ij and dP_ij = <dO_i, v_j>:
//
//   softmax: P_ij = 2^(x_ij log2(e) - lse2_i),  dS_ij = P_ij (dP_ij - Dv_i),
//            Dv_i = <dO_i, O_i>,  lse2_i the forward's row logsumexp, log2 units
//   GELU:    P_ij = gelu(x_ij) / Lkv,             dS_ij = gelu'(x_ij) dP_ij / Lkv
//   dV = P^T dO,   dQ = scale dS K,   dK = scale dS^T Q
//
// (the backward the techfeed summary of "GEM Training" describes in its JFA
// section: dQ, dK and dV computed without atomics, parallel over batch and
// heads.)  Two persistent kernels (one CTA per SM walking every gridDim.x-th
// item of a longest-first list), each output row written once:
//
//   gdpa_bwd_dq_kernel    item = 128 query rows of one (sequence, head); it
//     walks the 64-key K/V tiles its rows may see (all, or the window's):
//     S = Q K^T and dP = dO V^T into
//     tensor memory, the activation warps turn them into dS (bf16, written
//     over S), then dQ += dS K with dS read straight from tensor memory.
//   gdpa_bwd_dkdv_kernel  item = 128 keys of one (sequence, head); it walks
//     the 64-row query tiles that may see its keys: S^T = K Q^T and
//     dP^T = V dO^T, the
//     activation warps write P^T over S^T and dS^T over dP^T, then
//     dV += P^T dO and dK += dS^T Q.
//
// S and dP are double-buffered in tensor memory and the MMA issuer runs one
// tile ahead: it issues S, dP of tile t+1 before the accumulating MMAs of
// tile t, so the tensor core works while the activation warps turn tile t's
// scores into P and dS.
//
// Threads (192): warp 0 the TMA producer, warp 1 the MMA issuer (the whole
// warp runs the loop, one elected lane issues), warps 2-5 the activation and
// the epilogue (warp w owns tensor-memory lanes 32 (w mod 4) .. +31, one row
// each).  Tensor memory (512 columns): S0 0, dP0 64, S1 128, dP1 192,
// accumulators from 256 (dQ; or dV then dK).  Shared memory (D = 128): two
// buffers of the item's two resident 128-row tiles (Q and dO, or K and V;
// the next item's load overlaps the current one) and three stages of the
// two streamed 64-row ones.
// Rows past a sequence's end are masked to P = dS = 0 in the activation, so
// whatever the TMA box brought in for them never reaches an accumulator.
#pragma once

#include "gdpa_fwd_common.cuh"

namespace gdpa {

struct BwdParams {  // CUtensorMap members carry their own 64+ byte alignment
  CUtensorMap tm_q;   // 2-D views [T, H*D] bf16, box 64 columns x 64 rows, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  const int4* items;  // {sequence, head, first row of the item in its sequence, 0}
  const int32_t* q_off;
  const int32_t* kv_off;
  const float* lse2;  // [Tq, H]: row logsumexp of the forward, log2 units (softmax)
  const float* dvec;  // [Tq, H]: <dO_i, O_i> (softmax)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
  unsigned long long timeout_ns;
  int H;
  float score_scale;  // softmax: scale * log2(e); GELU: scale
  float scale;
  int align32;        // dq, dk and dv all 32-byte aligned: 32-byte stores allowed
  float act_a, act_c; // ALU activations: folded constants (alu_act_consts)
  int act_sfu;        // ALU activations: 1 = sigma on the special-function unit, 0 = the FMA polynomial
  int window;         // 0 full; > 0 block window of that many 64-token blocks;
                      // < 0 causal sliding window of -window tokens (self attention)
  int n_items;        // items in `items`; a persistent CTA takes every gridDim.x-th
};

// First key of query i's window (both counted from the sequence start).
__device__ __forceinline__ int win_key_lo(int i, int window) {
  if (window > 0) {
    const int blk = (i >> 6) - (window - 1);
    return blk > 0 ? blk << 6 : 0;
  }
  const int lo = i + window + 1;  // i - W + 1
  return lo > 0 ? lo : 0;
}

// Last query whose window holds key j: its window starts at or before j.
__device__ __forceinline__ int win_query_hi(int j, int window) {
  const long long hi = window > 0 ? (static_cast<long long>(j >> 6) + window) * 64 - 1  // block of j plus W - 1 blocks
                                  : static_cast<long long>(j) - window - 1;           // j + W - 1
  return hi < 0x7fffffffLL ? static_cast<int>(hi) : 0x7fffffff;
}

template <int D>
struct BwdCfg {
  static constexpr int KCH = D / 64;
  static constexpr int BN = 64;                         // rows of a streamed tile
  static constexpr int NS = 3;                          // stages of the streamed tiles
  static constexpr int RCHUNK = 128 * 128;              // resident: 128 rows x 64 bf16 columns
  static constexpr int RTILE = KCH * RCHUNK;            // resident: 128 rows x D
  static constexpr int SCHUNK = BN * 128;               // streamed: 64 rows x 64 bf16 columns
  static constexpr int STILE = KCH * SCHUNK;            // streamed: 64 rows x D
  // resident tiles, two buffers (the next item's load overlaps this one):
  // buffer b holds R1 (Q for dq, K for dkdv) and R2 (dO, or V)
  __host__ __device__ static constexpr int off_r(int b, int which) { return (2 * b + which) * RTILE; }
  static constexpr int OFF_S1 = 4 * RTILE;              // streamed stages: K (dq) or Q (dkdv)
  static constexpr int OFF_S2 = OFF_S1 + NS * STILE;    // streamed stages: V (dq) or dO (dkdv)
  static constexpr int OFF_VEC = OFF_S2 + NS * STILE;   // dkdv: lse2 and Dv of a query tile, 2 buffers
  static constexpr int OFF_BAR = OFF_VEC + 2 * 2 * BN * 4;
  static constexpr int BAR_BYTES = 256;
  // at least 117 KB so that one CTA fits per SM (each allocates 512 TMEM columns)
  static constexpr int SMEM_BYTES = (OFF_BAR + BAR_BYTES + 1024) > 119808 ? (OFF_BAR + BAR_BYTES + 1024) : 119808;
  __host__ __device__ static constexpr uint32_t tm_s(int b) { return 128u * b; }       // S (or S^T) buffers
  __host__ __device__ static constexpr uint32_t tm_p(int b) { return 128u * b + 64u; } // dP (or dP^T) buffers
  static constexpr uint32_t TM_A1 = 256, TM_A2 = 256 + D;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int THREADS = 192;
  static_assert(256 + 2 * D <= TM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct BwdBars {
  uint64_t res_full[2], res_empty[2];  // resident buffers
  uint64_t st_full[3], st_empty[3];    // streamed stages
  uint64_t mma_full[2];                // S and dP of a tile are in TMEM buffer b
  uint64_t act_full[2];                // P / dS of a tile are in TMEM buffer b
  uint64_t acc_full;                   // an item's accumulating MMAs completed
  uint64_t acc_empty;                  // the epilogue has read the accumulators
  uint64_t vec_full[2];                // dkdv: lse2 / Dv of a query tile staged by the activation warps
  uint64_t drain;                      // every MMA of the CTA completed
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block");

__device__ __forceinline__ void bwd_failure(const BwdParams& p, volatile int* abort, int bit) {
  *abort = 1;
  atomicOr(p.status, bit);
}

// An item's sequence geometry.
struct BwdItem {
  int b, h, row0, q_tok, kv_tok, Lq, Lkv;
};

__device__ __forceinline__ BwdItem bwd_item(const BwdParams& p, int idx) {
  const int4 it = __ldg(p.items + idx);
  BwdItem t;
  t.b = it.x;
  t.h = it.y;
  t.row0 = it.z;
  t.q_tok = __ldg(p.q_off + t.b);
  t.Lq = __ldg(p.q_off + t.b + 1) - t.q_tok;
  t.kv_tok = __ldg(p.kv_off + t.b);
  t.Lkv = __ldg(p.kv_off + t.b + 1) - t.kv_tok;
  return t;
}

// The streamed range of an item: dq streams the keys its rows may see, dk/dv
// the queries that may see its keys (all of them, or the window's).
struct BwdWork {
  int r_row;  // first resident row (token index)
  int s_row;  // first streamed row (token index)
  int lo;     // first streamed row within the sequence
  int len;    // streamed rows
  int n;      // streamed 64-row tiles
};

template <bool DKDV>
__device__ __forceinline__ BwdWork bwd_work(const BwdParams& p, const BwdItem& t) {
  BwdWork w;
  int lo, hi;
  if (!DKDV) {  // keys: all, or from the first row's window start (64-key tile) to the last row
    lo = 0;
    hi = t.Lkv;
    if (p.window != 0) {
      lo = win_key_lo(t.row0, p.window) / 64 * 64;
      hi = min(t.Lkv, t.row0 + 128);
    }
    w.r_row = t.q_tok + t.row0;
    w.s_row = t.kv_tok + lo;
  } else {  // queries: all, or from the first key to the last query whose window holds the last key
    lo = 0;
    hi = t.Lq;
    if (p.window != 0) {
      lo = t.row0;
      hi = min(t.Lq, win_query_hi(t.row0 + min(128, t.Lkv - t.row0) - 1, p.window) + 1);
    }
    w.r_row = t.kv_tok + t.row0;
    w.s_row = t.q_tok + lo;
  }
  w.lo = lo;
  w.len = hi > lo ? hi - lo : 0;
  w.n = (w.len + 63) / 64;
  return w;
}

// ------------------------------------------------------------------ producer

// Walks the CTA's items (blockIdx.x, + gridDim.x, ...) that have work: the
// two resident 128-row tiles of item k into buffer k & 1 (boxes of 64 rows),
// then its streamed 64-row tiles into the stages (a counter across items).
template <int D, bool DKDV>
__device__ void bwd_producer(const BwdParams& p, uint8_t* sm, BwdBars& B, int n_items) {
  using C = BwdCfg<D>;
  volatile int* abort = &B.abort;
  const CUtensorMap* r1 = DKDV ? &p.tm_k : &p.tm_q;
  const CUtensorMap* r2 = DKDV ? &p.tm_v : &p.tm_do;
  const CUtensorMap* s1 = DKDV ? &p.tm_q : &p.tm_k;
  const CUtensorMap* s2 = DKDV ? &p.tm_do : &p.tm_v;
  int res_armed[2] = {-1, -1}, st_armed[C::NS];
  for (int s = 0; s < C::NS; ++s) st_armed[s] = -1;
  bool ok = true;
  uint32_t k = 0, gt = 0;
  for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
    const BwdItem t = bwd_item(p, idx);
    const BwdWork w = bwd_work<DKDV>(p, t);
    if (w.n == 0) continue;
    const int rb = k & 1;
    const uint32_t rph = (k >> 1) & 1;
    ok = ptx::mbar_wait(&B.res_empty[rb], rph ^ 1, p.timeout_ns, abort);
    if (!ok) break;
    ptx::mbar_arrive_expect_tx(&B.res_full[rb], 2 * C::RTILE);
    res_armed[rb] = (int)rph;
#pragma unroll
    for (int c = 0; c < C::KCH; ++c)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int off = c * C::RCHUNK + half * C::SCHUNK;  // rows 64 half .. +63 of the chunk
        ptx::tma_load_2d(sm + C::off_r(rb, 0) + off, r1, &B.res_full[rb], t.h * D + 64 * c, w.r_row + 64 * half);
        ptx::tma_load_2d(sm + C::off_r(rb, 1) + off, r2, &B.res_full[rb], t.h * D + 64 * c, w.r_row + 64 * half);
      }
    for (int j = 0; j < w.n; ++j, ++gt) {
      const int s = gt % C::NS;
      const uint32_t ph = (gt / C::NS) & 1;
      ok = ptx::mbar_wait(&B.st_empty[s], ph ^ 1, p.timeout_ns, abort);
      if (!ok) break;
      ptx::mbar_arrive_expect_tx(&B.st_full[s], 2 * C::STILE);
      st_armed[s] = (int)ph;
#pragma unroll
      for (int c = 0; c < C::KCH; ++c) {
        ptx::tma_load_2d(sm + C::OFF_S1 + s * C::STILE + c * C::SCHUNK, s1, &B.st_full[s], t.h * D + 64 * c,
                         w.s_row + C::BN * j);
        ptx::tma_load_2d(sm + C::OFF_S2 + s * C::STILE + c * C::SCHUNK, s2, &B.st_full[s], t.h * D + 64 * c,
                         w.s_row + C::BN * j);
      }
    }
    ++k;
  }
  if (!ok) bwd_failure(p, abort, kStatusProducer);
  // no copy may be in flight when the CTA exits
  const int never = 0;
  const unsigned long long drain_ns = 100000000ull;
  for (int b = 0; b < 2; ++b)
    if (res_armed[b] >= 0) ptx::mbar_wait(&B.res_full[b], (uint32_t)res_armed[b], drain_ns, &never);
  for (int s = 0; s < C::NS; ++s)
    if (st_armed[s] >= 0) ptx::mbar_wait(&B.st_full[s], (uint32_t)st_armed[s], drain_ns, &never);
}

// ------------------------------------------------------------------ MMA issuer (whole warp)

// S (or S^T) = R1 S1^T and dP (or dP^T) = R2 S2^T for streamed tile gt (the
// CTA's tile counter; t-th tile of its item, `len` streamed rows in all)
// into TMEM buffer gt & 1, both operands K-major.
template <int D>
__device__ __forceinline__ bool bwd_issue_sdp(const BwdParams& p, uint8_t* sm, BwdBars& B, uint32_t tmem,
                                              uint32_t gt, int t, int len, uint64_t r1, uint64_t r2,
                                              volatile int* abort) {
  using C = BwdCfg<D>;
  const int s = gt % C::NS;
  if (!ptx::mbar_wait(&B.st_full[s], (gt / C::NS) & 1, p.timeout_ns, abort)) return false;
  ptx::tc_fence_after();
  const int n16 = (min(C::BN, len - C::BN * t) + 15) >> 4;
  const uint32_t idesc = ptx::idesc_bf16(128, n16 * 16, 0);
  const uint64_t s1 = ptx::sdesc_sw128(ptx::smem_u32(sm + C::OFF_S1 + s * C::STILE), 16, 1024);
  const uint64_t s2 = ptx::sdesc_sw128(ptx::smem_u32(sm + C::OFF_S2 + s * C::STILE), 16, 1024);
  const int b = gt & 1;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {  // K-dimension D, 16 per MMA
    const uint32_t off_r = ((kk >> 2) * C::RCHUNK + (kk & 3) * 32) >> 4;
    const uint32_t off_s = ((kk >> 2) * C::SCHUNK + (kk & 3) * 32) >> 4;
    ptx::mma_ss_elect(tmem + C::tm_s(b), r1 + off_r, s1 + off_s, idesc, kk > 0 ? 1u : 0u);
  }
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off_r = ((kk >> 2) * C::RCHUNK + (kk & 3) * 32) >> 4;
    const uint32_t off_s = ((kk >> 2) * C::SCHUNK + (kk & 3) * 32) >> 4;
    ptx::mma_ss_elect(tmem + C::tm_p(b), r2 + off_r, s2 + off_s, idesc, kk > 0 ? 1u : 0u);
  }
  ptx::mma_commit_elect(&B.mma_full[b]);
  return true;
}

// Per item: S, dP of tile t+1 first (look-ahead), then, once the activation
// has written its bf16 operands over tile t's S and dP, the accumulating
// MMAs with the operand from tensor memory and the streamed tile read
// MN-major (16 rows per MMA): dQ += dS K, or dV += P^T dO and dK += dS^T Q.
// S/dP of tile t+2 reuse tile t's buffer only after these (the tensor core
// runs one thread's MMAs in order).  An item's first accumulating MMA waits
// until the epilogue has read the previous item's accumulators.
template <int D, bool DKDV>
__device__ void bwd_mma(const BwdParams& p, uint8_t* sm, BwdBars& B, uint32_t tmem, int n_items) {
  using C = BwdCfg<D>;
  volatile int* abort = &B.abort;
  constexpr uint32_t idesc_acc = ptx::idesc_bf16(128, D, 1);
  bool ok = true;
  uint32_t k = 0, gt = 0;
  for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x) {
    const BwdItem t = bwd_item(p, idx);
    const BwdWork w = bwd_work<DKDV>(p, t);
    if (w.n == 0) continue;
    const int rb = k & 1;
    ok = ptx::mbar_wait(&B.res_full[rb], (k >> 1) & 1, p.timeout_ns, abort);
    if (!ok) break;
    ptx::tc_fence_after();
    const uint64_t r1 = ptx::sdesc_sw128(ptx::smem_u32(sm + C::off_r(rb, 0)), 16, 1024);
    const uint64_t r2 = ptx::sdesc_sw128(ptx::smem_u32(sm + C::off_r(rb, 1)), 16, 1024);
    ok = bwd_issue_sdp<D>(p, sm, B, tmem, gt, 0, w.len, r1, r2, abort);
    for (int j = 0; j < w.n && ok; ++j, ++gt) {
      if (j + 1 < w.n) {
        ok = bwd_issue_sdp<D>(p, sm, B, tmem, gt + 1, j + 1, w.len, r1, r2, abort);
        if (!ok) break;
      }
      const int b = gt & 1, s = gt % C::NS;
      ok = ptx::mbar_wait(&B.act_full[b], (gt >> 1) & 1, p.timeout_ns, abort);
      if (ok && j == 0 && k > 0) ok = ptx::mbar_wait(&B.acc_empty, (k - 1) & 1, p.timeout_ns, abort);
      if (!ok) break;
      ptx::tc_fence_after();
      const int n16 = (min(C::BN, w.len - C::BN * j) + 15) >> 4;
      const uint32_t s1_addr = ptx::smem_u32(sm + C::OFF_S1 + s * C::STILE);
      const uint32_t s2_addr = ptx::smem_u32(sm + C::OFF_S2 + s * C::STILE);
      if (DKDV) {
        // dV += P^T dO and dK += dS^T Q: B operands are the streamed dO and Q
        // tiles, MN-major, 16 query rows (2048 bytes) per MMA
        const uint64_t x1 = ptx::sdesc_sw128(s2_addr, C::SCHUNK, 1024);
        const uint64_t x2 = ptx::sdesc_sw128(s1_addr, C::SCHUNK, 1024);
        for (int kk = 0; kk < n16; ++kk)
          ptx::mma_ts_elect(tmem + C::TM_A1, tmem + C::tm_s(b) + 8 * kk, x1 + 128u * kk, idesc_acc,
                            (j > 0 || kk > 0) ? 1u : 0u);
        for (int kk = 0; kk < n16; ++kk)
          ptx::mma_ts_elect(tmem + C::TM_A2, tmem + C::tm_p(b) + 8 * kk, x2 + 128u * kk, idesc_acc,
                            (j > 0 || kk > 0) ? 1u : 0u);
      } else {
        // dQ += dS K: B operand is the streamed K tile, MN-major, 16 keys per MMA
        const uint64_t x1 = ptx::sdesc_sw128(s1_addr, C::SCHUNK, 1024);
        for (int kk = 0; kk < n16; ++kk)
          ptx::mma_ts_elect(tmem + C::TM_A1, tmem + C::tm_s(b) + 8 * kk, x1 + 128u * kk, idesc_acc,
                            (j > 0 || kk > 0) ? 1u : 0u);
      }
      ptx::mma_commit_elect(&B.st_empty[s]);  // the stage is free once these MMAs complete
    }
    if (!ok) break;
    ptx::mma_commit_elect(&B.res_empty[rb]);  // the resident buffer too
    ptx::mma_commit_elect(&B.acc_full);       // the item's accumulators are final
    ++k;
  }
  if (!ok) bwd_failure(p, abort, kStatusMma);
  // no MMA may be in flight when tensor memory is released
  ptx::mma_commit_elect(&B.drain);
  const int never = 0;
  ptx::mbar_wait(&B.drain, 0, 100000000ull, &never);
}

// ------------------------------------------------------------------ activation

// 32 columns of S and dP (one chunk) -> 16 packed bf16 words of P and of dS.
// lse2/dv: per column (dkdv: one value per query) or per row (dq: the same
// value in every column); columns outside [c_lo, c_hi] (tile-relative: the
// tile's ragged end, the window, or every column of a row past the end) get
// P = dS = 0.
template <int ACT, bool PER_COL>
__device__ __forceinline__ void bwd_chunk(const uint32_t (&sr)[32], const uint32_t (&dr)[32], const float* lse2c,
                                          const float* dvc, float lse2r, float dvr, int c0, int c_lo, int c_hi,
                                          float sl, float inv_l, uint64_t gA2, uint64_t gC2, bool sfu,
                                          uint32_t (&pk_p)[16], uint32_t (&pk_ds)[16]) {
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int c = 2 * u;
    const float s0 = __uint_as_float(sr[c]), s1 = __uint_as_float(sr[c + 1]);
    const float d0 = __uint_as_float(dr[c]), d1 = __uint_as_float(dr[c + 1]);
    float p0, p1, g0, g1;
    if (ACT == kActSoftmax) {
      float l0 = lse2r, l1 = lse2r, v0 = dvr, v1 = dvr;
      if (PER_COL) {
        l0 = lse2c[c];
        l1 = lse2c[c + 1];
        v0 = dvc[c];
        v1 = dvc[c + 1];
      }
      p0 = ptx::ex2_approx(fmaf(s0, sl, -l0));
      p1 = ptx::ex2_approx(fmaf(s1, sl, -l1));
      g0 = p0 * (d0 - v0);
      g1 = p1 * (d1 - v1);
    } else {
      float y0, y1;
      if (sfu) {  // the sigma route of the forward (gdpa_set_act_route)
        gelu_tanh_val_grad_sfu2(s0, s1, gA2, gC2, y0, y1, g0, g1);
      } else {
        gelu_tanh_alu2(s0, s1, gA2, gC2, y0, y1);  // gelu(x) / scale
        gelu_tanh_grad_alu2(s0, s1, gA2, gC2, g0, g1);
      }
      p0 = y0 * sl * inv_l;
      p1 = y1 * sl * inv_l;
      g0 *= d0 * inv_l;
      g1 *= d1 * inv_l;
    }
    const bool ok0 = c0 + c >= c_lo && c0 + c <= c_hi, ok1 = c0 + c + 1 >= c_lo && c0 + c + 1 <= c_hi;
    pk_p[u] = ptx::pack_bf16x2(ok0 ? p0 : 0.0f, ok1 ? p1 : 0.0f);
    pk_ds[u] = ptx::pack_bf16x2(ok0 ? g0 : 0.0f, ok1 ? g1 : 0.0f);
  }
}

// Stores one 128 x D fp32 accumulator row (times `mul`) as bf16 to dst.
template <int D>
__device__ __forceinline__ void bwd_store_row(uint32_t taddr, float mul, __nv_bfloat16* dst, bool store, bool v8) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t r[32];
    ptx::tmem_ld32(taddr + 32 * c, r);
    ptx::tmem_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = ptx::pack_bf16x2(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
    if (store) store_row32(dst + 32 * c, pk, v8);
  }
}

template <int D>
__device__ __forceinline__ void zero_row(__nv_bfloat16* dst) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < D / 8; ++i) d4[i] = make_uint4(0u, 0u, 0u, 0u);
}

// ------------------------------------------------------------------ kernels

// Barriers, tensor memory and the three roles; `activation` runs on warps 2-5.
template <int D, bool DKDV, typename Activation>
__device__ __forceinline__ void bwd_kernel_body(const BwdParams& p, Activation&& activation) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* sm = smem_raw + pad;
  BwdBars& B = *reinterpret_cast<BwdBars*>(sm + C::OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&B.res_full[b], 1);
      ptx::mbar_init(&B.res_empty[b], 1);
      ptx::mbar_init(&B.mma_full[b], 1);
      ptx::mbar_init(&B.act_full[b], 128);
      ptx::mbar_init(&B.vec_full[b], 128);
    }
    for (int s = 0; s < C::NS; ++s) {
      ptx::mbar_init(&B.st_full[s], 1);
      ptx::mbar_init(&B.st_empty[s], 1);
    }
    ptx::mbar_init(&B.acc_full, 1);
    ptx::mbar_init(&B.acc_empty, 128);
    ptx::mbar_init(&B.drain, 1);
    B.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&B.tmem_slot, C::TM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = B.tmem_slot;
  if (warp == 0) {
    if (lane == 0) bwd_producer<D, DKDV>(p, sm, B, p.n_items);
  } else if (warp == 1) {
    bwd_mma<D, DKDV>(p, sm, B, tmem, p.n_items);
  } else {
    activation(sm, B, tmem, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::TM_COLS);
}

// Persistent: CTA c takes items c, c + gridDim.x, ... of the list.
template <int D, int ACT>
__global__ void __launch_bounds__(192, 1) gdpa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  bwd_kernel_body<D, false>(p, [&](uint8_t* sm, BwdBars& B, uint32_t tmem, int warp, int lane) {
    volatile int* abort = &B.abort;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    uint64_t gA2 = 0, gC2 = 0;
    if (ACT == kActGelu) {
      gA2 = ptx::f2_splat(p.act_a);
      gC2 = ptx::f2_splat(p.act_c);
    }
    bool ok = true;
    uint32_t k = 0, gt = 0;
    for (int idx = blockIdx.x; idx < p.n_items && ok; idx += gridDim.x) {
      const BwdItem t = bwd_item(p, idx);
      const BwdWork w = bwd_work<false>(p, t);
      const bool row_ok = row < min(128, t.Lq - t.row0);
      const size_t ri = static_cast<size_t>(t.q_tok + t.row0 + row) * p.H + t.h;
      if (w.n == 0) {  // no keys: no gradient reaches these queries
        if (row_ok) zero_row<D>(p.dq + ri * D);
        continue;
      }
      float lse2 = 0.0f, dvr = 0.0f;
      if (ACT == kActSoftmax && row_ok) {
        lse2 = __ldg(p.lse2 + ri);
        dvr = __ldg(p.dvec + ri);
      }
      const float inv_l = 1.0f / static_cast<float>(max(t.Lkv, 1));
      for (int j = 0; j < w.n && ok; ++j, ++gt) {
        const int b = gt & 1;
        ok = ptx::mbar_wait(&B.mma_full[b], (gt >> 1) & 1, p.timeout_ns, abort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ptx::tc_fence_after();
        const int kv_t0 = w.lo + C::BN * j;
        const int ncols = min(C::BN, w.len - C::BN * j);
        const int nch = (ncols + 31) >> 5;
        int c_lo = 0, c_hi = row_ok ? ncols - 1 : -1;  // this row's valid columns of the tile
        if (p.window != 0 && row_ok) {
          const int i = t.row0 + row;
          c_lo = win_key_lo(i, p.window) - kv_t0;
          c_hi = min(c_hi, i - kv_t0);
        }
        for (int ch = 0; ch < nch; ++ch) {
          uint32_t sr[32], dr[32];
          ptx::tmem_ld32(tmem + lane_off + C::tm_s(b) + 32 * ch, sr);
          ptx::tmem_ld32(tmem + lane_off + C::tm_p(b) + 32 * ch, dr);
          ptx::tmem_wait_ld();
          uint32_t pk_p[16], pk_ds[16];
          bwd_chunk<ACT, false>(sr, dr, nullptr, nullptr, lse2, dvr, 32 * ch, c_lo, c_hi, p.score_scale, inv_l,
                                gA2, gC2, p.act_sfu != 0, pk_p, pk_ds);
          ptx::tmem_st16(tmem + lane_off + C::tm_s(b) + 16 * ch, pk_ds);  // dS over consumed S columns
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&B.act_full[b]);
      }
      if (!ok) break;
      ok = ptx::mbar_wait(&B.acc_full, k & 1, p.timeout_ns, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      bwd_store_row<D>(tmem + lane_off + C::TM_A1, p.scale, p.dq + ri * D, row_ok, p.align32 != 0);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&B.acc_empty);
      ++k;
    }
    if (!ok && lane == 0) bwd_failure(p, abort, kStatusActivation);
  });
}

template <int D, int ACT>
__global__ void __launch_bounds__(192, 1) gdpa_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  bwd_kernel_body<D, true>(p, [&](uint8_t* sm, BwdBars& B, uint32_t tmem, int warp, int lane) {
    volatile int* abort = &B.abort;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;     // key row of the item
    const int tid = (warp - 2) * 32 + lane;  // 0..127 over the four warps
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float* vec = reinterpret_cast<float*>(sm + C::OFF_VEC);  // [2 buffers][lse2, Dv][64]
    uint64_t gA2 = 0, gC2 = 0;
    if (ACT == kActGelu) {
      gA2 = ptx::f2_splat(p.act_a);
      gC2 = ptx::f2_splat(p.act_c);
    }
    bool ok = true;
    uint32_t k = 0, gt = 0;
    for (int idx = blockIdx.x; idx < p.n_items && ok; idx += gridDim.x) {
      const BwdItem t = bwd_item(p, idx);
      const BwdWork w = bwd_work<true>(p, t);
      const int keys = min(128, t.Lkv - t.row0);
      const size_t ri = static_cast<size_t>(t.kv_tok + t.row0 + row) * p.H + t.h;
      if (w.n == 0) {  // no queries: these keys receive no gradient
        if (row < keys) {
          zero_row<D>(p.dk + ri * D);
          zero_row<D>(p.dv + ri * D);
        }
        continue;
      }
      const float inv_l = 1.0f / static_cast<float>(max(t.Lkv, 1));
      const int jk = t.row0 + row;  // this thread's key, counted from the sequence start
      const int j_qhi = p.window != 0 ? win_query_hi(jk, p.window) : 0x7fffffff;
      for (int u = 0; u < w.n && ok; ++u, ++gt) {
        const int b = gt & 1;
        const int u0 = w.lo + C::BN * u;  // the tile's first query
        const int nq = min(C::BN, w.len - C::BN * u);
        float* vb = vec + b * 2 * C::BN;
        if (ACT == kActSoftmax) {
          // lse2 and Dv of the tile's queries, one per thread.  The buffer of
          // tile gt - 2 is free: this thread waited for every thread's
          // arrival at tile gt - 1, which each made after finishing gt - 2.
          if (tid < C::BN) {
            float l = 0.0f, d = 0.0f;
            if (tid < nq) {
              const size_t qi = static_cast<size_t>(t.q_tok + u0 + tid) * p.H + t.h;
              l = __ldg(p.lse2 + qi);
              d = __ldg(p.dvec + qi);
            }
            vb[tid] = l;
            vb[C::BN + tid] = d;
          }
          ptx::mbar_arrive(&B.vec_full[b]);
          ok = ptx::mbar_wait(&B.vec_full[b], (gt >> 1) & 1, p.timeout_ns, abort);
        }
        if (ok) ok = ptx::mbar_wait(&B.mma_full[b], (gt >> 1) & 1, p.timeout_ns, abort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ptx::tc_fence_after();
        const int nch = (nq + 31) >> 5;
        int c_lo = 0, c_hi = nq - 1;  // this key row's valid query columns of the tile
        if (p.window != 0) {
          c_lo = jk - u0;
          c_hi = min(c_hi, j_qhi - u0);
        }
        for (int ch = 0; ch < nch; ++ch) {
          uint32_t sr[32], dr[32];
          ptx::tmem_ld32(tmem + lane_off + C::tm_s(b) + 32 * ch, sr);
          ptx::tmem_ld32(tmem + lane_off + C::tm_p(b) + 32 * ch, dr);
          ptx::tmem_wait_ld();
          uint32_t pk_p[16], pk_ds[16];
          bwd_chunk<ACT, true>(sr, dr, vb + 32 * ch, vb + C::BN + 32 * ch, 0.0f, 0.0f, 32 * ch, c_lo, c_hi,
                               p.score_scale, inv_l, gA2, gC2, p.act_sfu != 0, pk_p, pk_ds);
          ptx::tmem_st16(tmem + lane_off + C::tm_s(b) + 16 * ch, pk_p);   // P^T over consumed S^T columns
          ptx::tmem_st16(tmem + lane_off + C::tm_p(b) + 16 * ch, pk_ds);  // dS^T over consumed dP^T columns
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&B.act_full[b]);
      }
      if (!ok) break;
      ok = ptx::mbar_wait(&B.acc_full, k & 1, p.timeout_ns, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const bool store = row < keys;
      bwd_store_row<D>(tmem + lane_off + C::TM_A1, 1.0f, p.dv + ri * D, store, p.align32 != 0);
      bwd_store_row<D>(tmem + lane_off + C::TM_A2, p.scale, p.dk + ri * D, store, p.align32 != 0);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&B.acc_empty);
      ++k;
    }
    if (!ok && lane == 0) bwd_failure(p, abort, kStatusActivation);
  });
}

// Dv_i = <dO_i, O_i> and lse2_i = lse_i log2(e), one warp per (token, head) row.
template <int D>
__global__ void __launch_bounds__(256) gdpa_bwd_prep_kernel(const __nv_bfloat16* out, const __nv_bfloat16* dout,
                                                            const float* lse, float* lse2, float* dvec,
                                                            int64_t rows) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  constexpr int PER = D / 32;  // bf16 values per lane (2 or 4)
  const __nv_bfloat16* o = out + r * D + lane * PER;
  const __nv_bfloat16* d = dout + r * D + lane * PER;
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < PER; i += 2) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(o + i);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(d + i);
    acc = fmaf(__low2float(a), __low2float(b), acc);
    acc = fmaf(__high2float(a), __high2float(b), acc);
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
  if (lane == 0) {
    dvec[r] = acc;
    lse2[r] = lse[r] * 1.4426950408889634f;
  }
}

}  // namespace gdpa
