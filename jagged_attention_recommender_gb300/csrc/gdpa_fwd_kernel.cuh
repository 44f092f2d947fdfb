// gdpa_fwd_kernel.cuh -- persistent, warp-specialised jagged GDPA forward
// kernel for sm_103a (tcgen05 tensor cores, tensor memory, TMA).
//
// One CTA per SM walks its own list of work items (a 128-row query tile of
// one (sequence, head) against its key range; built on the host, see
// gdpa_plan.cpp).  Roles inside the CTA (384 threads, three warpgroups):
//
//   warpgroup 0 (registers handed back to the pool):
//     warp 0    TMA producer for the Q tile (2 stages) and K tiles (NK
//               stages); warp 2 TMA producer for V tiles (NV stages); all
//               128-byte swizzled; K is released after Q K^T, V after P V;
//     warp 1    MMA issuer (the whole warp runs the loop, one elected
//               lane issues): S = Q K^T into tensor memory
//               (two S buffers), then O += P V with P read straight from
//               tensor memory (two O buffers, one per in-flight item);
//   warpgroup 1 (248 registers a thread): activation, one query row per
//               thread: reads its whole row of S from TMEM at once, masks the
//               ragged edge / window, applies the online softmax (running max
//               with lazy rescaling of O) or the GELU / SiLU, and writes P
//               (bf16) back over S; at the end of an item it hands the row
//               sum to the epilogue through shared memory;
//   warpgroup 2 epilogue: waits for the item's last O += P V, normalises O
//               (1/l, or 1/Lkv for GELU), stores it, and frees the O buffer,
//               while the activation warps already work on the next item.
//
// The MMA issuer runs one K/V tile ahead: it issues S(g+1) = Q K(g+1)^T
// before O += P(g) V(g), so the tensor core works on the next tile while the
// activation warps process the current one, and this look-ahead crosses item
// boundaries (the "outer loop" pipelining that matters when a key range is a
// single tile: GDPA section of the techfeed summary of "GEM Training").
//
// Masks are applied per 32-column chunk and the chunk's class (all keys
// valid, none valid, some valid) is agreed on by the warp: only the chunk
// that holds a row's ragged end or its causal diagonal pays for a per-element
// test, and chunks with no valid key are skipped (their P is zero).
//
// Synchronisation is by mbarriers only; every wait is bounded in time and a
// timeout is reported in the device status word instead of hanging.
#pragma once

#include "gdpa_fwd_common.cuh"

namespace gdpa {

// Item kinds, one kernel instantiation each:
//   full      128 query rows against the whole key range in 128-key tiles;
//   window    128 query rows against their block window;
//   key split at most 32 queries, each warp owns a 32-key block of every tile;
//   full MX   full attention with MXFP8 Q and K (D = 128): e4m3 tiles, one
//             E8M0 scale per 32 elements of a row, S = Q K^T by the
//             block-scaled MMA (32 elements of D per instruction, the scales
//             read from TMEM); P V stays bf16.  The activation warps put the
//             next tile's scale words into TMEM while they work on the
//             current one; the second O buffer gives its columns to them.
enum : int { kModeFull = 0, kModeWindow = 1, kModeKeySplit = 2, kModeFullMx = 3 };

template <int D, int MODE = kModeFull>
struct FwdCfg {
  static constexpr bool WIN = MODE == kModeWindow;
  static constexpr bool KS = MODE == kModeKeySplit;
  static constexpr int BM = 128;
  static constexpr int BN = 128;                   // keys per K/V tile
  static constexpr int KCH = D / 64;               // 64-element (128-byte) column chunks
  static constexpr int CHUNK_BYTES = 128 * 128;    // Q chunk: 128 rows x 128 bytes
  static constexpr int TILE_BYTES = KCH * CHUNK_BYTES;
  static constexpr int KV_CHUNK_BYTES = BN * 128;  // K/V chunk: BN rows x 128 bytes
  static constexpr int KV_TILE_BYTES = KCH * KV_CHUNK_BYTES;
  static constexpr int NQ = 2;                                // Q stages
  static constexpr int NK = (D == 64) ? 4 : 3;                // K stages
  static constexpr int NV = (D == 64) ? 4 : 2;                // V stages
  static constexpr bool MX = MODE == kModeFullMx;
  // staged tile sizes: an e4m3 row of D = 128 is one 128-byte swizzle row
  static constexpr int Q_BYTES = MX ? BM * D : TILE_BYTES;
  static constexpr int K_BYTES = MX ? BN * D : KV_TILE_BYTES;
  static constexpr int V_BYTES = KV_TILE_BYTES;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQ * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NK * K_BYTES;
  static constexpr int OFF_L = OFF_V + NV * V_BYTES;  // row sums, 2 x 128 floats
  // Key split only: row maxima (2 x 128 floats) and the exchange buffer in
  // which the four warps' partial output rows meet (4 x 32 rows of 64
  // floats, rows padded to 68 floats so that 16-byte accesses by a warp are
  // free of bank conflicts).
  static constexpr int OFF_M = OFF_L + 2 * 128 * 4;
  static constexpr int X_STRIDE = 68;
  static constexpr int OFF_X = OFF_M + (KS ? 2 * 128 * 4 : 0);
  static constexpr int OFF_BAR = OFF_X + (KS ? 4 * 32 * X_STRIDE * 4 : 0);
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;  // + slack for 1024-byte alignment
  // O buffers: two (an item's epilogue overlaps the next item), one with MX
  static constexpr int NOB = MX ? 1 : 2;
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = MX ? 256 : 256 + D;
  // MX scale words (4 columns a slot, slots 32 columns apart): Q of items
  // qi & 1, K of tiles g & 1
  static constexpr uint32_t TM_SFA = 256 + D, TM_SFB = 256 + D + 64;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int THREADS = 384;  // 3 warpgroups
  // Registers per thread after reallocation: control warpgroup, activation
  // warpgroup; the epilogue keeps the launch count.  Each SM sub-partition
  // holds one warp of each warpgroup, so the launch count R must satisfy
  // REGS_CTRL + REGS_ACT + R <= 3 R.
  static constexpr int REGS_CTRL = 88;
  static constexpr int REGS_ACT = 248;
  static constexpr int MIN_LAUNCH_REGS = (REGS_CTRL + REGS_ACT + 1) / 2;
  static_assert(TM_O1 + D <= TM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(!KS || D == 64, "key split is built for D = 64");
  static_assert(!MX || (D == 128 && TM_SFB + 32 + 4 <= TM_COLS), "MXFP8 is built for D = 128");
};

// Shared-memory barrier block.
template <int NQ, int NK, int NV>
struct Bars {
  uint64_t q_full[NQ], q_empty[NQ];
  uint64_t k_full[NK], k_empty[NK], v_full[NV], v_empty[NV];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done;              // after every O += P V (activation)
  uint64_t o_full[2];           // after an item's last O += P V into O[b] (epilogue)
  uint64_t o_empty[2];          // the epilogue has drained O[b] (MMA)
  uint64_t l_full[2], l_empty[2];  // row sums of the item using O[b] (activation <-> epilogue)
  uint64_t x_full, x_empty;     // key split: partial rows written / read (epilogue warps)
  uint64_t sf_full[2];          // MX: scale words of tile g (and of its item's Q) in TMEM (activation)
  uint64_t mma_drain;
  uint32_t tmem_slot;
  int abort;
};

template <int D, int MODE>
using FwdBars = Bars<FwdCfg<D, MODE>::NQ, FwdCfg<D, MODE>::NK, FwdCfg<D, MODE>::NV>;

struct ItemView {
  int h, q0, kv0, kv_end, n_kv, q_rows, q_tok, kv_tok, Lkv;
};

template <int MODE, bool FLAG = false>
__device__ __forceinline__ ItemView decode_item(const FwdParams& p, int idx) {
  constexpr bool WIN = MODE == kModeWindow;
  constexpr int BN = 128;
  const int4 it = __ldg(p.items + idx);
  ItemView v;
  const int b = it.x;
  v.h = it.y;
  v.q0 = it.z;
  v.kv0 = it.w;
  const ItemRows r = item_rows<FLAG>(p, b);
  v.q_tok = r.qs + v.q0;
  v.kv_tok = r.ks;
  v.Lkv = r.Lkv;
  v.q_rows = max(0, min(128, r.Lq - v.q0));
  v.kv_end = WIN ? min(v.Lkv, v.q0 + 128) : v.Lkv;
  v.n_kv = v.kv_end > v.kv0 && v.q_rows > 0 ? (v.kv_end - v.kv0 + BN - 1) / BN : 0;  // no rows: nothing to do
  return v;
}

// ------------------------------------------------------------------ producer

// Two producer threads, each in order on its own resource: one stages Q and
// K tiles, the other V tiles.  A K load therefore never waits behind a V
// slot (freed only when an earlier P V completes), which would otherwise
// chain one load latency into every pair of tiles.
template <int D, int MODE, bool LOAD_V>
__device__ void run_producer(const FwdParams& p, uint8_t* sm, FwdBars<D, MODE>& B, int ibeg, int iend) {
  using C = FwdCfg<D, MODE>;
  constexpr bool KS = C::KS;
  volatile int* abort = &B.abort;
  int qi = 0;
  uint32_t g = 0;
  bool ok = true;
  int q_armed[C::NQ];  // last parity armed per stage (for draining)
#pragma unroll
  for (int s = 0; s < C::NQ; ++s) q_armed[s] = -1;
  int k_armed[C::NK], v_armed[C::NV];
#pragma unroll
  for (int s = 0; s < C::NK; ++s) k_armed[s] = -1;
#pragma unroll
  for (int s = 0; s < C::NV; ++s) v_armed[s] = -1;
  if (LOAD_V) {
    ptx::prefetch_tensormap(&p.tm_v);
  } else {
    ptx::prefetch_tensormap(&p.tm_q);
    ptx::prefetch_tensormap(&p.tm_k);
  }
  for (int idx = ibeg; idx < iend && ok; ++idx) {
    const ItemView t = decode_item<MODE, !LOAD_V>(p, idx);
    if (t.n_kv == 0) continue;
    if (!LOAD_V) {
      const int qs = qi % C::NQ;
      const uint32_t qph = (qi / C::NQ) & 1;
      ok = ptx::mbar_wait(&B.q_empty[qs], qph ^ 1, p.timeout_ns, abort);
      if (!ok) break;
      ptx::mbar_arrive_expect_tx(&B.q_full[qs], C::Q_BYTES);
      q_armed[qs] = (int)qph;
      uint8_t* sq = sm + C::OFF_Q + qs * C::Q_BYTES;
      if (C::MX) {  // e4m3: the whole row of D = 128 bytes in one box
        ptx::tma_load_2d(sq, &p.tm_q, &B.q_full[qs], t.h * D, t.q_tok);
      } else if (KS) {  // the (at most) 32 queries in each lane quarter: the Q map's box is 32 rows
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
#pragma unroll
          for (int r = 0; r < 4; ++r)
            ptx::tma_load_2d(sq + c * C::CHUNK_BYTES + r * 32 * 128, &p.tm_q, &B.q_full[qs], t.h * D + 64 * c, t.q_tok);
      } else {
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          ptx::tma_load_2d(sq + c * C::CHUNK_BYTES, &p.tm_q, &B.q_full[qs], t.h * D + 64 * c, t.q_tok);
      }
    }
    for (int j = 0; j < t.n_kv; ++j, ++g) {
      const int y = t.kv_tok + t.kv0 + C::BN * j;
      if (!LOAD_V) {  // K is released once its Q K^T is done
        const int si = g % C::NK;
        const uint32_t ph = (g / C::NK) & 1;
        ok = ptx::mbar_wait(&B.k_empty[si], ph ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        uint8_t* dst = sm + C::OFF_K + si * C::K_BYTES;
        ptx::mbar_arrive_expect_tx(&B.k_full[si], C::K_BYTES);
        if (C::MX) {
          ptx::tma_load_2d(dst, &p.tm_k, &B.k_full[si], t.h * D, y);
        } else {
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
            ptx::tma_load_2d(dst + c * C::KV_CHUNK_BYTES, &p.tm_k, &B.k_full[si], t.h * D + 64 * c, y);
        }
        k_armed[si] = (int)ph;
      } else {  // V is released once its P V is done
        const int si = g % C::NV;
        const uint32_t ph = (g / C::NV) & 1;
        ok = ptx::mbar_wait(&B.v_empty[si], ph ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        uint8_t* dst = sm + C::OFF_V + si * C::V_BYTES;
        ptx::mbar_arrive_expect_tx(&B.v_full[si], C::V_BYTES);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          ptx::tma_load_2d(dst + c * C::KV_CHUNK_BYTES, &p.tm_v, &B.v_full[si], t.h * D + 64 * c, y);
        v_armed[si] = (int)ph;
      }
    }
    ++qi;
  }
  if (!ok) report_failure(p, abort, kStatusProducer);
  // Let every bulk copy this thread started land before the CTA can exit.
  const int never = 0;
  const unsigned long long drain_ns = 100000000ull;
  for (int s = 0; s < C::NQ; ++s)
    if (q_armed[s] >= 0) ptx::mbar_wait(&B.q_full[s], (uint32_t)q_armed[s], drain_ns, &never);
#pragma unroll
  for (int s = 0; s < C::NK; ++s)
    if (k_armed[s] >= 0) ptx::mbar_wait(&B.k_full[s], (uint32_t)k_armed[s], drain_ns, &never);
#pragma unroll
  for (int s = 0; s < C::NV; ++s)
    if (v_armed[s] >= 0) ptx::mbar_wait(&B.v_full[s], (uint32_t)v_armed[s], drain_ns, &never);
}

// ------------------------------------------------------------------ MMA issuer

struct PendingPV {
  uint32_t g;
  int sb, ob, qi, first, last, n16;
};

template <int D, int MODE>
__device__ __forceinline__ bool issue_pv(const FwdParams& p, uint8_t* sm, FwdBars<D, MODE>& B, uint32_t tmem,
                                         const PendingPV& P) {
  using C = FwdCfg<D, MODE>;
  volatile int* abort = &B.abort;
  if (!ptx::mbar_wait(&B.p_full[P.sb], (P.g >> 1) & 1, p.timeout_ns, abort)) return false;
  if (P.first && !ptx::mbar_wait(&B.o_empty[P.ob], ((P.qi / C::NOB) & 1) ^ 1, p.timeout_ns, abort)) return false;
  const int sv = P.g % C::NV;
  if (!ptx::mbar_wait(&B.v_full[sv], (P.g / C::NV) & 1, p.timeout_ns, abort)) return false;
  ptx::tc_fence_after();
  const uint32_t v_base = ptx::smem_u32(sm + C::OFF_V + sv * C::V_BYTES);
  const uint32_t o_col = P.ob ? C::TM_O1 : C::TM_O0;
  const uint32_t p_col = P.sb ? C::TM_S1 : C::TM_S0;
  constexpr uint32_t idesc = ptx::idesc_bf16(128, D, 1);
  for (int kk = 0; kk < P.n16; ++kk) {
    // B = V tile, MN-major: 16 keys = two 8-row groups (SBO = 1024 B apart);
    // the two 64-column halves of D sit one chunk apart (LBO).
    const uint64_t bdesc = ptx::sdesc_sw128(v_base + kk * 2048, C::KV_CHUNK_BYTES, 1024);
    ptx::mma_ts_elect(tmem + o_col, tmem + p_col + 8 * kk, bdesc, idesc, (P.first && kk == 0) ? 0u : 1u);
  }
  ptx::mma_commit_elect(&B.v_empty[sv]);
  ptx::mma_commit_elect(&B.o_done);
  if (P.last) ptx::mma_commit_elect(&B.o_full[P.ob]);
  return true;
}

template <int D, int MODE>
__device__ void run_mma(const FwdParams& p, uint8_t* sm, FwdBars<D, MODE>& B, uint32_t tmem, int ibeg, int iend) {
  using C = FwdCfg<D, MODE>;
  volatile int* abort = &B.abort;
  int qi = 0;
  uint32_t g = 0;
  bool ok = true;
  bool have_prev = false;
  PendingPV prev = {0, 0, 0, 0, 0, 0, 0};
  for (int idx = ibeg; idx < iend && ok; ++idx) {
    const ItemView t = decode_item<MODE>(p, idx);
    if (t.n_kv == 0) continue;
    const int qs = qi % C::NQ;
    ok = ptx::mbar_wait(&B.q_full[qs], (qi / C::NQ) & 1, p.timeout_ns, abort);
    if (!ok) break;
    const uint32_t q_base = ptx::smem_u32(sm + C::OFF_Q + qs * C::Q_BYTES);
    for (int j = 0; j < t.n_kv; ++j, ++g) {
      const int s = g % C::NK;
      ok = ptx::mbar_wait(&B.k_full[s], (g / C::NK) & 1, p.timeout_ns, abort);
      const int sb = g & 1;
      if (C::MX && ok) ok = ptx::mbar_wait(&B.sf_full[sb], (g >> 1) & 1, p.timeout_ns, abort);
      if (!ok) break;
      ptx::tc_fence_after();
      const int ncols = min(C::BN, t.kv_end - t.kv0 - C::BN * j);
      const int n16 = (ncols + 15) >> 4;
      const uint32_t k_base = ptx::smem_u32(sm + C::OFF_K + s * C::K_BYTES);
      const uint32_t s_col = sb ? C::TM_S1 : C::TM_S0;
      if constexpr (C::MX) {
        // 32 e4m3 elements of D = 32 bytes of the 128-byte swizzle row per
        // MMA, scale byte kk of each row's word; all 128 key columns (the
        // ragged end's extra columns are masked by the activation).
        const uint32_t sfa = tmem + C::TM_SFA + 32u * (qi & 1), sfb = tmem + C::TM_SFB + 32u * sb;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_mx_elect(tmem + s_col, ptx::sdesc_sw128(q_base + 32 * kk, 16, 1024),
                            ptx::sdesc_sw128(k_base + 32 * kk, 16, 1024), ptx::idesc_mx_e4m3(128, 128, kk), sfa, sfb,
                            kk > 0 ? 1u : 0u);
      } else {
        const uint32_t idesc = ptx::idesc_bf16(128, n16 * 16, 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-major operands: 16 columns of D = 32 bytes inside a 128-byte swizzle row.
          const uint32_t qoff = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * C::KV_CHUNK_BYTES + (kk & 3) * 32;
          ptx::mma_ss_elect(tmem + s_col, ptx::sdesc_sw128(q_base + qoff, 16, 1024),
                            ptx::sdesc_sw128(k_base + koff, 16, 1024), idesc, kk > 0 ? 1u : 0u);
        }
      }
      ptx::mma_commit_elect(&B.s_full[sb]);
      ptx::mma_commit_elect(&B.k_empty[s]);
      if (j == t.n_kv - 1) ptx::mma_commit_elect(&B.q_empty[qs]);
      if (have_prev) {
        ok = issue_pv<D, MODE>(p, sm, B, tmem, prev);
        if (!ok) break;
      }
      prev = PendingPV{g, sb, qi % C::NOB, qi, j == 0 ? 1 : 0, j == t.n_kv - 1 ? 1 : 0, n16};
      have_prev = true;
    }
    ++qi;
  }
  if (ok && have_prev) ok = issue_pv<D, MODE>(p, sm, B, tmem, prev);
  if (!ok) report_failure(p, abort, kStatusMma);
  // Every MMA this thread issued is complete once this commit lands.
  ptx::mma_commit_elect(&B.mma_drain);
  const int never = 0;
  ptx::mbar_wait(&B.mma_drain, 0, 100000000ull, &never);
}

// ------------------------------------------------------------------ activation

// MX: where the activation warps stand in the CTA's tile sequence when they
// stage scale words -- item index, tile of the item, non-empty item count.
template <int MODE>
struct MxCursor {
  int idx, j, qi;
  ItemView t;
  bool valid;
  __device__ __forceinline__ void seek(const FwdParams& p, int iend) {  // first non-empty item from idx on
    for (valid = false; idx < iend; ++idx) {
      t = decode_item<MODE>(p, idx);
      if (t.n_kv > 0) {
        valid = true;
        return;
      }
    }
  }
  __device__ __forceinline__ void advance(const FwdParams& p, int iend) {
    if (++j < t.n_kv) return;
    j = 0;
    ++qi;
    ++idx;
    seek(p, iend);
  }
  // This thread's four scale words of the tile (keys 128 j + 32 c + lane) and,
  // at an item's first tile, of its Q (rows 32 c + lane); scale 1 (0x7F) past
  // the end.
  __device__ __forceinline__ void load(const FwdParams& p, int lane, uint32_t (&wk)[4], uint32_t (&wq)[4]) const {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int key = 128 * j + 32 * c + lane, row = 32 * c + lane;
      wk[c] = key < t.Lkv ? __ldg(p.k_sf + static_cast<size_t>(t.kv_tok + key) * p.H + t.h) : 0x7F7F7F7Fu;
      wq[c] = (j == 0 && row < t.q_rows) ? __ldg(p.q_sf + static_cast<size_t>(t.q_tok + row) * p.H + t.h)
                                         : 0x7F7F7F7Fu;
    }
  }
};

// Per-element validity of score column c (tile-relative) for this row.
__device__ __forceinline__ bool col_ok(int c, int c_lo, int c_hi) { return c >= c_lo && c <= c_hi; }

template <int D, int ACT, int MODE>
__device__ void run_activation(const FwdParams& p, FwdBars<D, MODE>& B, float* l_buf, float* m_buf, uint32_t tmem,
                               int ibeg, int iend, int warp, int lane) {
  using C = FwdCfg<D, MODE>;
  constexpr bool WIN = C::WIN, KS = C::KS;
  constexpr int NCH = C::BN / 32;  // 32-column chunks of a score tile
  volatile int* abort = &B.abort;
  const int quarter = warp & 3;  // TMEM lane quarter this warp may access
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const float sl = p.score_scale;
  const ActK ak = act_k(p.act_a, p.act_c, p.act_sfu);  // GELU / SiLU: the scale folded into the cubic
  int qi = 0;
  uint32_t g = 0;
  bool ok = true;
  // MX: the scale words of tile 0 go to TMEM now, those of tile g + 1 at the
  // start of tile g (S(g) complete, so S(g - 1) and the previous item's
  // Q K^T, the slots' last readers, are too); their loads run a tile ahead.
  MxCursor<MODE> cur;
  uint32_t wk[4], wq[4];
  if constexpr (C::MX) {
    cur.idx = ibeg;
    cur.j = 0;
    cur.qi = 0;
    cur.seek(p, iend);
    if (cur.valid) {
      cur.load(p, lane, wk, wq);
      ptx::tmem_st4(tmem + lane_off + C::TM_SFB, wk[0], wk[1], wk[2], wk[3]);
      ptx::tmem_st4(tmem + lane_off + C::TM_SFA, wq[0], wq[1], wq[2], wq[3]);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&B.sf_full[0]);
      cur.advance(p, iend);
      if (cur.valid) cur.load(p, lane, wk, wq);
    }
  }
  for (int idx = ibeg; idx < iend && ok; ++idx) {
    const ItemView t = decode_item<MODE>(p, idx);
    if (t.n_kv == 0) continue;  // the epilogue writes the zero rows
    const int ob = qi % C::NOB;
    const uint32_t o_addr = tmem + lane_off + (ob ? C::TM_O1 : C::TM_O0);
    float m_run = -INFINITY, l_run = 0.0f;
    const int i_seq = t.q0 + row;  // query index inside its sequence
    int win_lo = 0;
    if (WIN) {
      const int blk = i_seq / 64 - (p.window_blocks - 1);
      win_lo = blk > 0 ? blk * 64 : 0;
    }
    // A warp whose 32 rows all lie past the end of the query tile keeps the
    // barrier protocol but skips the math (e.g. 3 of 4 warps for 32 queries).
    const bool rows_live = __any_sync(0xffffffffu, (KS ? lane : row) < t.q_rows);
    for (int j = 0; j < t.n_kv; ++j, ++g) {
      const int sb = g & 1;
      ok = ptx::mbar_wait(&B.s_full[sb], (g >> 1) & 1, p.timeout_ns, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      if constexpr (C::MX) {
        if (cur.valid) {  // tile g + 1: its K scales, and its item's Q scales if it starts one
          const uint32_t nb = (g + 1) & 1;
          ptx::tmem_st4(tmem + lane_off + C::TM_SFB + 32 * nb, wk[0], wk[1], wk[2], wk[3]);
          if (cur.j == 0)
            ptx::tmem_st4(tmem + lane_off + C::TM_SFA + 32 * (cur.qi & 1), wq[0], wq[1], wq[2], wq[3]);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(&B.sf_full[nb]);
          cur.advance(p, iend);
          if (cur.valid) cur.load(p, lane, wk, wq);
        }
      }
      const uint32_t s_addr = tmem + lane_off + (sb ? C::TM_S1 : C::TM_S0);
      float alpha = 1.0f;
      bool rescale = false;
      if constexpr (KS) {
        if (rows_live) {
          // Key split: every warp holds the same queries and owns the 32-key
          // block [32 q, 32 q + 32) of the tile (its diagonal block of S).
          const int ncols = min(128, t.kv_end - 128 * j);
          const int nch = (ncols + 31) >> 5;
          const int cb = 32 * quarter;
          const bool live = cb < ncols, full = cb + 32 <= ncols;  // warp-uniform
          uint32_t sr[32];
          uint32_t pk[16];
          if (live) {
            ptx::tmem_ld32(s_addr + cb, sr);
            ptx::tmem_wait_ld();
          }
          if (ACT == kActSoftmax) {
            const bool fold = sl > 0.0f;
            float mx = -INFINITY;
            if (live) {
              float m2[2] = {-INFINITY, -INFINITY};
              if (full && fold) {
#pragma unroll
                for (int u = 0; u < 32; u += 4) {
                  m2[0] = ptx::max3(m2[0], __uint_as_float(sr[u]), __uint_as_float(sr[u + 1]));
                  m2[1] = ptx::max3(m2[1], __uint_as_float(sr[u + 2]), __uint_as_float(sr[u + 3]));
                }
              } else {
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                  float x = __uint_as_float(sr[u]);
                  if (!fold) x *= sl;
                  if (cb + u >= ncols) x = -INFINITY;
                  sr[u] = __float_as_uint(x);
                  m2[u & 1] = fmaxf(m2[u & 1], x);
                }
              }
              mx = fmaxf(m2[0], m2[1]);
              if (fold) mx *= sl;
            }
            const float m_new = fmaxf(m_run, mx);
            if (j == 0) {
              m_run = m_new;
            } else if (m_new > m_run + 8.0f) {
              alpha = ptx::ex2_approx(m_run - m_new);
              l_run *= alpha;
              m_run = m_new;
              rescale = true;
            }
            if (live) {
              const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
              const uint64_t mul2 = ptx::f2_splat(fold ? sl : 1.0f);
              const uint64_t neg2 = ptx::f2_splat(-m_use);
              uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const uint64_t x2 =
                    ptx::f2_fma(ptx::f2_pack(__uint_as_float(sr[2 * u]), __uint_as_float(sr[2 * u + 1])), mul2, neg2);
                float a, b;
                ptx::f2_unpack(x2, a, b);
                a = ptx::ex2_approx(a);
                b = ptx::ex2_approx(b);
                acc[u & 3] = ptx::f2_add(acc[u & 3], ptx::f2_pack(a, b));
                pk[u] = ptx::pack_bf16x2(a, b);
              }
              const uint64_t acc01 = ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3]));
              float sa, sb2;
              ptx::f2_unpack(acc01, sa, sb2);
              l_run += sa + sb2;
            }
          } else if (live) {  // GELU
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              float a, b;
              act_eval2(ak, __uint_as_float(sr[2 * u]), __uint_as_float(sr[2 * u + 1]), a, b);
              if (!full) {
                a = cb + 2 * u < ncols ? a : 0.0f;
                b = cb + 2 * u + 1 < ncols ? b : 0.0f;
              }
              pk[u] = ptx::pack_bf16x2(a, b);
            }
          }
          // P: this warp's block, zeros in the other blocks P V reads
          uint32_t zero[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) zero[u] = 0u;
#pragma unroll
          for (int jb = 0; jb < 4; ++jb) {
            if (jb >= nch) break;
            if (jb == quarter && live)
              ptx::tmem_st16(s_addr + 16 * jb, pk);
            else
              ptx::tmem_st16(s_addr + 16 * jb, zero);
          }
          ptx::tmem_wait_st();
        }
      } else {
        if (rows_live) {
          // valid key columns of this row: [c_lo, c_hi] (tile-relative)
          const int kv_t0 = t.kv0 + C::BN * j;
          const int ncols = min(C::BN, t.kv_end - kv_t0);  // the tile's key extent
          int c_lo = 0, c_hi = ncols - 1;
          if (WIN) {
            c_lo = max(0, win_lo - kv_t0);
            c_hi = min(c_hi, i_seq - kv_t0);
          }
          const int nch = (ncols + 31) >> 5;  // chunks P V reads
          // chunk classes agreed on by the warp: bit ch of `fullm` = every key
          // of chunk ch is valid for all 32 rows; bit ch of `livem` = some row
          // has a valid key in it
          uint32_t fullm = 0, livem = 0;
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            const int lo = 32 * ch, hi = 32 * ch + 31;
            if (__all_sync(0xffffffffu, lo >= c_lo && hi <= c_hi)) fullm |= 1u << ch;
            if (__any_sync(0xffffffffu, ch < nch && hi >= c_lo && lo <= c_hi)) livem |= 1u << ch;
          }
          // The whole row of scores in registers, one TMEM round trip.
          uint32_t sr[C::BN];
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch)
            if ((livem >> ch) & 1u) ptx::tmem_ld32(s_addr + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * ch]));
          ptx::tmem_wait_ld();
          if (ACT == kActSoftmax) {
            // Scores become log2-domain values x = s * scale * log2(e); masked
            // columns become -inf.  With scale > 0 the scaling is folded into
            // the exponent's FMA; otherwise it is applied first.
            const bool fold = sl > 0.0f;
            float m2[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              if (!((livem >> ch) & 1u)) continue;
              if (((fullm >> ch) & 1u) && fold) {
#pragma unroll
                for (int u = 0; u < 32; u += 4) {
                  const int c = 32 * ch + u;
                  m2[0] = ptx::max3(m2[0], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                  m2[1] = ptx::max3(m2[1], __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
                }
              } else {  // ragged end / diagonal chunk, or scale <= 0
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                  const int c = 32 * ch + u;
                  float x = __uint_as_float(sr[c]);
                  if (!fold) x *= sl;
                  if (!col_ok(c, c_lo, c_hi)) x = -INFINITY;
                  sr[c] = __float_as_uint(x);
                  m2[u & 1] = fmaxf(m2[u & 1], x);
                }
              }
            }
            float mx = fmaxf(m2[0], m2[1]);
            if (fold) mx *= sl;
            const float m_new = fmaxf(m_run, mx);
            if (j == 0) {
              m_run = m_new;
            } else if (m_new > m_run + 8.0f) {  // lazy rescale: only when the max grew by more than 2^8
              alpha = ptx::ex2_approx(m_run - m_new);
              l_run *= alpha;
              m_run = m_new;
              rescale = true;
            }
            const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
            // masked entries hold -inf and give exactly 0; with scale > 0 the
            // entries are still unscaled and take the scale in the packed FMA
            const uint64_t mul2 = ptx::f2_splat(fold ? sl : 1.0f);
            const uint64_t neg2 = ptx::f2_splat(-m_use);
            uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              if (ch >= nch) continue;
              if (!((livem >> ch) & 1u)) {  // no valid key in the chunk: P = 0
#pragma unroll
                for (int u = 0; u < 16; ++u) sr[16 * ch + u] = 0u;
                continue;
              }
  #pragma unroll
              for (int u = 0; u < 16; ++u) {
                const int c = 32 * ch + 2 * u;
                const uint64_t x2 =
                    ptx::f2_fma(ptx::f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), mul2, neg2);
                float a, b;
                ptx::f2_unpack(x2, a, b);
                a = ptx::ex2_approx(a);
                b = ptx::ex2_approx(b);
                acc[u & 3] = ptx::f2_add(acc[u & 3], ptx::f2_pack(a, b));
                sr[16 * ch + u] = ptx::pack_bf16x2(a, b);  // P overwrites scores already consumed
              }
            }
            const uint64_t acc01 = ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3]));
            float sa, sb2;
            ptx::f2_unpack(acc01, sa, sb2);
            l_run += sa + sb2;
          } else {  // GELU
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              if (ch >= nch) continue;
              if (!((livem >> ch) & 1u)) {
#pragma unroll
                for (int u = 0; u < 16; ++u) sr[16 * ch + u] = 0u;
                continue;
              }
              const bool full = (fullm >> ch) & 1u;
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const int c = 32 * ch + 2 * u;
                float a, b;
                act_eval2(ak, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), a, b);
                if (!full) {
                  a = col_ok(c, c_lo, c_hi) ? a : 0.0f;
                  b = col_ok(c + 1, c_lo, c_hi) ? b : 0.0f;
                }
                sr[16 * ch + u] = ptx::pack_bf16x2(a, b);
              }
            }
          }
          // P (bf16 pairs) overwrites the first 16 * nch columns of this S
          // buffer; P V reads no column beyond them.
          ptx::tmem_st32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
          if (nch > 2) ptx::tmem_st32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
          ptx::tmem_wait_st();
        }
      }
      if (g >= 1) {  // O += P(g-1) V(g-1) has landed
        ok = ptx::mbar_wait(&B.o_done, (g - 1) & 1, p.timeout_ns, abort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      if (ACT == kActSoftmax && __any_sync(0xffffffffu, rescale)) {
        ptx::tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          ptx::tmem_ld32(o_addr + 32 * c, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          ptx::tmem_st32(o_addr + 32 * c, r);
        }
        ptx::tmem_wait_st();
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&B.p_full[sb]);
    }
    if (!ok) break;
    if (ACT == kActSoftmax) {  // hand the row sum to the epilogue
      ok = ptx::mbar_wait(&B.l_empty[ob], ((qi / C::NOB) & 1) ^ 1, p.timeout_ns, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      l_buf[ob * 128 + row] = l_run;
      if (KS) m_buf[ob * 128 + row] = m_run;
      ptx::mbar_arrive(&B.l_full[ob]);
      if (!KS && p.lse && row < t.q_rows)
        p.lse[static_cast<size_t>(t.q_tok + row) * p.H + t.h] = row_lse(m_run, l_run);
    }
    ++qi;
  }
  if (!ok && lane == 0) report_failure(p, abort, kStatusActivation);
}

// ------------------------------------------------------------------ epilogue

// Key split: the four warps hold partial results of the same queries over
// disjoint key blocks (row max m_k, row sum l_k, unnormalised O_k).  Thread
// (k, i) weighs its partial row by 2^(m_k - M) / sum_j 2^(m_j - M) l_j (the
// softmax merge; 1/Lkv for GELU), writes it to the exchange buffer, and after
// all four have written sums the four rows over its 16-column share of the
// output row of query i.
template <int D, int ACT>
__device__ __forceinline__ bool epilogue_key_split(const FwdParams& p, FwdBars<D, kModeKeySplit>& B,
                                                   const float* l_buf, const float* m_buf, float* x_buf, uint32_t tmem,
                                                   const ItemView& t, int ob, uint32_t ph, uint32_t& xr, int quarter,
                                                   int lane, bool v8) {
  using C = FwdCfg<D, kModeKeySplit>;
  volatile int* abort = &B.abort;
  float w;
  if (ACT == kActSoftmax) {
    bool ok = ptx::mbar_wait(&B.l_full[ob], ph, p.timeout_ns, abort);
    if (!__all_sync(0xffffffffu, ok)) return false;
    float mk[4], lk[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      mk[k] = m_buf[ob * 128 + 32 * k + lane];
      lk[k] = l_buf[ob * 128 + 32 * k + lane];
    }
    ptx::mbar_arrive(&B.l_empty[ob]);
    const float M = fmaxf(fmaxf(mk[0], mk[1]), fmaxf(mk[2], mk[3]));
    float den = 0.0f, own = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float e = mk[k] == -INFINITY ? 0.0f : ptx::ex2_approx(mk[k] - M);
      den += e * lk[k];
      if (k == quarter) own = e;
    }
    w = den > 0.0f ? own / den : 0.0f;
    if (quarter == 0 && p.lse && lane < t.q_rows)  // sum_j 2^(x_j - M) = den
      p.lse[static_cast<size_t>(t.q_tok + lane) * p.H + t.h] = row_lse(M, den);
  } else {
    w = p.score_scale / static_cast<float>(t.Lkv);  // the GELU's folded scale, then 1/Lkv
  }
  bool ok = ptx::mbar_wait(&B.o_full[ob], ph, p.timeout_ns, abort);
  if (!__all_sync(0xffffffffu, ok)) return false;
  ok = ptx::mbar_wait(&B.x_empty, (xr & 1) ^ 1, p.timeout_ns, abort);
  if (!__all_sync(0xffffffffu, ok)) return false;
  ptx::tc_fence_after();
  const uint32_t o_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + (ob ? C::TM_O1 : C::TM_O0);
  float* xrow = x_buf + (quarter * 32 + lane) * C::X_STRIDE;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t r[32];
    ptx::tmem_ld32(o_addr + 32 * c, r);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; i += 4)
      *reinterpret_cast<float4*>(xrow + 32 * c + i) =
          make_float4(__uint_as_float(r[i]) * w, __uint_as_float(r[i + 1]) * w, __uint_as_float(r[i + 2]) * w,
                      __uint_as_float(r[i + 3]) * w);
  }
  ptx::tc_fence_before();
  ptx::mbar_arrive(&B.o_empty[ob]);  // O[ob] has been read
  ptx::mbar_arrive(&B.x_full);
  ok = ptx::mbar_wait(&B.x_full, xr & 1, p.timeout_ns, abort);
  if (!__all_sync(0xffffffffu, ok)) return false;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float* src = x_buf + (k * 32 + lane) * C::X_STRIDE + 16 * quarter;
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const float4 v = *reinterpret_cast<const float4*>(src + i);
      acc[i] += v.x;
      acc[i + 1] += v.y;
      acc[i + 2] += v.z;
      acc[i + 3] += v.w;
    }
  }
  ptx::mbar_arrive(&B.x_empty);
  ++xr;
  if (lane < t.q_rows) {
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pk[i] = ptx::pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
    __nv_bfloat16* dst = p.out + (static_cast<size_t>(t.q_tok + lane) * p.H + t.h) * D + 16 * quarter;
    if (v8) {
      asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(pk[0]), "r"(pk[1]),
                   "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7])
                   : "memory");
    } else {
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
  }
  return true;
}

template <int D, int ACT, int MODE>
__device__ void run_epilogue(const FwdParams& p, FwdBars<D, MODE>& B, const float* l_buf, const float* m_buf,
                             float* x_buf, uint32_t tmem, int ibeg, int iend, int warp, int lane) {
  using C = FwdCfg<D, MODE>;
  constexpr bool KS = C::KS;
  volatile int* abort = &B.abort;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const int H = p.H;
  const bool v8 = p.out_align32 != 0;
  int qi = 0;
  uint32_t xr = 0;  // key split: exchange rounds
  bool ok = true;
  for (int idx = ibeg; idx < iend && ok; ++idx) {
    const ItemView t = decode_item<MODE>(p, idx);
    __nv_bfloat16* orow = p.out + (static_cast<size_t>(t.q_tok + row) * H + t.h) * D;
    if (t.n_kv == 0) {  // no keys: the output rows are zero
      if (KS ? (quarter == 0 && lane < t.q_rows) : row < t.q_rows) {
        if (KS) orow = p.out + (static_cast<size_t>(t.q_tok + lane) * H + t.h) * D;
        if (ACT == kActSoftmax && p.lse) p.lse[static_cast<size_t>(t.q_tok + (KS ? lane : row)) * H + t.h] = -INFINITY;
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    const int ob = qi % C::NOB;
    const uint32_t ph = (qi / C::NOB) & 1;
    if constexpr (KS) {
      ok = epilogue_key_split<D, ACT>(p, B, l_buf, m_buf, x_buf, tmem, t, ob, ph, xr, quarter, lane, v8);
      ++qi;
      continue;
    }
    float inv;
    if (ACT == kActSoftmax) {
      ok = ptx::mbar_wait(&B.l_full[ob], ph, p.timeout_ns, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const float l = l_buf[ob * 128 + row];
      ptx::mbar_arrive(&B.l_empty[ob]);
      inv = l > 0.0f ? 1.0f / l : 0.0f;
    } else {
      inv = p.score_scale / static_cast<float>(t.Lkv);  // the GELU's folded scale, then 1/Lkv
    }
    ok = ptx::mbar_wait(&B.o_full[ob], ph, p.timeout_ns, abort);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    ptx::tc_fence_after();
    if (__any_sync(0xffffffffu, row < t.q_rows)) {
      const uint32_t o_addr = tmem + lane_off + (ob ? C::TM_O1 : C::TM_O0);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(o_addr + 32 * c, r);
        ptx::tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = ptx::pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
        if (row < t.q_rows) store_row32(orow + 32 * c, pk, v8);
      }
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(&B.o_empty[ob]);
    ++qi;
  }
  if (!ok && lane == 0) report_failure(p, abort, kStatusEpilogue);
}

// ------------------------------------------------------------------ kernel

template <int D, int ACT, int MODE>
__global__ void __launch_bounds__(384, 1) gdpa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D, MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* sm = smem_raw + pad;
  FwdBars<D, MODE>& B = *reinterpret_cast<FwdBars<D, MODE>*>(sm + C::OFF_BAR);
  float* l_buf = reinterpret_cast<float*>(sm + C::OFF_L);
  float* m_buf = reinterpret_cast<float*>(sm + C::OFF_M);  // key split only
  float* x_buf = reinterpret_cast<float*>(sm + C::OFF_X);  // key split only
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ibeg = p.cta_begin[blockIdx.x];
  const int iend = p.cta_begin[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NQ; ++i) {
      ptx::mbar_init(&B.q_full[i], 1);
      ptx::mbar_init(&B.q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&B.s_full[i], 1);
      ptx::mbar_init(&B.p_full[i], 128);
      ptx::mbar_init(&B.o_full[i], 1);
      ptx::mbar_init(&B.o_empty[i], 128);
      ptx::mbar_init(&B.l_full[i], 128);
      ptx::mbar_init(&B.l_empty[i], 128);
    }
    for (int i = 0; i < C::NK; ++i) {
      ptx::mbar_init(&B.k_full[i], 1);
      ptx::mbar_init(&B.k_empty[i], 1);
    }
    for (int i = 0; i < C::NV; ++i) {
      ptx::mbar_init(&B.v_full[i], 1);
      ptx::mbar_init(&B.v_empty[i], 1);
    }
    ptx::mbar_init(&B.o_done, 1);
    ptx::mbar_init(&B.x_full, 128);
    ptx::mbar_init(&B.x_empty, 128);
    ptx::mbar_init(&B.sf_full[0], 128);
    ptx::mbar_init(&B.sf_full[1], 128);
    ptx::mbar_init(&B.mma_drain, 1);
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

  if (warp < 4) {  // warpgroup 0: producers and MMA issuer, few registers
    ptx::regs_dec<C::REGS_CTRL>();
    if (warp == 0) {
      if (lane == 0) run_producer<D, MODE, false>(p, sm, B, ibeg, iend);
    } else if (warp == 2) {
      if (lane == 0) run_producer<D, MODE, true>(p, sm, B, ibeg, iend);
    } else if (warp == 1) {
      run_mma<D, MODE>(p, sm, B, tmem, ibeg, iend);  // the whole warp: MMAs issued warp-uniformly
    }
  } else if (warp < 8) {  // warpgroup 1: activation, a whole row of scores in registers
    ptx::regs_inc<C::REGS_ACT>();
    run_activation<D, ACT, MODE>(p, B, l_buf, m_buf, tmem, ibeg, iend, warp, lane);
  } else {  // warpgroup 2: epilogue, at the launch register count
    run_epilogue<D, ACT, MODE>(p, B, l_buf, m_buf, x_buf, tmem, ibeg, iend, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::TM_COLS);
}

}  // namespace gdpa
