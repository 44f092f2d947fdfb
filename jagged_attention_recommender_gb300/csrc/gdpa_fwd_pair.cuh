// gdpa_fwd_pair.cuh -- jagged GDPA forward, two query tiles per work item.
//
// A work item is 256 query rows of one (sequence, head) -- tile A = rows
// [q0, q0+128), tile B = [q0+128, q0+256), B may be empty -- against the
// sequence's whole key range (full attention) or against the keys of the
// two tiles' block windows, each tile taking only the K/V tiles its rows
// may see (window).  Every K/V tile
// staged in shared memory feeds both tiles' MMAs, which halves the K/V
// traffic per FLOP against one tile per item, and the two activation
// warpgroups (one per tile) take turns with the tensor core:
//
//   MMA warp, per K/V tile g:  O_A += P_A(g-1) V(g-1);  S_A = Q_A K(g)^T;
//                              O_B += P_B(g-1) V(g-1);  S_B = Q_B K(g)^T
//   warpgroup A works on S_A(g) while the tensor core runs the B half, and
//   the other way round.
//
// Items are claimed at run time (see ItemRing): the Q/K producer claims and
// decodes each item and every other role reads it from the ring.
//
// Threads (384, three warpgroups): warpgroup 0 holds the TMA producer for Q
// and K and claimer (warp 0), the MMA issuer + TMEM owner (warp 1, the whole warp runs
// the issue loop and one elected lane issues) and the TMA producer for V
// (warp 2), and hands registers to warpgroups 1 and 2, the activation /
// epilogue of tiles A and B (200 registers a thread, so a whole row of 128
// scores stays in registers: S is read from TMEM once).  TMEM (512
// columns): S_A 0, S_B 128, O_A 256, O_B 384.
#pragma once

#include "gdpa_fwd_common.cuh"

namespace gdpa {

template <int D>
struct PairCfg {
  static constexpr int KCH = D / 64;
  static constexpr int CHUNK_BYTES = 128 * 128;
  static constexpr int TILE_BYTES = KCH * CHUNK_BYTES;  // one 128-row tile of Q, K or V
  static constexpr int NQS = (D == 64) ? 2 : 1;          // Q stages per query tile
  static constexpr int NK = (D == 64) ? 4 : 3;
  static constexpr int NV = (D == 64) ? 4 : 2;
  static constexpr int OFF_QA = 0;
  static constexpr int OFF_QB = OFF_QA + NQS * TILE_BYTES;
  static constexpr int OFF_K = OFF_QB + NQS * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NV * TILE_BYTES;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;
  __host__ __device__ static constexpr uint32_t tm_s(int x) { return x ? 128u : 0u; }    // S_A, S_B
  __host__ __device__ static constexpr uint32_t tm_o(int x) { return x ? 384u : 256u; }  // O_A, O_B
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int THREADS = 384;  // 3 warpgroups
  // Registers per thread after reallocation: the control warpgroup hands
  // registers to the two activation warpgroups.  Each SM sub-partition holds
  // one warp of each, so the launch count R must satisfy
  // REGS_CTRL + 2 REGS_ACT <= 3 R.
  static constexpr int REGS_CTRL = 104;
  static constexpr int REGS_ACT = 200;
  static constexpr int MIN_LAUNCH_REGS = (REGS_CTRL + 2 * REGS_ACT + 2) / 3;
  static_assert(384 + D <= TM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct PairItem {
  int h, q0, kv0, kv_end, n_kv, q_tok, kv_tok, Lkv;
  int rows[2];  // valid rows of tile A and tile B (B may be 0)
  int t0[2], t1[2];  // K/V tiles [t0, t1) of the item each tile attends to
};

template <int D>
struct PairBars {
  uint64_t q_full[2][PairCfg<D>::NQS], q_empty[2][PairCfg<D>::NQS];
  uint64_t k_full[PairCfg<D>::NK], k_empty[PairCfg<D>::NK];
  uint64_t v_full[PairCfg<D>::NV], v_empty[PairCfg<D>::NV];
  uint64_t s_full[2], p_full[2][2], o_done[2], o_empty[2];  // p_full per side and half of the keys
  uint64_t mma_drain;
  ItemRing<PairItem> ring;  // the CTA's items, in claim order
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(PairBars<64>) <= PairCfg<64>::BAR_BYTES && sizeof(PairBars<128>) <= PairCfg<128>::BAR_BYTES, "barrier area");

// Full attention: both tiles attend to every K/V tile of the item.  Block
// window: the item's keys run from the first key tile A's rows may see to
// the last query of tile B; tile A takes the K/V tiles up to its own last
// query, tile B those from the first tile that holds a key its rows may see.
template <bool WIN, bool FLAG = false>
__device__ __forceinline__ PairItem decode_pair(const FwdParams& p, int idx) {
  const int4 it = __ldg(p.items + idx);
  PairItem v;
  const int b = it.x;
  v.h = it.y;
  v.q0 = it.z;
  v.kv0 = WIN ? it.w : 0;
  const ItemRows r = item_rows<FLAG>(p, b);
  v.q_tok = r.qs + v.q0;
  v.kv_tok = r.ks;
  v.Lkv = r.Lkv;
  const int left = r.Lq - v.q0;
  v.rows[0] = max(0, min(128, left));
  v.rows[1] = max(0, min(128, left - 128));
  v.kv_end = WIN ? min(v.Lkv, v.q0 + v.rows[0] + v.rows[1]) : v.Lkv;
  v.n_kv = v.kv_end > v.kv0 && v.rows[0] > 0 ? (v.kv_end - v.kv0 + 127) / 128 : 0;  // no rows: nothing to do
  v.t0[0] = 0;
  v.t1[0] = v.n_kv;
  v.t0[1] = 0;
  v.t1[1] = v.rows[1] > 0 ? v.n_kv : 0;
  if (WIN) {
    const int end_a = min(v.Lkv, v.q0 + 128);
    v.t1[0] = end_a > v.kv0 ? (end_a - v.kv0 + 127) / 128 : 0;
    const int blk = (v.q0 + 128) / 64 - (p.window_blocks - 1);
    const int lo_b = blk > 0 ? blk * 64 : 0;
    v.t0[1] = (lo_b - v.kv0) / 128;
  }
  return v;
}

// ------------------------------------------------------------------ producer

// Two producer threads: one stages Q and K, the other V, so that a K load
// never waits behind a V slot.
// The Q/K producer thread is also the CTA's claimer: it claims each item,
// decodes it (flagging a bad plan) and publishes it for the other roles
// before staging its Q and K tiles; the V producer reads the items from the
// ring.
template <int D, bool WIN, bool LOAD_V>
__device__ void pair_producer(const FwdParams& p, uint8_t* sm, PairBars<D>& B) {
  using C = PairCfg<D>;
  volatile int* abort = &B.abort;
  int qn[2] = {0, 0};
  uint32_t g = 0;
  bool ok = true;
  int q_armed[2][C::NQS], k_armed[C::NK], v_armed[C::NV];
  for (int t = 0; t < 2; ++t)
    for (int s = 0; s < C::NQS; ++s) q_armed[t][s] = -1;
  for (int s = 0; s < C::NK; ++s) k_armed[s] = -1;
  for (int s = 0; s < C::NV; ++s) v_armed[s] = -1;
  if (LOAD_V) {
    ptx::prefetch_tensormap(&p.tm_v);
  } else {
    ptx::prefetch_tensormap(&p.tm_q);
    ptx::prefetch_tensormap(&p.tm_k);
  }
  ListClaim L;
  if (!LOAD_V) L = claim_init(p);
  for (uint32_t k = 0; ok; ++k) {
    PairItem t;
    if (!LOAD_V) {
      const int idx = claim_next(p, L);
      if (idx >= 0) t = decode_pair<WIN, true>(p, idx);
      ok = ring_publish(p, B.ring, k, t, idx >= 0, abort);
      if (!ok || idx < 0) break;
    } else if (!ring_read(p, B.ring, k, t, 0u, abort, ok)) {
      break;
    }
    if (t.n_kv == 0) continue;
    if (!LOAD_V) {
      for (int x = 0; x < 2 && ok; ++x) {
        if (t.rows[x] == 0) continue;
        const int s = qn[x] % C::NQS;
        const uint32_t ph = (qn[x] / C::NQS) & 1;
        ok = ptx::mbar_wait(&B.q_empty[x][s], ph ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&B.q_full[x][s], C::TILE_BYTES);
        q_armed[x][s] = (int)ph;
        uint8_t* sq = sm + (x ? C::OFF_QB : C::OFF_QA) + s * C::TILE_BYTES;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          ptx::tma_load_2d(sq + c * C::CHUNK_BYTES, &p.tm_q, &B.q_full[x][s], t.h * D + 64 * c, t.q_tok + 128 * x);
        ++qn[x];
      }
    }
    for (int j = 0; j < t.n_kv && ok; ++j, ++g) {
      const int y = t.kv_tok + t.kv0 + 128 * j;
      if (!LOAD_V) {
        const int sk = g % C::NK;
        const uint32_t phk = (g / C::NK) & 1;
        ok = ptx::mbar_wait(&B.k_empty[sk], phk ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&B.k_full[sk], C::TILE_BYTES);
        uint8_t* dk = sm + C::OFF_K + sk * C::TILE_BYTES;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          ptx::tma_load_2d(dk + c * C::CHUNK_BYTES, &p.tm_k, &B.k_full[sk], t.h * D + 64 * c, y);
        k_armed[sk] = (int)phk;
      } else {
        const int sv = g % C::NV;
        const uint32_t phv = (g / C::NV) & 1;
        ok = ptx::mbar_wait(&B.v_empty[sv], phv ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&B.v_full[sv], C::TILE_BYTES);
        uint8_t* dv = sm + C::OFF_V + sv * C::TILE_BYTES;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          ptx::tma_load_2d(dv + c * C::CHUNK_BYTES, &p.tm_v, &B.v_full[sv], t.h * D + 64 * c, y);
        v_armed[sv] = (int)phv;
      }
    }
  }
  if (!ok) report_failure(p, abort, kStatusProducer);
  const int never = 0;
  const unsigned long long drain_ns = 100000000ull;
  for (int x = 0; x < 2; ++x)
    for (int s = 0; s < C::NQS; ++s)
      if (q_armed[x][s] >= 0) ptx::mbar_wait(&B.q_full[x][s], (uint32_t)q_armed[x][s], drain_ns, &never);
  for (int s = 0; s < C::NK; ++s)
    if (k_armed[s] >= 0) ptx::mbar_wait(&B.k_full[s], (uint32_t)k_armed[s], drain_ns, &never);
  for (int s = 0; s < C::NV; ++s)
    if (v_armed[s] >= 0) ptx::mbar_wait(&B.v_full[s], (uint32_t)v_armed[s], drain_ns, &never);
}

// ------------------------------------------------------------------ MMA issuer

struct PairPV {
  uint32_t gx;  // this side's tile counter
  uint32_t g;   // K/V tile counter (selects the V stage)
  int item;     // this side's item counter
  int first, last, n16;
};

// O_x += P_x V for one K/V tile, in two halves of the keys: the activation
// signals P of keys 0-63 before it computes keys 64-127, so the first four
// MMAs run while it finishes the row.  Only an item's last P V signals
// o_done (its epilogue waits for it): the scores' barrier already implies
// every earlier P V of the side, since a commit tracks all the issuing
// thread's earlier MMAs and S_x(g) is issued after O_x += P_x(g-1) V(g-1).
template <int D>
__device__ __forceinline__ bool pair_issue_pv(const FwdParams& p, uint8_t* sm, PairBars<D>& B, uint32_t tmem, int x,
                                              const PairPV& P) {
  using C = PairCfg<D>;
  volatile int* abort = &B.abort;
  if (!ptx::mbar_wait(&B.p_full[x][0], P.gx & 1, p.timeout_ns, abort)) return false;
  if (P.first && !ptx::mbar_wait(&B.o_empty[x], (P.item & 1) ^ 1, p.timeout_ns, abort)) return false;
  const int sv = P.g % C::NV;
  if (!ptx::mbar_wait(&B.v_full[sv], (P.g / C::NV) & 1, p.timeout_ns, abort)) return false;
  ptx::tc_fence_after();
  // One descriptor, advanced by 16 keys (2048 bytes, 128 in the address
  // field) per MMA: the V stage lies below 256 KB, so the 14-bit field
  // never carries.
  const uint64_t bd0 = ptx::sdesc_sw128(ptx::smem_u32(sm + C::OFF_V + sv * C::TILE_BYTES), C::CHUNK_BYTES, 1024);
  constexpr uint32_t idesc = ptx::idesc_bf16(128, D, 1);
  const uint32_t d_tm = tmem + C::tm_o(x), a_tm = tmem + C::tm_s(x);
  const uint32_t acc0 = P.first ? 0u : 1u;
  const int n_lo = min(P.n16, 4);
  if (n_lo == 4) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) ptx::mma_ts_elect(d_tm, a_tm + 8 * kk, bd0 + 128u * kk, idesc, kk == 0 ? acc0 : 1u);
  } else {
    for (int kk = 0; kk < n_lo; ++kk) ptx::mma_ts_elect(d_tm, a_tm + 8 * kk, bd0 + 128u * kk, idesc, kk == 0 ? acc0 : 1u);
  }
  if (!ptx::mbar_wait(&B.p_full[x][1], P.gx & 1, p.timeout_ns, abort)) return false;
  ptx::tc_fence_after();
  if (P.n16 == 8) {
#pragma unroll
    for (int kk = 4; kk < 8; ++kk) ptx::mma_ts_elect(d_tm, a_tm + 8 * kk, bd0 + 128u * kk, idesc, 1u);
  } else {
    for (int kk = 4; kk < P.n16; ++kk) ptx::mma_ts_elect(d_tm, a_tm + 8 * kk, bd0 + 128u * kk, idesc, 1u);
  }
  if (P.last) ptx::mma_commit_elect(&B.o_done[x]);
  return true;
}

template <int D, bool WIN>
__device__ void pair_mma(const FwdParams& p, uint8_t* sm, PairBars<D>& B, uint32_t tmem) {
  using C = PairCfg<D>;
  volatile int* abort = &B.abort;
  int qn[2] = {0, 0};       // items seen by each side (Q stage and O buffer use counts)
  uint32_t gx[2] = {0, 0};  // tiles processed by each side
  uint32_t g = 0;
  bool ok = true;
  bool pend[2] = {false, false};
  PairPV pv[2] = {{0, 0, 0, 0, 0, 0}, {0, 0, 0, 0, 0, 0}};
  // Every staged V tile is read by tile A's P V (an item without rows in
  // tile A has no tiles), so its release always follows a read that waited
  // for the load: the producer never refills a stage with a copy in flight.
  bool pend_v = false;
  uint32_t pend_v_g = 0;
  for (uint32_t k = 0; ok; ++k) {
    PairItem t;
    if (!ring_read(p, B.ring, k, t, 0xffffffffu, abort, ok)) break;
    if (t.n_kv == 0) continue;
    const bool has[2] = {t.rows[0] > 0, t.rows[1] > 0};
    uint32_t q_base[2] = {0, 0};
    for (int x = 0; x < 2 && ok; ++x) {
      if (!has[x]) continue;
      const int s = qn[x] % C::NQS;
      ok = ptx::mbar_wait(&B.q_full[x][s], (qn[x] / C::NQS) & 1, p.timeout_ns, abort);
      q_base[x] = ptx::smem_u32(sm + (x ? C::OFF_QB : C::OFF_QA) + s * C::TILE_BYTES);
    }
    if (!ok) break;
    for (int j = 0; j < t.n_kv; ++j, ++g) {
      // O_A += P_A(prev) V(prev) needs no K: issue it before waiting for K(g).
      if (pend[0]) {
        ok = pair_issue_pv<D>(p, sm, B, tmem, 0, pv[0]);
        if (!ok) break;
        pend[0] = false;
      }
      const int sk = g % C::NK;
      ok = ptx::mbar_wait(&B.k_full[sk], (g / C::NK) & 1, p.timeout_ns, abort);
      if (!ok) break;
      ptx::tc_fence_after();
      const int ncols = min(128, t.kv_end - t.kv0 - 128 * j);
      const int n16 = (ncols + 15) >> 4;
      const uint32_t idesc = ptx::idesc_bf16(128, n16 * 16, 0);
      const uint32_t k_base = ptx::smem_u32(sm + C::OFF_K + sk * C::TILE_BYTES);
      bool act[2];
      for (int x = 0; x < 2; ++x) {
        // O_x += P_x(prev) V(prev) must precede S_x = Q_x K^T: P_x lives in
        // S_x's columns.  A pending P V is issued here even when this tile
        // has no S_x, so that every P V of the previous tile is issued now.
        if (pend[x]) {
          ok = pair_issue_pv<D>(p, sm, B, tmem, x, pv[x]);
          if (!ok) break;
          pend[x] = false;
        }
        act[x] = has[x] && j >= t.t0[x] && j < t.t1[x];
        if (!act[x]) continue;
        // descriptors advanced in their address field (16-byte units)
        const uint64_t qd = ptx::sdesc_sw128(q_base[x], 16, 1024), kd = ptx::sdesc_sw128(k_base, 16, 1024);
        const uint32_t d_tm = tmem + C::tm_s(x);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4;
          ptx::mma_ss_elect(d_tm, qd + off, kd + off, idesc, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit_elect(&B.s_full[x]);
      }
      if (!ok) break;
      if (pend_v) ptx::mma_commit_elect(&B.v_empty[pend_v_g % C::NV]);  // both P V of the previous tile issued
      ptx::mma_commit_elect(&B.k_empty[sk]);
      if (j == t.n_kv - 1) {
        for (int x = 0; x < 2; ++x)
          if (has[x]) ptx::mma_commit_elect(&B.q_empty[x][qn[x] % C::NQS]);
      }
      for (int x = 0; x < 2; ++x) {
        if (!act[x]) continue;
        pv[x] = PairPV{gx[x], g, qn[x], j == t.t0[x] ? 1 : 0, j == t.t1[x] - 1 ? 1 : 0, n16};
        pend[x] = true;
        ++gx[x];
      }
      pend_v = true;
      pend_v_g = g;
    }
    for (int x = 0; x < 2; ++x)
      if (has[x]) ++qn[x];
  }
  for (int x = 0; x < 2 && ok; ++x)
    if (pend[x]) ok = pair_issue_pv<D>(p, sm, B, tmem, x, pv[x]);
  if (ok && pend_v) ptx::mma_commit_elect(&B.v_empty[pend_v_g % C::NV]);
  if (!ok) report_failure(p, abort, kStatusMma);
  ptx::mma_commit_elect(&B.mma_drain);
  const int never = 0;
  ptx::mbar_wait(&B.mma_drain, 0, 100000000ull, &never);
}

// ------------------------------------------------------------------ activation + epilogue

template <int D, int ACT, bool WIN>
__device__ void pair_activation(const FwdParams& p, PairBars<D>& B, uint32_t tmem, int x, int warp, int lane) {
  using C = PairCfg<D>;
  volatile int* abort = &B.abort;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t s_addr = tmem + lane_off + C::tm_s(x);
  const uint32_t o_addr = tmem + lane_off + C::tm_o(x);
  const float sl = p.score_scale;
  const ActK ak = act_k(p.act_a, p.act_c, p.act_sfu);  // GELU / SiLU: the scale folded into the cubic
  const int H = p.H;
  uint32_t gx = 0;  // this side's K/V tiles (phase of s_full, p_full)
  uint32_t ix = 0;  // this side's items (phase of o_done)
  bool ok = true;
  for (uint32_t k = 0; ok; ++k) {
    PairItem t;
    if (!ring_read(p, B.ring, k, t, 0xffffffffu, abort, ok)) break;
    const int rows = x ? t.rows[1] : t.rows[0];
    __nv_bfloat16* orow = p.out + (static_cast<size_t>(t.q_tok + 128 * x + row) * H + t.h) * D;
    if (t.n_kv == 0) {  // no keys: zero output rows
      if (row < rows) {
        if (ACT == kActSoftmax && p.lse) p.lse[static_cast<size_t>(t.q_tok + 128 * x + row) * H + t.h] = -INFINITY;
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    if (rows == 0) continue;  // this side has no tile in the item
    const bool rows_live = __any_sync(0xffffffffu, row < rows);
    float m_run = -INFINITY, l_run = 0.0f;
    const int i_seq = t.q0 + 128 * x + row;  // query index inside its sequence
    int win_lo = 0;
    if (WIN) {
      const int blk = i_seq / 64 - (p.window_blocks - 1);
      win_lo = blk > 0 ? blk * 64 : 0;
    }
    const int j0 = x ? t.t0[1] : t.t0[0], j1 = x ? t.t1[1] : t.t1[0];  // this side's K/V tiles
    const int kv0 = t.kv0, kv_end = t.kv_end;
    const float inv_lkv = sl / static_cast<float>(max(t.Lkv, 1));  // the GELU's folded scale, then 1/Lkv
    for (int j = j0; j < j1; ++j, ++gx) {
      ok = ptx::mbar_wait(&B.s_full[x], gx & 1, p.timeout_ns, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      float alpha = 1.0f;
      bool rescale = false;
      if (rows_live) {
        // valid key columns of this row: [c_lo, c_hi] (tile-relative)
        const int kv_t0 = kv0 + 128 * j;
        const int ncols = min(128, kv_end - kv_t0);  // the tile's key extent
        int c_lo = 0, c_hi = ncols - 1;
        if (WIN) {
          c_lo = max(0, win_lo - kv_t0);
          c_hi = min(c_hi, i_seq - kv_t0);
        }
        const int nch = (ncols + 31) >> 5;  // chunks P V reads
        // chunk classes agreed on by the warp: bit ch of `fullm` = every key
        // of chunk ch is valid for all 32 rows; bit ch of `livem` = some row
        // has a valid key in it.  Full attention masks only the ragged end
        // of the last tile, the same for every row.
        uint32_t fullm, livem;
        if (WIN) {
          fullm = 0;
          livem = 0;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int lo = 32 * ch, hi = 32 * ch + 31;
            if (__all_sync(0xffffffffu, lo >= c_lo && hi <= c_hi)) fullm |= 1u << ch;
            if (__any_sync(0xffffffffu, ch < nch && hi >= c_lo && lo <= c_hi)) livem |= 1u << ch;
          }
        } else {
          livem = (1u << nch) - 1u;
          fullm = (1u << (ncols >> 5)) - 1u;
        }
        if constexpr (ACT != kActSoftmax) {
          // ALU activation: no row maximum, so the scores stream through
          // registers 32 columns at a time (the next chunk's load in flight
          // while this one is evaluated), which keeps the packed fp32x2
          // polynomial's register pairs from spilling.  P chunk ch lands on
          // columns [16 ch, 16 ch + 16), scores this thread has already read.
          uint32_t sc[2][32];
          if (livem & 1u) ptx::tmem_ld32(s_addr, sc[0]);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            if (ch >= nch) continue;
            ptx::tmem_wait_ld_r32(sc[ch & 1]);
            if (ch + 1 < nch && ((livem >> (ch + 1)) & 1u)) ptx::tmem_ld32(s_addr + 32 * (ch + 1), sc[(ch + 1) & 1]);
            uint32_t pk[16];
            if (!((livem >> ch) & 1u)) {
#pragma unroll
              for (int u = 0; u < 16; ++u) pk[u] = 0u;
            } else {
              const bool full = (fullm >> ch) & 1u;
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const int c = 32 * ch + 2 * u;
                float e0, e1;
                act_eval2(ak, __uint_as_float(sc[ch & 1][2 * u]), __uint_as_float(sc[ch & 1][2 * u + 1]), e0, e1);
                if (!full) {
                  e0 = (c >= c_lo && c <= c_hi) ? e0 : 0.0f;
                  e1 = (c + 1 >= c_lo && c + 1 <= c_hi) ? e1 : 0.0f;
                }
                pk[u] = ptx::pack_bf16x2(e0, e1);
              }
            }
            ptx::tmem_st16(s_addr + 16 * ch, pk);
            if (ch == 1) {  // keys 0-63 done: their P V may start
              ptx::tmem_wait_st();
              ptx::tc_fence_before();
              ptx::mbar_arrive(&B.p_full[x][0]);
            }
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          if (nch <= 1) ptx::mbar_arrive(&B.p_full[x][0]);
          ptx::mbar_arrive(&B.p_full[x][1]);
        } else {
        // The whole row of scores in registers, one TMEM round trip.
        uint32_t sr[128];
        // A whole tile of valid keys (softmax, scale > 0): the second half
        // of the row loads while the first half's maximum is taken.
        const bool split_ld = !WIN && ACT == kActSoftmax && fullm == 0xFu && sl > 0.0f;
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (split_ld) {
          ptx::tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
          ptx::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
          ptx::tmem_wait_ld_r64(&sr[0]);
          ptx::tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
          ptx::tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            m4[0] = ptx::max3(m4[0], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            m4[1] = ptx::max3(m4[1], __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
            m4[2] = ptx::max3(m4[2], __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
            m4[3] = ptx::max3(m4[3], __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
          }
          ptx::tmem_wait_ld_r64(&sr[64]);
#pragma unroll
          for (int c = 64; c < 128; c += 8) {
            m4[0] = ptx::max3(m4[0], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            m4[1] = ptx::max3(m4[1], __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
            m4[2] = ptx::max3(m4[2], __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
            m4[3] = ptx::max3(m4[3], __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch)
            if ((livem >> ch) & 1u) ptx::tmem_ld32(s_addr + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * ch]));
          ptx::tmem_wait_ld();
        }
        {
          // Scores in log2 units: x = s * scale * log2(e); masked columns
          // become -inf.  With scale > 0 the scaling is folded into the
          // exponent's FMA; otherwise it is applied first.
          const bool fold = sl > 0.0f;
          if (split_ld) {
            // maximum taken with the loads
          } else
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            if (!((livem >> ch) & 1u)) continue;
            if (((fullm >> ch) & 1u) && fold) {
#pragma unroll
              for (int u = 0; u < 32; u += 8) {
                const int c = 32 * ch + u;
                m4[0] = ptx::max3(m4[0], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                m4[1] = ptx::max3(m4[1], __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
                m4[2] = ptx::max3(m4[2], __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
                m4[3] = ptx::max3(m4[3], __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
              }
            } else {  // ragged end / window edge / diagonal chunk, or scale <= 0
#pragma unroll
              for (int u = 0; u < 32; ++u) {
                const int c = 32 * ch + u;
                float v = __uint_as_float(sr[c]);
                if (!fold) v *= sl;
                if (c < c_lo || c > c_hi) v = -INFINITY;
                sr[c] = __float_as_uint(v);
                m4[u & 3] = fmaxf(m4[u & 3], v);
              }
            }
          }
          float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
          if (fold) mx *= sl;
          const float m_new = fmaxf(m_run, mx);
          if (j == j0) {
            m_run = m_new;
          } else if (m_new > m_run + 8.0f) {
            alpha = ptx::ex2_approx(m_run - m_new);
            l_run *= alpha;
            m_run = m_new;
            rescale = true;
          }
          // O rescale before this tile's P: the scores' barrier implies that
          // O_x += P_x(g-1) V(g-1) has completed (see pair_issue_pv)
          // (16 columns at a time: the row of scores is still in registers)
          if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
              uint32_t r[16];
              ptx::tmem_ld16(o_addr + 16 * c, r);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
              ptx::tmem_st16(o_addr + 16 * c, r);
            }
          }
          const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
          // masked entries hold -inf and give exactly 0; with scale > 0 the
          // entries are still unscaled and take the scale in the FMA.  The
          // exponent's argument is a scalar FMA and the row sum a packed
          // add: packing both (fma.f32x2 into add.f32x2) measured about
          // twice as slow, the register pairs it needs pushing the row of
          // scores out of registers.  P goes to TMEM chunk by chunk (16
          // columns of bf16 pairs over scores already held in registers).
          const float mul = fold ? sl : 1.0f, nm = -m_use;
          uint64_t acc[4] = {0, 0, 0, 0};  // +0.0f pairs
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            if (ch >= nch) continue;
            uint32_t pk[16];
            if (!((livem >> ch) & 1u)) {  // no valid key in the chunk: P = 0
#pragma unroll
              for (int u = 0; u < 16; ++u) pk[u] = 0u;
            } else {
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const int c = 32 * ch + 2 * u;
                const float e0 = ptx::ex2_approx(fmaf(__uint_as_float(sr[c]), mul, nm));
                const float e1 = ptx::ex2_approx(fmaf(__uint_as_float(sr[c + 1]), mul, nm));
                acc[u & 3] = ptx::f2_add(acc[u & 3], ptx::f2_pack(e0, e1));
                pk[u] = ptx::pack_bf16x2(e0, e1);
              }
            }
            ptx::tmem_st16(s_addr + 16 * ch, pk);
            if (ch == 1) {  // keys 0-63 done (and O rescaled): their P V may start
              ptx::tmem_wait_st();
              ptx::tc_fence_before();
              ptx::mbar_arrive(&B.p_full[x][0]);
            }
          }
          const uint64_t acc01 = ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3]));
          float sa, sb;
          ptx::f2_unpack(acc01, sa, sb);
          l_run += sa + sb;
        }
        // P (bf16 pairs) now covers the first 16 * nch columns of S_x; P V
        // reads no column beyond them.
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        if (nch <= 1) ptx::mbar_arrive(&B.p_full[x][0]);
        ptx::mbar_arrive(&B.p_full[x][1]);
        }
      } else {  // no valid row in this warp: nothing to compute
        ptx::tc_fence_before();
        ptx::mbar_arrive(&B.p_full[x][0]);
        ptx::mbar_arrive(&B.p_full[x][1]);
      }
    }
    if (!ok) break;
    ok = ptx::mbar_wait(&B.o_done[x], ix & 1, p.timeout_ns, abort);  // the item's last P V
    ++ix;
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    ptx::tc_fence_after();
    const float inv = (ACT == kActSoftmax) ? (l_run > 0.0f ? 1.0f / l_run : 0.0f) : inv_lkv;
    if (ACT == kActSoftmax && p.lse && row < rows)
      p.lse[static_cast<size_t>(t.q_tok + 128 * x + row) * H + t.h] = row_lse(m_run, l_run);
    if (rows_live) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        ptx::tmem_ld32(o_addr + 32 * c, r);
        ptx::tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = ptx::pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
        if (row < rows) store_row32(orow + 32 * c, pk, p.out_align32 != 0);
      }
    }
    ptx::tc_fence_before();
    // failure-path test: one warp of CTA 0 withholds the first item's arrival
    const bool withhold = p.test_skip_arrive && blockIdx.x == 0 && warp == 4 && ix == 1;
    if (!withhold) ptx::mbar_arrive(&B.o_empty[x]);
  }
  if (!ok && lane == 0) report_failure(p, abort, kStatusActivation);
}

// ------------------------------------------------------------------ kernel

template <int D, int ACT, bool WIN>
__global__ void __launch_bounds__(384, 1) gdpa_fwd_pair_kernel(const __grid_constant__ FwdParams p) {
  static_assert(!WIN, "block windows run on the 64-key pair kernel (gdpa_fwd_pair64.cuh)");
  using C = PairCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* sm = smem_raw + pad;
  PairBars<D>& B = *reinterpret_cast<PairBars<D>*>(sm + C::OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      for (int s = 0; s < C::NQS; ++s) {
        ptx::mbar_init(&B.q_full[x][s], 1);
        ptx::mbar_init(&B.q_empty[x][s], 1);
      }
      ptx::mbar_init(&B.s_full[x], 1);
      ptx::mbar_init(&B.p_full[x][0], 128);
      ptx::mbar_init(&B.p_full[x][1], 128);
      ptx::mbar_init(&B.o_done[x], 1);
      ptx::mbar_init(&B.o_empty[x], 128);
    }
    for (int s = 0; s < C::NK; ++s) {
      ptx::mbar_init(&B.k_full[s], 1);
      ptx::mbar_init(&B.k_empty[s], 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      ptx::mbar_init(&B.v_full[s], 1);
      ptx::mbar_init(&B.v_empty[s], 1);
    }
    ptx::mbar_init(&B.mma_drain, 1);
    for (int r = 0; r < kRing; ++r) {  // readers: the V producer, the MMA warp, the eight activation warps
      ptx::mbar_init(&B.ring.full[r], 1);
      ptx::mbar_init(&B.ring.empty[r], 10);
    }
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
      if (lane == 0) pair_producer<D, WIN, false>(p, sm, B);
    } else if (warp == 2) {
      if (lane == 0) pair_producer<D, WIN, true>(p, sm, B);
    } else if (warp == 1) {
      pair_mma<D, WIN>(p, sm, B, tmem);  // the whole warp: MMAs issued warp-uniformly
    }
  } else {  // warpgroups 1 and 2: tiles A and B, a whole row of scores in registers
    ptx::regs_inc<C::REGS_ACT>();
    pair_activation<D, ACT, WIN>(p, B, tmem, warp < 8 ? 0 : 1, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::TM_COLS);
  if (threadIdx.x == 0) claim_finish(p);
}

}  // namespace gdpa
