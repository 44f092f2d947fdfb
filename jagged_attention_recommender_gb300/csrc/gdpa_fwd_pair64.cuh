// gdpa_fwd_pair64.cuh -- jagged GDPA forward, two query tiles per work item,
// 64-key K/V tiles with the scores double-buffered (block windows and short
// key ranges; long key ranges take gdpa_fwd_pair.cuh).
//
// A work item is 256 query rows of one (sequence, head) -- tile A = rows
// [q0, q0+128), tile B = [q0+128, q0+256), B may be empty -- against the
// sequence's whole key range (full attention) or against the keys of the
// two tiles' block windows, each tile taking only the K/V tiles its rows
// may see (window).  Every K/V tile staged in shared memory feeds both
// tiles' MMAs, which halves the K/V traffic per FLOP against one tile per
// item.
//
// K/V tiles are 64 keys, and each side has two S buffers in tensor memory.
// Each side has its own MMA warp, which for every K/V tile g its rows attend
// to issues S_x(g) = Q_x K(g)^T into one buffer and then O_x += P_x(g-1)
// V(g-1) from the other (the P of the previous tile), so when a side's
// activation has finished a tile its next scores are already there:
//
//   MMA warp of side x, per K/V tile g:  S_x(g)                (buffer g & 1)
//                                        O_x += P_x(g-1) V(g-1)
//
// This look-ahead also crosses item boundaries (the next item's Q is staged
// ahead), which is what a one-tile key range needs (the "outer loop"
// pipelining of the GDPA section of the techfeed summary of "GEM Training").
// With 64-key tiles a block window's 64-key blocks are whole tiles, so each
// side skips every block outside its window; the two sides' windows start
// two tiles apart, and with separate issuers (and five K/V stages for
// windows at D = 128) neither side waits for the other's tiles.  Each K/V
// stage is released by both MMA warps, a side that does not attend to a
// tile releasing it once it has landed.
//
// Items are claimed at run time (see ItemRing): the Q/K producer claims and
// decodes each item and every other role reads it from the ring.
//
// Threads (384, three warpgroups): warpgroup 0 holds the TMA producer for Q
// and K and claimer (warp 0), the MMA issuers of tiles A and B (warps 1 and
// 3; the whole warp runs the issue loop and one elected lane issues; warp 1
// owns the tensor memory) and the TMA producer for V (warp 2), and hands its
// registers to warpgroups 1 and 2, the activation/epilogue of tiles A and B.
// TMEM (512 columns): S_A buffers 0 and 64, S_B buffers 128 and 192, O_A 256,
// O_B 384.  An activation thread holds one query row; it reads its 64 scores
// of a tile from TMEM at once.
#pragma once

#include "gdpa_fwd_common.cuh"

namespace gdpa {

template <int D, bool WIN>
struct Pair64Cfg {
  static constexpr int BN = 64;                           // keys per K/V tile
  static constexpr int KCH = D / 64;
  static constexpr int Q_CHUNK = 128 * 128;               // Q: 128 rows x 128 bytes per 64-column chunk
  static constexpr int Q_TILE = KCH * Q_CHUNK;
  static constexpr int KV_CHUNK = BN * 128;               // K/V: 64 rows x 128 bytes per chunk
  static constexpr int KV_TILE = KCH * KV_CHUNK;
  // Windows store whole 128-row output tiles in bulk through a staging area
  // per side (full attention keeps per-thread stores: there the area would
  // cost a K and a V stage, which measured slower: cross_gelu 0.456 -> 0.482 ms).
  static constexpr bool BULK = WIN;
  // Q stages per query tile, K and V stages: block windows at D = 128 trade
  // the second Q stage for more K/V stages, so that a side may run ahead of
  // the other (their windows start two tiles apart).
  static constexpr int NQS = (WIN && D == 128) ? 1 : 2;
  static constexpr int NK = (D == 64) ? 6 : (WIN ? 4 : 3);
  static constexpr int NV = (D == 64) ? 6 : (WIN ? 4 : 3);
  static constexpr int OFF_QA = 0;
  static constexpr int OFF_QB = OFF_QA + NQS * Q_TILE;
  static constexpr int OFF_K = OFF_QB + NQS * Q_TILE;
  static constexpr int OFF_V = OFF_K + NK * KV_TILE;
  // Output staging, one area per side: 128 rows x 64 columns of bf16 in the
  // 128-byte-swizzled layout of the output tensor map's box, written by the
  // side's threads and stored by one bulk tensor store per 64 columns.
  static constexpr int STG_BYTES = 128 * 128;
  static constexpr int OFF_STG = OFF_V + NV * KV_TILE;
  static constexpr int OFF_BAR = OFF_STG + (BULK ? 2 * STG_BYTES : 0);
  static constexpr int BAR_BYTES = 1024;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;
  __host__ __device__ static constexpr uint32_t tm_s(int x, int b) { return 128u * x + 64u * b; }  // S_x buffer b
  __host__ __device__ static constexpr uint32_t tm_o(int x) { return x ? 384u : 256u; }           // O_A, O_B
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int THREADS = 384;  // 3 warpgroups
  // Registers per thread after reallocation: the control warpgroup hands
  // registers to the two activation warpgroups (the split that compiled
  // without spills for each activation).  Each SM sub-partition holds one
  // warp of each, so the launch count R must satisfy
  // regs_ctrl + 2 regs_act <= 3 R.
  __host__ __device__ static constexpr int regs_ctrl(int act) { return act == kActGelu ? 120 : 88; }
  __host__ __device__ static constexpr int regs_act(int act) { return act == kActGelu ? 192 : 208; }
  static constexpr int MIN_LAUNCH_REGS = 168;
  static_assert(regs_ctrl(kActGelu) + 2 * regs_act(kActGelu) <= 3 * MIN_LAUNCH_REGS, "register split");
  static_assert(regs_ctrl(kActSoftmax) + 2 * regs_act(kActSoftmax) <= 3 * MIN_LAUNCH_REGS, "register split");
  static_assert(384 + D <= TM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(OFF_STG % 1024 == 0, "staging areas on the swizzle's 1024-byte period");
};

struct Pair64Item {
  int h, q0, kv0, kv_end, n_kv, q_tok, kv_tok, Lkv;
  int rows[2];       // valid rows of tile A and tile B (B may be 0)
  int t0[2], t1[2];  // K/V tiles [t0, t1) of the item each query tile attends to
};

template <int D, bool WIN>
struct Pair64Bars {
  uint64_t q_full[2][Pair64Cfg<D, WIN>::NQS], q_empty[2][Pair64Cfg<D, WIN>::NQS];
  uint64_t k_full[Pair64Cfg<D, WIN>::NK], k_empty[Pair64Cfg<D, WIN>::NK];
  uint64_t v_full[Pair64Cfg<D, WIN>::NV], v_empty[Pair64Cfg<D, WIN>::NV];
  uint64_t s_full[2][2], p_full[2][2];  // per side and S buffer
  uint64_t o_done[2], o_empty[2];
  uint64_t mma_drain[2];  // one per MMA warp
  uint64_t epi_bar[2];    // per side: its 128 activation threads meet around a bulk output store
  ItemRing<Pair64Item> ring;  // the CTA's items, in claim order
  uint32_t tmem_slot;
  int abort;
};
static_assert(sizeof(Pair64Bars<64, false>) <= Pair64Cfg<64, false>::BAR_BYTES &&
                  sizeof(Pair64Bars<128, false>) <= Pair64Cfg<128, false>::BAR_BYTES &&
                  sizeof(Pair64Bars<64, true>) <= Pair64Cfg<64, true>::BAR_BYTES &&
                  sizeof(Pair64Bars<128, true>) <= Pair64Cfg<128, true>::BAR_BYTES,
              "barrier area");

// Full attention: both tiles attend to every K/V tile of the item.  Block
// window: the item's keys run from the first key tile A's rows may see to
// the last query of tile B; each tile takes the 64-key blocks of its own
// window (blocks are K/V tiles).
template <bool WIN, bool FLAG = false>
__device__ __forceinline__ Pair64Item decode_pair64_from(const FwdParams& p, const int4 it, const SeqOffs& offs) {
  constexpr int BN = 64;
  Pair64Item v;
  v.h = it.y;
  v.q0 = it.z;
  v.kv0 = WIN ? it.w : 0;
  const ItemRows r = item_rows_from<FLAG>(p, offs);
  v.q_tok = r.qs + v.q0;
  v.kv_tok = r.ks;
  v.Lkv = r.Lkv;
  const int left = r.Lq - v.q0;
  v.rows[0] = max(0, min(128, left));
  v.rows[1] = max(0, min(128, left - 128));
  v.kv_end = WIN ? min(v.Lkv, v.q0 + v.rows[0] + v.rows[1]) : v.Lkv;
  v.n_kv = v.kv_end > v.kv0 && v.rows[0] > 0 ? (v.kv_end - v.kv0 + BN - 1) / BN : 0;  // no rows: nothing to do
  v.t0[0] = 0;
  v.t1[0] = v.n_kv;
  v.t0[1] = 0;
  v.t1[1] = v.rows[1] > 0 ? v.n_kv : 0;
  if (WIN) {
    const int end_a = min(v.Lkv, v.q0 + 128);
    v.t1[0] = end_a > v.kv0 ? (end_a - v.kv0 + BN - 1) / BN : 0;
    int lo_b;  // first key any row of tile B may see, rounded down to its tile
    if (p.window_blocks < 0) {  // sliding window of -window_blocks tokens
      const int lo = v.q0 + 128 + p.window_blocks + 1;
      lo_b = lo > 0 ? lo / BN * BN : 0;
    } else {
      const int blk = (v.q0 + 128) / 64 - (p.window_blocks - 1);
      lo_b = blk > 0 ? blk * 64 : 0;
    }
    v.t0[1] = (lo_b - v.kv0) / BN;
  }
  return v;
}
template <bool WIN, bool FLAG = false>
__device__ __forceinline__ Pair64Item decode_pair64(const FwdParams& p, int idx) {
  const int4 it = __ldg(p.items + idx);
  return decode_pair64_from<WIN, FLAG>(p, it, load_seq_offs(p, it.x));
}

// ------------------------------------------------------------------ producer

// Two producer threads: one stages Q and K, the other V, so that a K load
// never waits behind a V slot.
// The Q/K producer thread is also the CTA's claimer: it claims each item,
// decodes it (flagging a bad plan) and publishes it for the other roles
// before staging its Q tiles and K tiles; the V producer reads the items from
// the ring.
template <int D, bool WIN, bool LOAD_V>
__device__ void pair64_producer(const FwdParams& p, uint8_t* sm, Pair64Bars<D, WIN>& B) {
  using C = Pair64Cfg<D, WIN>;
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
    Pair64Item t;
    if (!LOAD_V) {
      const int idx = claim_next(p, L);
      if (idx >= 0) t = decode_pair64<WIN, true>(p, idx);
      ok = ring_publish(p, B.ring, k, t, idx >= 0, abort);
      if (!ok || idx < 0) break;
    } else if (!ring_read(p, B.ring, k, t, 0u, abort, ok)) {
      break;
    }
    if (t.n_kv == 0) continue;
    for (int j = 0; j < t.n_kv && ok; ++j, ++g) {
      const int y = t.kv_tok + t.kv0 + C::BN * j;
      // Each tile's Q goes up just before the first K tile it attends to:
      // with windows tile B's keys start two tiles later, and its Q stage is
      // freed late (its window ends last), so tile A's first K tiles of the
      // next item do not wait behind it.
      for (int x = 0; x < 2 && ok && !LOAD_V; ++x) {
        if (t.rows[x] == 0 || j != min(t.t0[x], t.n_kv - 1)) continue;
        const int s = qn[x] % C::NQS;
        const uint32_t ph = (qn[x] / C::NQS) & 1;
        ok = ptx::mbar_wait(&B.q_empty[x][s], ph ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&B.q_full[x][s], C::Q_TILE);
        q_armed[x][s] = (int)ph;
        uint8_t* sq = sm + (x ? C::OFF_QB : C::OFF_QA) + s * C::Q_TILE;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          ptx::tma_load_2d(sq + c * C::Q_CHUNK, &p.tm_q, &B.q_full[x][s], t.h * D + 64 * c, t.q_tok + 128 * x);
        ++qn[x];
      }
      if (!ok) break;
      if (!LOAD_V) {
        const int sk = g % C::NK;
        const uint32_t phk = (g / C::NK) & 1;
        ok = ptx::mbar_wait(&B.k_empty[sk], phk ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&B.k_full[sk], C::KV_TILE);
        uint8_t* dk = sm + C::OFF_K + sk * C::KV_TILE;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          ptx::tma_load_2d(dk + c * C::KV_CHUNK, &p.tm_k, &B.k_full[sk], t.h * D + 64 * c, y);
        k_armed[sk] = (int)phk;
      } else {
        const int sv = g % C::NV;
        const uint32_t phv = (g / C::NV) & 1;
        ok = ptx::mbar_wait(&B.v_empty[sv], phv ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&B.v_full[sv], C::KV_TILE);
        uint8_t* dv = sm + C::OFF_V + sv * C::KV_TILE;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          ptx::tma_load_2d(dv + c * C::KV_CHUNK, &p.tm_v, &B.v_full[sv], t.h * D + 64 * c, y);
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

struct Pair64PV {
  uint32_t gx;  // this side's tile counter (selects the S buffer)
  uint32_t g;   // K/V tile counter (selects the V stage)
  int item;     // this side's item counter (O buffer use count)
  int first, n16;
};

// SPLIT (the ALU activations): P is carried as two bf16 parts, P_hi in the
// buffer's first 32 columns and P_lo = bf16(P - P_hi) in the next 32, and
// O += P_hi V + P_lo V, so the weights keep ~16 significant bits: with a few
// keys and no softmax normalisation, a single bf16 rounding of P would move
// the output by up to 2^-8 of each term.
template <int D, bool WIN, bool SPLIT>
__device__ __forceinline__ bool pair64_issue_pv(const FwdParams& p, uint8_t* sm, Pair64Bars<D, WIN>& B, uint32_t tmem, int x,
                                              const Pair64PV& P) {
  using C = Pair64Cfg<D, WIN>;
  volatile int* abort = &B.abort;
  const int b = P.gx & 1;
  if (!ptx::mbar_wait(&B.p_full[x][b], (P.gx >> 1) & 1, p.timeout_ns, abort)) return false;
  if (P.first && !ptx::mbar_wait(&B.o_empty[x], (P.item & 1) ^ 1, p.timeout_ns, abort)) return false;
  const int sv = P.g % C::NV;
  if (!ptx::mbar_wait(&B.v_full[sv], (P.g / C::NV) & 1, p.timeout_ns, abort)) return false;
  ptx::tc_fence_after();
  const uint32_t v_base = ptx::smem_u32(sm + C::OFF_V + sv * C::KV_TILE);
  constexpr uint32_t idesc = ptx::idesc_bf16(128, D, 1);
  for (int kk = 0; kk < P.n16; ++kk) {
    // B = V tile, MN-major: 16 keys = two 8-row groups (SBO = 1024 B apart);
    // the two 64-column halves of D sit one chunk apart (LBO).
    const uint64_t bdesc = ptx::sdesc_sw128(v_base + kk * 2048, C::KV_CHUNK, 1024);
    ptx::mma_ts_elect(tmem + C::tm_o(x), tmem + C::tm_s(x, b) + 8 * kk, bdesc, idesc, (P.first && kk == 0) ? 0u : 1u);
  }
  if (SPLIT) {
    for (int kk = 0; kk < P.n16; ++kk) {
      const uint64_t bdesc = ptx::sdesc_sw128(v_base + kk * 2048, C::KV_CHUNK, 1024);
      ptx::mma_ts_elect(tmem + C::tm_o(x), tmem + C::tm_s(x, b) + 32 + 8 * kk, bdesc, idesc, 1u);
    }
  }
  ptx::mma_commit_elect(&B.o_done[x]);
  return true;
}

// One MMA warp per side, so that a side whose P is ready never waits behind
// the other side's (measured: cross_gelu 0.631 -> 0.600 ms, cross_silu
// 0.646 -> 0.604 ms against one issuer for both sides; block windows
// 1.16 -> 1.13 ms once they had five K/V stages -- with three, one issuer
// measured faster for them).
// Side x's warp walks every item; for each K/V tile it waits for K, issues
// S_x into its next buffer (if its rows attend to the tile), releases its
// hold on K, then issues the pending O_x += P_x V of its previous tile and
// releases its hold on that V.  A tile the side does not attend to is
// released once it has landed.  K and V stages then have two-count empty
// barriers (one arrival per side).
template <int D, bool WIN, bool SPLIT>
__device__ void pair64_mma_side(const FwdParams& p, uint8_t* sm, Pair64Bars<D, WIN>& B, uint32_t tmem, int x) {
  using C = Pair64Cfg<D, WIN>;
  volatile int* abort = &B.abort;
  int qn = 0;        // this side's items (Q stage and O use counts)
  uint32_t gx = 0;   // this side's tiles (S buffers)
  uint32_t g = 0;    // K/V tiles
  bool ok = true;
  bool pend = false;
  Pair64PV pv = {0, 0, 0, 0, 0};
  for (uint32_t k = 0; ok; ++k) {
    Pair64Item t;
    if (!ring_read(p, B.ring, k, t, 0xffffffffu, abort, ok)) break;
    if (t.n_kv == 0) continue;
    const bool has = t.rows[x] > 0;
    const int qs = qn % C::NQS;
    const uint32_t q_base = ptx::smem_u32(sm + (x ? C::OFF_QB : C::OFF_QA) + qs * C::Q_TILE);
    // the side's last tile reading Q (then its stage is released)
    const int q_last = t.t1[x] > t.t0[x] ? min(t.t1[x], t.n_kv) - 1 : t.n_kv - 1;
    bool q_ready = false;
    for (int j = 0; j < t.n_kv; ++j, ++g) {
      const int sk = g % C::NK;
      ok = ptx::mbar_wait(&B.k_full[sk], (g / C::NK) & 1, p.timeout_ns, abort);
      if (!ok) break;
      ptx::tc_fence_after();
      const bool act = has && j >= t.t0[x] && j < t.t1[x];
      if (has && !q_ready && (act || j == q_last)) {
        // The item's Q.  With windows (one Q stage per side), if it has not
        // landed yet the previous tile's P V goes first rather than wait
        // behind the load; short key ranges keep S before P V.
        if (WIN && pend && !ptx::mbar_test_wait(&B.q_full[x][qs], (qn / C::NQS) & 1)) {
          ok = pair64_issue_pv<D, WIN, SPLIT>(p, sm, B, tmem, x, pv);
          if (!ok) break;
          ptx::mma_commit_elect(&B.v_empty[pv.g % C::NV]);
          pend = false;
        }
        ok = ptx::mbar_wait(&B.q_full[x][qs], (qn / C::NQS) & 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::tc_fence_after();
        q_ready = true;
      }
      const int ncols = min(C::BN, t.kv_end - t.kv0 - C::BN * j);
      const int n16 = (ncols + 15) >> 4;
      if (act) {
        const uint32_t idesc = ptx::idesc_bf16(128, n16 * 16, 0);
        const uint32_t k_base = ptx::smem_u32(sm + C::OFF_K + sk * C::KV_TILE);
        const uint32_t s_col = C::tm_s(x, gx & 1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qoff = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
          ptx::mma_ss_elect(tmem + s_col, ptx::sdesc_sw128(q_base + qoff, 16, 1024),
                            ptx::sdesc_sw128(k_base + koff, 16, 1024), idesc, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit_elect(&B.s_full[x][gx & 1]);
      }
      ptx::mma_commit_elect(&B.k_empty[sk]);
      if (has && j == q_last) ptx::mma_commit_elect(&B.q_empty[x][qs]);
      if (pend) {
        ok = pair64_issue_pv<D, WIN, SPLIT>(p, sm, B, tmem, x, pv);
        if (!ok) break;
        ptx::mma_commit_elect(&B.v_empty[pv.g % C::NV]);
        pend = false;
      }
      if (act) {
        pv = Pair64PV{gx, g, qn, j == t.t0[x] ? 1 : 0, n16};
        pend = true;
        ++gx;
      } else {  // V(g) is not read by this side: release it once it has landed
        ok = ptx::mbar_wait(&B.v_full[g % C::NV], (g / C::NV) & 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mma_commit_elect(&B.v_empty[g % C::NV]);
      }
    }
    if (has) ++qn;
  }
  if (ok && pend) {
    ok = pair64_issue_pv<D, WIN, SPLIT>(p, sm, B, tmem, x, pv);
    if (ok) ptx::mma_commit_elect(&B.v_empty[pv.g % C::NV]);
  }
  if (!ok) report_failure(p, abort, kStatusMma);
  ptx::mma_commit_elect(&B.mma_drain[x]);
  const int never = 0;
  ptx::mbar_wait(&B.mma_drain[x], 0, 100000000ull, &never);
}

// ------------------------------------------------------------------ activation + epilogue

// One query row's output: O (fp32, TMEM columns [o_addr, o_addr + D)) times
// inv, rounded to bf16 and stored to dst when `store`, 32 columns at a time.
// (Keeping the next 16 columns' load in flight during each conversion
// measured no faster: the stores, not the TMEM loads, set the epilogue's pace.)
template <int D>
__device__ __forceinline__ void store_o_row(uint32_t o_addr, float inv, __nv_bfloat16* dst, bool store, bool v8) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t r[32];
    ptx::tmem_ld32(o_addr + 32 * c, r);
    ptx::tmem_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = ptx::pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
    if (store) store_row32(dst + 32 * c, pk, v8);
  }
}

// The side's 128 activation threads meet on their barrier (bounded wait, so
// a warp that has stopped on a timeout cannot hold the others forever).
__device__ __forceinline__ bool side_sync(const FwdParams& p, uint64_t* bar, uint32_t& phase, volatile int* abort) {
  ptx::mbar_arrive(bar);
  bool ok = ptx::mbar_wait(bar, phase & 1, p.timeout_ns, abort);
  ++phase;
  return __all_sync(0xffffffffu, ok);
}

// A whole 128-row tile's output by bulk tensor stores: per 64 columns, each
// thread converts its row (O times inv, bf16) into the side's staging area
// (16-byte chunk j of row r at chunk position j ^ (r mod 8): the 128-byte
// swizzle of the output map's box), the side's 128 threads meet, and the
// leader (row 0) issues the store.  Before it is rewritten the area must
// have been read by the previous store: the leader waits for that, then the
// meeting lets the others write.  False on a timeout.
template <int D>
__device__ __forceinline__ bool store_o_tile_bulk(const FwdParams& p, uint32_t o_addr, float inv, uint8_t* stg, int row,
                                                  uint64_t* bar, uint32_t& phase, volatile int* abort, int x0, int y0) {
  const bool leader = row == 0;
  const uint32_t base = ptx::smem_u32(stg) + static_cast<uint32_t>(row) * 128u;
#pragma unroll
  for (int c2 = 0; c2 < D / 64; ++c2) {
    if (leader) ptx::bulk_wait_read_all();
    if (!side_sync(p, bar, phase, abort)) return false;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t r[32];
      ptx::tmem_ld32(o_addr + 64 * c2 + 32 * cc, r);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 16-byte chunk j = 4 cc + q: eight bf16 = four words
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w[i] = ptx::pack_bf16x2(__uint_as_float(r[8 * q + 2 * i]) * inv, __uint_as_float(r[8 * q + 2 * i + 1]) * inv);
        const uint32_t j = static_cast<uint32_t>(4 * cc + q) ^ static_cast<uint32_t>(row & 7);
        ptx::st_shared_v4(base + 16u * j, w[0], w[1], w[2], w[3]);
      }
    }
    ptx::fence_proxy_async_smem();
    if (!side_sync(p, bar, phase, abort)) return false;
    if (leader) {
      ptx::tma_store_2d(&p.tm_o, stg, x0 + 64 * c2, y0);
      ptx::bulk_commit();
    }
  }
  return true;
}

template <int D, int ACT, bool WIN>
__device__ void pair64_activation(const FwdParams& p, uint8_t* sm, Pair64Bars<D, WIN>& B, uint32_t tmem, int x,
                                  int warp, int lane) {
  using C = Pair64Cfg<D, WIN>;
  volatile int* abort = &B.abort;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t o_addr = tmem + lane_off + C::tm_o(x);
  const float sl = p.score_scale;
  const ActK ak = act_k(p.act_a, p.act_c, p.act_sfu);  // GELU / SiLU: the scale folded into the cubic
  const int H = p.H;
  uint8_t* stg = sm + C::OFF_STG + x * C::STG_BYTES;  // this side's output staging area
  uint32_t epi_phase = 0;                               // uses of this side's epi_bar
  uint32_t gx = 0;
  bool ok = true;
  // The epilogue of an item waits for its last P V.  With full attention it
  // is deferred until the next item's first P is stored, so that wait
  // overlaps that activation (short key ranges: an item is one or two
  // tiles).  Window items hold several tiles per side, and there holding
  // back the next item's first P V stalls the MMA issuer: no deferral.
  bool pend = false, pend_live = false, pend_row_ok = false, pend_bulk = false;
  float pend_inv = 0.0f;
  int pend_x0 = 0, pend_y0 = 0;
  __nv_bfloat16* pend_orow = nullptr;
  auto epilogue = [&]() {
    ptx::tc_fence_after();
    if (pend_bulk) {  // a whole tile: staged and stored in bulk
      if (!store_o_tile_bulk<D>(p, o_addr, pend_inv, stg, row, &B.epi_bar[x], epi_phase, abort, pend_x0, pend_y0))
        ok = false;
    } else if (pend_live) {
      store_o_row<D>(o_addr, pend_inv, pend_orow, pend_row_ok, p.out_align32 != 0);
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(&B.o_empty[x]);
    pend = false;
  };
  // Items come decoded through the CTA's ring (no global loads here).
  for (uint32_t k = 0; ok; ++k) {
    Pair64Item t;
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
    if (WIN) {  // first key of this row's window
      if (p.window_blocks < 0) {
        win_lo = max(0, i_seq + p.window_blocks + 1);
      } else {
        const int blk = i_seq / 64 - (p.window_blocks - 1);
        win_lo = blk > 0 ? blk * 64 : 0;
      }
    }
    const int j0 = x ? t.t0[1] : t.t0[0], j1 = x ? t.t1[1] : t.t1[0];  // this side's K/V tiles
    const int kv0 = t.kv0, kv_end = t.kv_end;
    const float inv_lkv = sl / static_cast<float>(max(t.Lkv, 1));  // the GELU's folded scale, then 1/Lkv
    for (int j = j0; j < j1; ++j, ++gx) {
      const int sb = gx & 1;
      ok = ptx::mbar_wait(&B.s_full[x][sb], (gx >> 1) & 1, p.timeout_ns, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t s_addr = tmem + lane_off + C::tm_s(x, sb);
      float alpha = 1.0f;
      bool rescale = false;
      if (rows_live) {
        // valid key columns of this row: [c_lo, c_hi] (tile-relative)
        const int kv_t0 = kv0 + C::BN * j;
        const int ncols = min(C::BN, kv_end - kv_t0);  // the tile's key extent
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
          for (int ch = 0; ch < 2; ++ch) {
            const int lo = 32 * ch, hi = 32 * ch + 31;
            if (__all_sync(0xffffffffu, lo >= c_lo && hi <= c_hi)) fullm |= 1u << ch;
            if (__any_sync(0xffffffffu, ch < nch && hi >= c_lo && lo <= c_hi)) livem |= 1u << ch;
          }
        } else {
          livem = (1u << nch) - 1u;
          fullm = (1u << (ncols >> 5)) - 1u;
        }
        // The tile's 64 scores of this row in registers, one TMEM round trip.
        uint32_t sr[64];
        // A whole tile of valid keys (full attention, softmax, scale > 0):
        // the second half of the row loads while the first half's maximum is
        // taken.  (Window tiles keep one load: the split measured slower there.)
        const bool split_ld = !WIN && ACT == kActSoftmax && fullm == 0x3u && sl > 0.0f;
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (split_ld) {
          ptx::tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
          ptx::tmem_wait_ld_r32(&sr[0]);
          ptx::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            m4[0] = ptx::max3(m4[0], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            m4[1] = ptx::max3(m4[1], __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
            m4[2] = ptx::max3(m4[2], __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
            m4[3] = ptx::max3(m4[3], __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
          }
          ptx::tmem_wait_ld_r32(&sr[32]);
#pragma unroll
          for (int c = 32; c < 64; c += 8) {
            m4[0] = ptx::max3(m4[0], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            m4[1] = ptx::max3(m4[1], __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
            m4[2] = ptx::max3(m4[2], __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
            m4[3] = ptx::max3(m4[3], __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < 2; ++ch)
            if ((livem >> ch) & 1u) ptx::tmem_ld32(s_addr + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * ch]));
          ptx::tmem_wait_ld();
        }
        if (ACT == kActSoftmax) {
          // Scores in log2 units: x = s * scale * log2(e); masked columns
          // become -inf.  With scale > 0 the scaling is folded into the
          // exponent's FMA; otherwise it is applied first.
          const bool fold = sl > 0.0f;
#pragma unroll
          for (int ch = 0; ch < 2 && !split_ld; ++ch) {
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
          uint64_t acc[4] = {0, 0, 0, 0};  // +0.0f pairs
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
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
              float e0, e1;
              ptx::f2_unpack(x2, e0, e1);
              e0 = ptx::ex2_approx(e0);
              e1 = ptx::ex2_approx(e1);
              acc[u & 3] = ptx::f2_add(acc[u & 3], ptx::f2_pack(e0, e1));
              sr[16 * ch + u] = ptx::pack_bf16x2(e0, e1);  // P overwrites scores already consumed
            }
          }
          const uint64_t acc01 = ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3]));
          float sa, sb2;
          ptx::f2_unpack(acc01, sa, sb2);
          l_run += sa + sb2;
        } else {  // GELU / SiLU: P = P_hi + P_lo, two bf16 parts (see pair64_issue_pv)
          uint32_t plo[32];
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            if (ch >= nch) continue;
            if (!((livem >> ch) & 1u)) {
#pragma unroll
              for (int u = 0; u < 16; ++u) sr[16 * ch + u] = plo[16 * ch + u] = 0u;
              continue;
            }
            const bool full = (fullm >> ch) & 1u;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const int c = 32 * ch + 2 * u;
              float e0, e1;
              act_eval2(ak, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), e0, e1);
              if (!full) {
                e0 = (c >= c_lo && c <= c_hi) ? e0 : 0.0f;
                e1 = (c + 1 >= c_lo && c + 1 <= c_hi) ? e1 : 0.0f;
              }
              const uint32_t hi = ptx::pack_bf16x2(e0, e1);
              const uint64_t rem = ptx::f2_sub(ptx::f2_pack(e0, e1),
                                               ptx::f2_pack(__uint_as_float(hi << 16), __uint_as_float(hi & 0xFFFF0000u)));
              float r0, r1;
              ptx::f2_unpack(rem, r0, r1);
              sr[16 * ch + u] = hi;
              plo[16 * ch + u] = ptx::pack_bf16x2(r0, r1);
            }
          }
          ptx::tmem_st32(s_addr + 32, plo);  // P_lo over the buffer's last 32 columns
        }
        // P (bf16 pairs, 32 columns) over the first columns of this S
        // buffer; P V reads no column beyond 8 * n16 (and, for P_lo, 32 + 8 * n16).
        ptx::tmem_st32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        ptx::tmem_wait_st();
      }
      // O_x += P_x(t-1) V has landed once this wait returns (it was issued
      // after S_x(t), so the S barrier does not imply it); the wait also
      // keeps this side's view of the barrier phase exact.
      if (gx >= 1) {
        ok = ptx::mbar_wait(&B.o_done[x], (gx - 1) & 1, p.timeout_ns, abort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      if constexpr (!WIN) {
        if (pend) epilogue();  // the previous item's last P V has landed
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
      ptx::mbar_arrive(&B.p_full[x][sb]);
    }
    if (!ok) break;
    if (ACT == kActSoftmax && p.lse && row < rows)
      p.lse[static_cast<size_t>(t.q_tok + 128 * x + row) * H + t.h] = row_lse(m_run, l_run);
    const float inv = (ACT == kActSoftmax) ? (l_run > 0.0f ? 1.0f / l_run : 0.0f) : inv_lkv;
    if constexpr (WIN) {  // no deferral: the epilogue now
      ok = ptx::mbar_wait(&B.o_done[x], (gx - 1) & 1, p.timeout_ns, abort);  // the item's last P V
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      if (C::BULK && p.out_tma && rows == 128) {
        ok = store_o_tile_bulk<D>(p, o_addr, inv, stg, row, &B.epi_bar[x], epi_phase, abort, t.h * D,
                                  t.q_tok + 128 * x);
        if (!ok) break;
      } else if (rows_live) {
        store_o_row<D>(o_addr, inv, orow, row < rows, p.out_align32 != 0);
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&B.o_empty[x]);
    } else {
      pend = true;
      pend_live = rows_live;
      pend_row_ok = row < rows;
      pend_bulk = C::BULK && p.out_tma && rows == 128;
      pend_x0 = t.h * D;
      pend_y0 = t.q_tok + 128 * x;
      pend_inv = inv;
      pend_orow = orow;
    }
  }
  if constexpr (!WIN) {
    if (ok && pend) {  // the last item's epilogue
      ok = ptx::mbar_wait(&B.o_done[x], (gx - 1) & 1, p.timeout_ns, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) epilogue();
    }
  }
  if (row == 0) ptx::bulk_wait_all();  // the side's last bulk stores
  if (!ok && lane == 0) report_failure(p, abort, kStatusActivation);
}

// ------------------------------------------------------------------ kernel

template <int D, int ACT, bool WIN>
__global__ void __launch_bounds__(384, 1) gdpa_fwd_pair64_kernel(const __grid_constant__ FwdParams p) {
  using C = Pair64Cfg<D, WIN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* sm = smem_raw + pad;
  Pair64Bars<D, WIN>& B = *reinterpret_cast<Pair64Bars<D, WIN>*>(sm + C::OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      for (int s = 0; s < C::NQS; ++s) {
        ptx::mbar_init(&B.q_full[x][s], 1);
        ptx::mbar_init(&B.q_empty[x][s], 1);
      }
      for (int b = 0; b < 2; ++b) {
        ptx::mbar_init(&B.s_full[x][b], 1);
        ptx::mbar_init(&B.p_full[x][b], 128);
      }
      ptx::mbar_init(&B.o_done[x], 1);
      ptx::mbar_init(&B.o_empty[x], 128);
    }
    constexpr uint32_t n_mma = 2;  // MMA warps, each releasing every K and V stage once
    for (int s = 0; s < C::NK; ++s) {
      ptx::mbar_init(&B.k_full[s], 1);
      ptx::mbar_init(&B.k_empty[s], n_mma);
    }
    for (int s = 0; s < C::NV; ++s) {
      ptx::mbar_init(&B.v_full[s], 1);
      ptx::mbar_init(&B.v_empty[s], n_mma);
    }
    ptx::mbar_init(&B.mma_drain[0], 1);
    ptx::mbar_init(&B.mma_drain[1], 1);
    ptx::mbar_init(&B.epi_bar[0], 128);
    ptx::mbar_init(&B.epi_bar[1], 128);
    for (int r = 0; r < kRing; ++r) {  // readers: the V producer, the MMA warps, the eight activation warps
      ptx::mbar_init(&B.ring.full[r], 1);
      ptx::mbar_init(&B.ring.empty[r], 1 + n_mma + 8);
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
    ptx::regs_dec<C::regs_ctrl(ACT)>();
    if (warp == 0) {
      if (lane == 0) pair64_producer<D, WIN, false>(p, sm, B);
    } else if (warp == 2) {
      if (lane == 0) pair64_producer<D, WIN, true>(p, sm, B);
    } else {  // warps 1 and 3: the MMA issuers of tiles A and B
      pair64_mma_side<D, WIN, ACT == kActGelu>(p, sm, B, tmem, warp == 1 ? 0 : 1);
    }
  } else {  // warpgroups 1 and 2: tiles A and B
    ptx::regs_inc<C::regs_act(ACT)>();
    pair64_activation<D, ACT, WIN>(p, sm, B, tmem, warp < 8 ? 0 : 1, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::TM_COLS);
  if (threadIdx.x == 0) claim_finish(p);
}

}  // namespace gdpa
