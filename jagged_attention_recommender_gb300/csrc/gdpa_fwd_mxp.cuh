// gdpa_fwd_mxp.cuh -- jagged GDPA forward with Q, K and V in MXFP8 and the
// weights P rounded to MXFP8 on chip, so that both products run on the
// block-scaled e4m3 tensor-core MMA (kind::mxf8f6f4, one E8M0 scale per 32
// elements of the contraction).  MXFP8 attention: techfeed summary of "GEM
// Training", section on MXFP8 ultra-low-precision training; aigeeknews
// translation, compute-efficiency section.  Full attention, softmax, D = 128.
//
// A work item is 256 query rows of one (sequence, head) -- tile A = rows
// [q0, q0+128), tile B = [q0+128, q0+256), B may be empty -- against the
// sequence's keys, in 64-key score tiles; K and V are staged 128 keys at a
// time (two score tiles) and each staged block feeds both query tiles.
//
//   S_x = Q_x K^T      A = Q_x (e4m3, smem), B = K rows (e4m3, smem),
//                      scales: Q's per (row, 32 coordinates), K's per (key,
//                      32 coordinates)
//   P_x = exp2(S_x log2(e) scale - m) in e4m3 with one E8M0 scale per
//         (row, 32 keys), written by the activation into tensor memory
//   O_x += P_x V       A = P_x (tensor memory), B = V^T rows (e4m3, smem,
//                      key-major), scales: P's, and V's per (coordinate,
//                      32 keys)
//
// Tensor memory (512 columns): each side x has 128 columns at 128 x: S_x in
// the first 64 (the fp32 scores of a tile; once read, the P scale words in
// columns 0-3, the P codes in 8-23 and the V scale words in 32-35), Q_x's
// scale words at +64 and the K scale words of side x's next tile at +96;
// O_A at 256, O_B at 384.  Every scale area starts on a 32-column boundary,
// which is what limits the score tile to 64 keys: two 128-column score
// buffers and two 128-column outputs would leave no column for the scales.
// With one score buffer per side, side x's MMA warp issues O_x += P_x(t-1)
// V(t-1) and then S_x(t) (the tensor core runs them in order, so S_x(t)
// cannot overwrite P_x(t-1) before it is read); a side's activation waits
// for its next scores while the other side's runs.  P is released in two
// halves of 32 keys, so the first half's P V runs while the second half's
// weights are computed.
//
// Scale words in tensor memory (one 32-bit word = four E8M0 codes, byte i
// for the i-th 32-element block of the MMA's K, selected per instruction):
// an A operand's row m reads lane m, column m / 32 of its area; a B
// operand's row n reads column n / 32 at lane n % 32 of the lane quarter of
// the accumulator row, so B's words are written into all four quarters.
//
// Threads (384): warpgroup 0 holds the TMA producer for Q and K (warp 0),
// the MMA issuers of tiles A (warp 1, also TMEM owner) and B (warp 3) and
// the TMA producer for V (warp 2); warpgroups 1 and 2 are the activation /
// epilogue of tiles A and B.  Each side is a pipeline of its own: its
// activation warpgroup stages its Q scale words and the K scale words of
// its next tile, and a staged K or V block is released when both MMA warps
// are done with it (a side without rows in an item releases the item's
// blocks as they land).
#pragma once

#include "gdpa_fwd_common.cuh"
#include "gdpa_fwd_pair64.cuh"

namespace gdpa {

struct MxpCfg {
  static constexpr int D = 128;
  static constexpr int BN = 64;                   // keys per score tile
  static constexpr int KB = 128;                  // keys per staged K / V block (two tiles)
  static constexpr int Q_TILE = 128 * 128;        // e4m3 Q: 128 rows x 128 bytes
  static constexpr int K_STAGE = KB * 128;        // e4m3 K: 128 keys x 128 bytes
  static constexpr int V_STAGE = 128 * KB;        // e4m3 V^T: 128 coordinates x 128 keys
  static constexpr int NQS = 2, NK = 3, NV = 3;
  static constexpr int OFF_QA = 0;
  static constexpr int OFF_QB = OFF_QA + NQS * Q_TILE;
  static constexpr int OFF_K = OFF_QB + NQS * Q_TILE;
  static constexpr int OFF_V = OFF_K + NK * K_STAGE;
  static constexpr int OFF_BAR = OFF_V + NV * V_STAGE;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;
  __host__ __device__ static constexpr uint32_t tm_s(int x) { return 128u * x; }
  __host__ __device__ static constexpr uint32_t tm_sfq(int x) { return 128u * x + 64u; }
  __host__ __device__ static constexpr uint32_t tm_sfk(int x) { return 128u * x + 96u; }
  __host__ __device__ static constexpr uint32_t tm_o(int x) { return x ? 384u : 256u; }
  static constexpr uint32_t P_SF = 0, P_CODES = 8, V_SF = 32;  // inside S_x, after the scores are read
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int THREADS = 384;
  static constexpr int REGS_CTRL = 88;
  static constexpr int REGS_ACT = 208;
  static constexpr int MIN_LAUNCH_REGS = 168;
  static_assert(REGS_CTRL + 2 * REGS_ACT <= 3 * MIN_LAUNCH_REGS, "register split");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct MxpBars {
  uint64_t q_full[2][MxpCfg::NQS], q_empty[2][MxpCfg::NQS];
  uint64_t k_full[MxpCfg::NK], k_empty[MxpCfg::NK];
  uint64_t v_full[MxpCfg::NV], v_empty[MxpCfg::NV];
  uint64_t s_full[2], p_full[2][2];  // per side; P per 32-key half
  uint64_t o_done[2], o_empty[2];
  uint64_t sf_init[2];  // side x's first Q and K scale words are in TMEM
  uint64_t mma_drain[2];
  uint32_t tmem_slot;
  int abort;
};

// ------------------------------------------------------------------ producer

template <bool LOAD_V>
__device__ void mxp_producer(const FwdParams& p, uint8_t* sm, MxpBars& B, int ibeg, int iend) {
  using C = MxpCfg;
  volatile int* abort = &B.abort;
  int qn[2] = {0, 0};
  uint32_t gb = 0;  // staged 128-key blocks
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
  for (int idx = ibeg; idx < iend && ok; ++idx) {
    const Pair64Item t = decode_pair64<false, !LOAD_V>(p, idx);
    if (t.n_kv == 0) continue;
    if (!LOAD_V) {
      for (int x = 0; x < 2 && ok; ++x) {
        if (t.rows[x] == 0) continue;
        const int s = qn[x] % C::NQS;
        const uint32_t ph = (qn[x] / C::NQS) & 1;
        ok = ptx::mbar_wait(&B.q_empty[x][s], ph ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&B.q_full[x][s], C::Q_TILE);
        q_armed[x][s] = (int)ph;
        ptx::tma_load_2d(sm + (x ? C::OFF_QB : C::OFF_QA) + s * C::Q_TILE, &p.tm_q, &B.q_full[x][s], t.h * C::D,
                         t.q_tok + 128 * x);
        ++qn[x];
      }
    }
    const int nkb = (t.n_kv + 1) >> 1;
    const int vcol = LOAD_V ? __ldg(p.vt_col + __ldg(p.items + idx).x) : 0;
    for (int u = 0; u < nkb && ok; ++u, ++gb) {
      const int s = gb % (LOAD_V ? C::NV : C::NK);
      const uint32_t ph = (gb / (LOAD_V ? C::NV : C::NK)) & 1;
      if (!LOAD_V) {
        ok = ptx::mbar_wait(&B.k_empty[s], ph ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&B.k_full[s], C::K_STAGE);
        ptx::tma_load_2d(sm + C::OFF_K + s * C::K_STAGE, &p.tm_k, &B.k_full[s], t.h * C::D, t.kv_tok + C::KB * u);
        k_armed[s] = (int)ph;
      } else {
        // V^T rows h*D .. h*D+127, the block's 128 key columns (a multiple of
        // 32 bytes from the row start: the TMA x coordinate stays aligned)
        ok = ptx::mbar_wait(&B.v_empty[s], ph ^ 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&B.v_full[s], C::V_STAGE);
        ptx::tma_load_2d(sm + C::OFF_V + s * C::V_STAGE, &p.tm_v, &B.v_full[s], vcol + C::KB * u, t.h * C::D);
        v_armed[s] = (int)ph;
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

struct MxpPV {
  uint32_t gx;   // this side's tile counter (p_full phase)
  uint32_t gb;   // the V block the tile lies in (stage and phase)
  int half;      // which 64 keys of the block
  int item;      // this side's item counter (o_empty phase)
  int first;     // the item's first tile: O is overwritten
  int n32;       // 32-key blocks of the tile holding keys
  int last;      // the block's last tile: its V stage is released after this P V
};

// O_x += P_x V for one tile: the first 32 keys once the activation has
// released them, then the second 32.
__device__ __forceinline__ bool mxp_issue_pv(const FwdParams& p, uint8_t* sm, MxpBars& B, uint32_t tmem, int x,
                                             const MxpPV& P, uint32_t& v_seen) {
  using C = MxpCfg;
  volatile int* abort = &B.abort;
  const uint32_t ph = P.gx & 1;
  if (!ptx::mbar_wait(&B.p_full[x][0], ph, p.timeout_ns, abort)) return false;
  if (P.first && !ptx::mbar_wait(&B.o_empty[x], (P.item & 1) ^ 1, p.timeout_ns, abort)) return false;
  const int sv = P.gb % C::NV;
  if (v_seen != P.gb + 1) {  // the block's first tile: wait for its V
    if (!ptx::mbar_wait(&B.v_full[sv], (P.gb / C::NV) & 1, p.timeout_ns, abort)) return false;
    v_seen = P.gb + 1;
  }
  ptx::tc_fence_after();
  const uint32_t v_base = ptx::smem_u32(sm + C::OFF_V + sv * C::V_STAGE) + 64u * P.half;
  const uint32_t s = tmem + C::tm_s(x);
  // B = V^T, K-major: 32 keys = 32 bytes of each coordinate's 128-byte swizzle row
  ptx::mma_mx_ts_elect(tmem + C::tm_o(x), s + C::P_CODES, ptx::sdesc_sw128(v_base, 16, 1024),
                       ptx::idesc_mx_e4m3(128, 128, 0), s + C::P_SF, s + C::V_SF, P.first ? 0u : 1u);
  if (!ptx::mbar_wait(&B.p_full[x][1], ph, p.timeout_ns, abort)) return false;
  if (P.n32 > 1) {
    ptx::tc_fence_after();
    ptx::mma_mx_ts_elect(tmem + C::tm_o(x), s + C::P_CODES + 8, ptx::sdesc_sw128(v_base + 32, 16, 1024),
                         ptx::idesc_mx_e4m3(128, 128, 1), s + C::P_SF, s + C::V_SF, 1u);
  }
  ptx::mma_commit_elect(&B.o_done[x]);
  if (P.last) ptx::mma_commit_elect(&B.v_empty[sv]);
  return true;
}

// The MMA warp of side x.  It walks every item; for an item without rows on
// its side it only releases the item's K and V blocks (after they land, so
// that it never arrives twice in one phase of a stage's empty barrier).
__device__ void mxp_mma(const FwdParams& p, uint8_t* sm, MxpBars& B, uint32_t tmem, int ibeg, int iend, int x) {
  using C = MxpCfg;
  volatile int* abort = &B.abort;
  int qn = 0;           // items of this side (Q stage and O use counts)
  uint32_t gx = 0;      // tiles of this side
  uint32_t gb = 0;      // 128-key blocks
  uint32_t v_seen = 0;  // 1 + the V block whose load this warp has seen land
  bool ok = ptx::mbar_wait(&B.sf_init[x], 0, p.timeout_ns, abort);
  bool pend = false;
  MxpPV pv = {0, 0, 0, 0, 0, 0, 0};
  for (int idx = ibeg; idx < iend && ok; ++idx) {
    const Pair64Item t = decode_pair64<false>(p, idx);
    if (t.n_kv == 0) continue;
    const int nkb = (t.n_kv + 1) >> 1;
    if (t.rows[x] == 0) {  // nothing to compute here: release the item's blocks
      if (pend) {
        ok = mxp_issue_pv(p, sm, B, tmem, x, pv, v_seen);
        pend = false;
      }
      for (int u = 0; u < nkb && ok; ++u) {
        const uint32_t kb = gb + u;
        ok = ptx::mbar_wait(&B.k_full[kb % C::NK], (kb / C::NK) & 1, p.timeout_ns, abort);
        if (ok) ok = ptx::mbar_wait(&B.v_full[kb % C::NV], (kb / C::NV) & 1, p.timeout_ns, abort);
        if (!ok) break;
        ptx::mma_commit_elect(&B.k_empty[kb % C::NK]);
        ptx::mma_commit_elect(&B.v_empty[kb % C::NV]);
      }
      gb += nkb;
      continue;
    }
    const int sq = qn % C::NQS;
    ok = ptx::mbar_wait(&B.q_full[x][sq], (qn / C::NQS) & 1, p.timeout_ns, abort);
    if (!ok) break;
    const uint32_t q_base = ptx::smem_u32(sm + (x ? C::OFF_QB : C::OFF_QA) + sq * C::Q_TILE);
    for (int j = 0; j < t.n_kv; ++j, ++gx) {
      const uint32_t kb = gb + (j >> 1);
      const int sk = kb % C::NK;
      // O_x += P_x(previous tile) V first: it reads P from S_x
      if (pend) {
        ok = mxp_issue_pv(p, sm, B, tmem, x, pv, v_seen);
        pend = false;
        if (!ok) break;
      }
      if ((j & 1) == 0) {
        ok = ptx::mbar_wait(&B.k_full[sk], (kb / C::NK) & 1, p.timeout_ns, abort);
        if (!ok) break;
      }
      ptx::tc_fence_after();
      const uint32_t k_base = ptx::smem_u32(sm + C::OFF_K + sk * C::K_STAGE) + (j & 1) * (C::BN * 128);
      // S_x = Q_x K^T: 32 coordinates (32 bytes of the 128-byte swizzle row)
      // per MMA, scale byte kk of each row's word
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        ptx::mma_mx_elect(tmem + C::tm_s(x), ptx::sdesc_sw128(q_base + 32 * kk, 16, 1024),
                          ptx::sdesc_sw128(k_base + 32 * kk, 16, 1024), ptx::idesc_mx_e4m3(128, C::BN, kk),
                          tmem + C::tm_sfq(x), tmem + C::tm_sfk(x), kk > 0 ? 1u : 0u);
      ptx::mma_commit_elect(&B.s_full[x]);
      const bool block_end = (j & 1) || j == t.n_kv - 1;
      if (block_end) ptx::mma_commit_elect(&B.k_empty[sk]);
      if (j == t.n_kv - 1) ptx::mma_commit_elect(&B.q_empty[x][sq]);
      const int ncols = min(C::BN, t.kv_end - C::BN * j);
      pv = MxpPV{gx, kb, j & 1, qn, j == 0 ? 1 : 0, (ncols + 31) >> 5, block_end ? 1 : 0};
      pend = true;
    }
    if (!ok) break;
    gb += nkb;
    ++qn;
  }
  if (ok && pend) ok = mxp_issue_pv(p, sm, B, tmem, x, pv, v_seen);
  if (!ok) report_failure(p, abort, kStatusMma);
  // Every MMA this warp issued is complete once this commit lands.
  ptx::mma_commit_elect(&B.mma_drain[x]);
  const int never = 0;
  ptx::mbar_wait(&B.mma_drain[x], 0, 100000000ull, &never);
}

// ------------------------------------------------------------------ activation + epilogue

// Side x's walk over its tiles, for staging the K scale words of the next
// one: this thread's words are those of keys 64 j + lane and 64 j + 32 +
// lane of the item's sequence (scale 1 past the end).
struct MxpKCursor {
  int idx, j, x;
  Pair64Item t;
  bool valid;
  __device__ __forceinline__ void seek(const FwdParams& p, int iend) {  // first item from idx on with rows on side x
    for (valid = false; idx < iend; ++idx) {
      t = decode_pair64<false>(p, idx);
      if (t.n_kv > 0 && t.rows[x] > 0) {
        valid = true;
        return;
      }
    }
  }
  __device__ __forceinline__ void advance(const FwdParams& p, int iend) {
    if (!valid) return;
    if (++j < t.n_kv) return;
    j = 0;
    ++idx;
    seek(p, iend);
  }
  __device__ __forceinline__ void load(const FwdParams& p, int lane, uint32_t (&w)[2]) const {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int key = 64 * j + 32 * c + lane;
      w[c] = (valid && key < t.Lkv) ? __ldg(p.k_sf + static_cast<size_t>(t.kv_tok + key) * p.H + t.h) : 0x7F7F7F7Fu;
    }
  }
};

// Next item from idx on with rows in tile x (iend if none).
__device__ __forceinline__ int mxp_next_item(const FwdParams& p, int idx, int iend, int x, Pair64Item& t) {
  for (; idx < iend; ++idx) {
    t = decode_pair64<false>(p, idx);
    if (t.n_kv > 0 && t.rows[x] > 0) return idx;
  }
  return iend;
}

// This thread's Q scale word for item t, tile x (scale 1 for rows past the end).
__device__ __forceinline__ uint32_t mxp_q_word(const FwdParams& p, const Pair64Item& t, int x, int row) {
  return row < t.rows[x] ? __ldg(p.q_sf + static_cast<size_t>(t.q_tok + 128 * x + row) * p.H + t.h) : 0x7F7F7F7Fu;
}

// P of one 32-key block: 2^(x - m_use - e) for the block's 32 scores (x =
// score * mul), rounded to e4m3 into eight words (key k at byte k % 4 of
// word k / 4); returns the sum of the unrounded values.
__device__ __forceinline__ float mxp_block(const uint32_t* sr, uint64_t mul2, float neg, uint32_t (&pw)[8]) {
  const uint64_t neg2 = ptx::f2_splat(neg);
  uint64_t acc[2] = {0, 0};
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint64_t x01 = ptx::f2_fma(ptx::f2_pack(__uint_as_float(sr[4 * u]), __uint_as_float(sr[4 * u + 1])), mul2, neg2);
    const uint64_t x23 =
        ptx::f2_fma(ptx::f2_pack(__uint_as_float(sr[4 * u + 2]), __uint_as_float(sr[4 * u + 3])), mul2, neg2);
    float e0, e1, e2, e3;
    ptx::f2_unpack(x01, e0, e1);
    ptx::f2_unpack(x23, e2, e3);
    e0 = ptx::ex2_approx(e0);
    e1 = ptx::ex2_approx(e1);
    e2 = ptx::ex2_approx(e2);
    e3 = ptx::ex2_approx(e3);
    acc[u & 1] = ptx::f2_add(acc[u & 1], ptx::f2_add(ptx::f2_pack(e0, e1), ptx::f2_pack(e2, e3)));
    pw[u] = ptx::pack_e4m3x4(e0, e1, e2, e3);
  }
  float s0, s1;
  ptx::f2_unpack(ptx::f2_add(acc[0], acc[1]), s0, s1);
  return s0 + s1;
}

__device__ void mxp_activation(const FwdParams& p, MxpBars& B, uint32_t tmem, int ibeg, int iend, int x, int warp,
                               int lane) {
  using C = MxpCfg;
  constexpr int D = C::D;
  volatile int* abort = &B.abort;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t o_addr = tmem + lane_off + C::tm_o(x);
  const uint32_t s_addr = tmem + lane_off + C::tm_s(x);
  const float sl = p.score_scale;
  const bool fold = sl > 0.0f;
  const int H = p.H;
  const size_t vsf_row = static_cast<size_t>(H) * D;  // bytes per 32-key block of the V scales
  bool ok = true;

  // Scale words before side x's first MMA: its first item's Q words and its
  // first tile's K words.
  Pair64Item qt;
  int q_next = mxp_next_item(p, ibeg, iend, x, qt);
  uint32_t qw = q_next < iend ? mxp_q_word(p, qt, x, row) : 0x7F7F7F7Fu;
  MxpKCursor cur;
  cur.idx = ibeg;
  cur.j = 0;
  cur.x = x;
  cur.seek(p, iend);
  uint32_t kw[2];
  cur.load(p, lane, kw);
  ptx::tmem_st2(tmem + lane_off + C::tm_sfk(x), kw[0], kw[1]);
  cur.advance(p, iend);
  cur.load(p, lane, kw);  // the second tile's words, staged during the first
  if (q_next < iend) ptx::tmem_st1(tmem + lane_off + C::tm_sfq(x) + quarter, qw);
  ptx::tmem_wait_st();
  ptx::tc_fence_before();
  ptx::mbar_arrive(&B.sf_init[x]);

  uint32_t gx = 0;
  bool pend = false, pend_row_ok = false;
  float pend_inv = 0.0f;
  __nv_bfloat16* pend_orow = nullptr;
  auto epilogue = [&]() {
    ptx::tc_fence_after();
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t r[32];
      ptx::tmem_ld32(o_addr + 32 * c, r);
      ptx::tmem_wait_ld();
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pk[i] = ptx::pack_bf16x2(__uint_as_float(r[2 * i]) * pend_inv, __uint_as_float(r[2 * i + 1]) * pend_inv);
      if (pend_row_ok) store_row32(pend_orow + 32 * c, pk, p.out_align32 != 0);
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(&B.o_empty[x]);
    pend = false;
  };
  for (int idx = ibeg; idx < iend && ok; ++idx) {
    const Pair64Item t = decode_pair64<false>(p, idx);
    const int rows = t.rows[x];
    __nv_bfloat16* orow = p.out + (static_cast<size_t>(t.q_tok + 128 * x + row) * H + t.h) * D;
    if (t.n_kv == 0) {  // no keys: zero output rows
      if (row < rows) {
        if (p.lse) p.lse[static_cast<size_t>(t.q_tok + 128 * x + row) * H + t.h] = -INFINITY;
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    if (rows == 0) continue;
    // the Q scale words of this side's next item, staged at this item's end
    q_next = mxp_next_item(p, idx + 1, iend, x, qt);
    qw = q_next < iend ? mxp_q_word(p, qt, x, row) : 0x7F7F7F7Fu;
    const int blk0 = __ldg(p.vt_col + __ldg(p.items + idx).x) >> 5;  // the sequence's first V scale block
    const uint8_t* vsf = p.vt_sf + static_cast<size_t>(max(blk0, 0)) * vsf_row + t.h * D + lane;
    // 32-key blocks of the sequence (none read past the scales' end)
    const int nblk = min((t.Lkv + 31) >> 5, p.vt_blocks - blk0);
    float m_run = -INFINITY, l_run = 0.0f;
    for (int j = 0; j < t.n_kv; ++j, ++gx) {
      // V scale codes of the tile's two key blocks for coordinates lane + 32 c
      uint32_t vw[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t b0 = 2 * j < nblk ? __ldg(vsf + (2 * j) * vsf_row + 32 * c) : 127u;
        const uint32_t b1 = 2 * j + 1 < nblk ? __ldg(vsf + (2 * j + 1) * vsf_row + 32 * c) : 127u;
        vw[c] = b0 | (b1 << 8) | 0x7F7F0000u;
      }
      ok = ptx::mbar_wait(&B.s_full[x], gx & 1, p.timeout_ns, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const int ncols = min(C::BN, t.kv_end - C::BN * j);
      uint32_t sr[64];
      ptx::tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      ptx::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      ptx::tmem_wait_ld_r64(sr);
      if (ncols < C::BN || !fold) {  // the ragged end of the sequence (or scale <= 0: scale first)
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float v = __uint_as_float(sr[c]);
          if (!fold) v *= sl;
          sr[c] = __float_as_uint(c < ncols ? v : -INFINITY);
        }
      }
      // block maxima of the two 32-key halves (raw scores when folding)
      float mh[2];
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
        for (int c = 32 * hb; c < 32 * hb + 32; c += 4) {
          a0 = ptx::max3(a0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
          a1 = ptx::max3(a1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
        }
        mh[hb] = fmaxf(a0, a1);
        if (fold) mh[hb] *= sl;
      }
      const float m_new = fmaxf(m_run, fmaxf(mh[0], mh[1]));
      float alpha = 1.0f;
      bool rescale = false;
      if (j == 0) {
        m_run = m_new;
      } else if (m_new > m_run + 8.0f) {  // lazy rescale: only when the max grew by more than 2^8
        alpha = ptx::ex2_approx(m_run - m_new);
        l_run *= alpha;
        m_run = m_new;
        rescale = true;
      }
      // O_x += P_x(t-1) V was issued before S_x(t), so it has landed: O may
      // be rescaled now, before this tile's first P V is released.
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          ptx::tmem_ld32(o_addr + 32 * c, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          ptx::tmem_st32(o_addr + 32 * c, r);
        }
      }
      const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
      // Per 32-key block: the E8M0 exponent e puts the block's largest weight
      // 2^(mh - m_use) just under the e4m3 maximum 448 = 2^8.807..., so no
      // code saturates; P_q = 2^(x - m_use - e) is rounded to e4m3 and the
      // block's weights are P_q 2^e.  The row sum takes the unrounded values.
      int eb[2];
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) eb[hb] = max(-126, min(0, __float2int_ru(mh[hb] - m_use - 8.807354922057604f)));
      const uint64_t mul2 = ptx::f2_splat(fold ? sl : 1.0f);
      uint32_t pw[8];
      // first 32 keys, with the tile's P and V scale words: released at once
      l_run += mxp_block(&sr[0], mul2, -(m_use + static_cast<float>(eb[0])), pw) * __int_as_float((eb[0] + 127) << 23);
      ptx::tmem_st8(s_addr + C::P_CODES, pw);
      ptx::tmem_st1(s_addr + C::P_SF + quarter,
                    static_cast<uint32_t>(eb[0] + 127) | (static_cast<uint32_t>(eb[1] + 127) << 8) | 0x7F7F0000u);
      ptx::tmem_st4(s_addr + C::V_SF, vw[0], vw[1], vw[2], vw[3]);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&B.p_full[x][0]);
      // the previous item's last P V landed before S_x(t): its epilogue now,
      // while the first half's P V waits for O to be free
      if (pend) epilogue();
      // the second 32 keys
      l_run += mxp_block(&sr[32], mul2, -(m_use + static_cast<float>(eb[1])), pw) * __int_as_float((eb[1] + 127) << 23);
      ptx::tmem_st8(s_addr + C::P_CODES + 8, pw);
      // this side's next tile's K scale words (S_x(t), their slot's last
      // reader, has landed), and its next item's Q scale words
      ptx::tmem_st2(tmem + lane_off + C::tm_sfk(x), kw[0], kw[1]);
      cur.advance(p, iend);
      cur.load(p, lane, kw);
      if (j == t.n_kv - 1 && q_next < iend) ptx::tmem_st1(tmem + lane_off + C::tm_sfq(x) + quarter, qw);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&B.p_full[x][1]);
    }
    if (!ok) break;
    if (p.lse && row < rows) p.lse[static_cast<size_t>(t.q_tok + 128 * x + row) * H + t.h] = row_lse(m_run, l_run);
    pend = true;
    pend_row_ok = row < rows;
    pend_inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    pend_orow = orow;
  }
  if (ok && pend) {  // the last item's epilogue, after its last P V
    ok = ptx::mbar_wait(&B.o_done[x], (gx - 1) & 1, p.timeout_ns, abort);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) epilogue();
  }
  if (!ok && lane == 0) report_failure(p, abort, kStatusActivation);
}

// ------------------------------------------------------------------ kernel

__global__ void __launch_bounds__(384, 1) gdpa_fwd_mxp_kernel(const __grid_constant__ FwdParams p) {
  using C = MxpCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* sm = smem_raw + pad;
  MxpBars& B = *reinterpret_cast<MxpBars*>(sm + C::OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ibeg = p.cta_begin[blockIdx.x];
  const int iend = p.cta_begin[blockIdx.x + 1];
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
      ptx::mbar_init(&B.sf_init[x], 128);
      ptx::mbar_init(&B.mma_drain[x], 1);
    }
    for (int s = 0; s < C::NK; ++s) {  // K and V stages: released by both MMA warps
      ptx::mbar_init(&B.k_full[s], 1);
      ptx::mbar_init(&B.k_empty[s], 2);
    }
    for (int s = 0; s < C::NV; ++s) {
      ptx::mbar_init(&B.v_full[s], 1);
      ptx::mbar_init(&B.v_empty[s], 2);
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
  if (warp < 4) {  // warpgroup 0: producers and MMA issuers, few registers
    ptx::regs_dec<C::REGS_CTRL>();
    if (warp == 0) {
      if (lane == 0) mxp_producer<false>(p, sm, B, ibeg, iend);
    } else if (warp == 2) {
      if (lane == 0) mxp_producer<true>(p, sm, B, ibeg, iend);
    } else {
      mxp_mma(p, sm, B, tmem, ibeg, iend, warp == 1 ? 0 : 1);  // whole warps: MMAs issued warp-uniformly
    }
  } else {  // warpgroups 1 and 2: tiles A and B
    ptx::regs_inc<C::REGS_ACT>();
    mxp_activation(p, B, tmem, ibeg, iend, warp < 8 ? 0 : 1, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::TM_COLS);
}

}  // namespace gdpa
