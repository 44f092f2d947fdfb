// gdpa_fwd_pair.cuh -- jagged GDPA forward, two query tiles per work item.
//
// Full (non-window) attention.  A work item is 256 query rows of one
// (sequence, head) -- tile A = rows [q0, q0+128), tile B = [q0+128, q0+256),
// B may be empty -- against the sequence's whole key range.  Every K/V tile
// staged in shared memory feeds both tiles' MMAs, which halves the K/V
// traffic per FLOP against one tile per item, and the two activation
// warpgroups (one per tile) take turns with the tensor core:
//
//   MMA thread, per K/V tile g:  O_A += P_A(g-1) V(g-1);  S_A = Q_A K(g)^T;
//                                O_B += P_B(g-1) V(g-1);  S_B = Q_B K(g)^T
//   warpgroup A works on S_A(g) while the tensor core runs the B half, and
//   the other way round.
//
// Threads (352): warp 0 TMA producer for Q and K, warp 10 TMA producer for
// V, warp 1 MMA issuer + TMEM owner, warps 2-5 tile A activation/epilogue,
// warps 6-9 tile B.  TMEM (512
// columns): S_A 0, S_B 128, O_A 256, O_B 384.  An activation thread holds
// one query row; it reads S from TMEM twice (row max, then exponentials) in
// 32-column chunks, so only ~64 scores are live in registers at a time.
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
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;
  __host__ __device__ static constexpr uint32_t tm_s(int x) { return x ? 128u : 0u; }    // S_A, S_B
  __host__ __device__ static constexpr uint32_t tm_o(int x) { return x ? 384u : 256u; }  // O_A, O_B
  static constexpr uint32_t TM_COLS = 512;
  static constexpr int THREADS = 352;  // 11 warps
  static_assert(384 + D <= TM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <int D>
struct PairBars {
  uint64_t q_full[2][PairCfg<D>::NQS], q_empty[2][PairCfg<D>::NQS];
  uint64_t k_full[PairCfg<D>::NK], k_empty[PairCfg<D>::NK];
  uint64_t v_full[PairCfg<D>::NV], v_empty[PairCfg<D>::NV];
  uint64_t s_full[2], p_full[2], o_done[2], o_empty[2];
  uint64_t mma_drain;
  uint32_t tmem_slot;
  int abort;
};

struct PairItem {
  int h, q0, kv_end, n_kv, q_tok, kv_tok, Lkv;
  int rows[2];  // valid rows of tile A and tile B (B may be 0)
};

__device__ __forceinline__ PairItem decode_pair(const FwdParams& p, int idx) {
  const int4 it = __ldg(p.items + idx);
  PairItem v;
  const int b = it.x;
  v.h = it.y;
  v.q0 = it.z;
  const int qs = __ldg(p.q_off + b), qe = __ldg(p.q_off + b + 1);
  const int ks = __ldg(p.kv_off + b), ke = __ldg(p.kv_off + b + 1);
  v.q_tok = qs + v.q0;
  v.kv_tok = ks;
  v.Lkv = ke - ks;
  v.kv_end = v.Lkv;
  const int left = qe - qs - v.q0;
  v.rows[0] = min(128, left);
  v.rows[1] = max(0, min(128, left - 128));
  v.n_kv = (v.Lkv + 127) / 128;
  return v;
}

// ------------------------------------------------------------------ producer

// Two producer threads: one stages Q and K, the other V, so that a K load
// never waits behind a V slot.
template <int D, bool LOAD_V>
__device__ void pair_producer(const FwdParams& p, uint8_t* sm, PairBars<D>& B, int ibeg, int iend) {
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
  for (int idx = ibeg; idx < iend && ok; ++idx) {
    const PairItem t = decode_pair(p, idx);
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
      const int y = t.kv_tok + 128 * j;
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
  int first, n16;
};

template <int D>
__device__ __forceinline__ bool pair_issue_pv(const FwdParams& p, uint8_t* sm, PairBars<D>& B, uint32_t tmem, int x,
                                              const PairPV& P) {
  using C = PairCfg<D>;
  volatile int* abort = &B.abort;
  if (!ptx::mbar_wait(&B.p_full[x], P.gx & 1, p.timeout_ns, abort)) return false;
  if (P.first && !ptx::mbar_wait(&B.o_empty[x], (P.item & 1) ^ 1, p.timeout_ns, abort)) return false;
  const int sv = P.g % C::NV;
  if (!ptx::mbar_wait(&B.v_full[sv], (P.g / C::NV) & 1, p.timeout_ns, abort)) return false;
  ptx::tc_fence_after();
  const uint32_t v_base = ptx::smem_u32(sm + C::OFF_V + sv * C::TILE_BYTES);
  constexpr uint32_t idesc = ptx::idesc_bf16(128, D, 1);
  for (int kk = 0; kk < P.n16; ++kk) {
    const uint64_t bdesc = ptx::sdesc_sw128(v_base + kk * 2048, C::CHUNK_BYTES, 1024);
    ptx::mma_ts(tmem + C::tm_o(x), tmem + C::tm_s(x) + 8 * kk, bdesc, idesc, (P.first && kk == 0) ? 0u : 1u);
  }
  ptx::mma_commit(&B.o_done[x]);
  return true;
}

template <int D>
__device__ void pair_mma(const FwdParams& p, uint8_t* sm, PairBars<D>& B, uint32_t tmem, int ibeg, int iend) {
  using C = PairCfg<D>;
  volatile int* abort = &B.abort;
  int qn[2] = {0, 0};       // items seen by each side (Q stage and O buffer use counts)
  uint32_t gx[2] = {0, 0};  // tiles processed by each side
  uint32_t g = 0;
  bool ok = true;
  bool pend[2] = {false, false};
  PairPV pv[2] = {{0, 0, 0, 0, 0}, {0, 0, 0, 0, 0}};
  bool pend_v = false;
  uint32_t pend_v_g = 0;
  for (int idx = ibeg; idx < iend && ok; ++idx) {
    const PairItem t = decode_pair(p, idx);
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
      const int ncols = min(128, t.kv_end - 128 * j);
      const int n16 = (ncols + 15) >> 4;
      const uint32_t idesc = ptx::idesc_bf16(128, n16 * 16, 0);
      const uint32_t k_base = ptx::smem_u32(sm + C::OFF_K + sk * C::TILE_BYTES);
      for (int x = 0; x < 2; ++x) {
        // O_x += P_x(prev) V(prev) must precede S_x = Q_x K^T: P_x lives in S_x's columns.
        if (pend[x]) {
          ok = pair_issue_pv<D>(p, sm, B, tmem, x, pv[x]);
          if (!ok) break;
          pend[x] = false;
        }
        if (!has[x]) continue;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          ptx::mma_ss(tmem + C::tm_s(x), ptx::sdesc_sw128(q_base[x] + off, 16, 1024),
                      ptx::sdesc_sw128(k_base + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(&B.s_full[x]);
      }
      if (!ok) break;
      if (pend_v) ptx::mma_commit(&B.v_empty[pend_v_g % C::NV]);  // both P V of the previous tile issued
      ptx::mma_commit(&B.k_empty[sk]);
      if (j == t.n_kv - 1) {
        for (int x = 0; x < 2; ++x)
          if (has[x]) ptx::mma_commit(&B.q_empty[x][qn[x] % C::NQS]);
      }
      for (int x = 0; x < 2; ++x) {
        if (!has[x]) continue;
        pv[x] = PairPV{gx[x], g, qn[x], j == 0 ? 1 : 0, n16};
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
  if (ok && pend_v) ptx::mma_commit(&B.v_empty[pend_v_g % C::NV]);
  if (!ok) report_failure(p, abort, kStatusMma);
  ptx::mma_commit(&B.mma_drain);
  const int never = 0;
  ptx::mbar_wait(&B.mma_drain, 0, 100000000ull, &never);
}

// ------------------------------------------------------------------ activation + epilogue

template <int D, int ACT>
__device__ void pair_activation(const FwdParams& p, PairBars<D>& B, uint32_t tmem, int ibeg, int iend, int x,
                                int warp, int lane) {
  using C = PairCfg<D>;
  volatile int* abort = &B.abort;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t s_addr = tmem + lane_off + C::tm_s(x);
  const uint32_t o_addr = tmem + lane_off + C::tm_o(x);
  const float sl = p.score_scale;
  const int H = p.H;
  uint32_t gx = 0;
  bool ok = true;
  for (int idx = ibeg; idx < iend && ok; ++idx) {
    const PairItem t = decode_pair(p, idx);
    const int rows = t.rows[x];
    __nv_bfloat16* orow = p.out + (static_cast<size_t>(t.q_tok + 128 * x + row) * H + t.h) * D;
    if (t.n_kv == 0) {  // no keys: zero output rows
      if (row < rows) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }
    if (rows == 0) continue;  // this side has no tile in the item
    const bool rows_live = __any_sync(0xffffffffu, row < rows);
    float m_run = -INFINITY, l_run = 0.0f;
    for (int j = 0; j < t.n_kv; ++j, ++gx) {
      ok = ptx::mbar_wait(&B.s_full[x], gx & 1, p.timeout_ns, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      float alpha = 1.0f;
      bool rescale = false;
      if (rows_live) {
        const int ncols = min(128, t.kv_end - 128 * j);  // same for every row
        const bool full = ncols == 128;
        const int nch = (ncols + 31) >> 5;
        if (ACT == kActSoftmax) {
          // Scores in log2 units: x = s * scale * log2(e).  With scale > 0
          // the scaling is folded into the exponent's FMA.
          const bool fold = sl > 0.0f;
          // pass 1: row max over the valid columns
          float m2[2] = {-INFINITY, -INFINITY};
#pragma unroll
          for (int cp = 0; cp < 2; ++cp) {
            if (2 * cp >= nch) break;
            uint32_t r[2][32];
            ptx::tmem_ld32(s_addr + 64 * cp, r[0]);
            if (2 * cp + 1 < nch) ptx::tmem_ld32(s_addr + 64 * cp + 32, r[1]);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (2 * cp + h >= nch) break;
              if (full && fold) {
#pragma unroll
                for (int u = 0; u < 32; u += 4) {
                  m2[0] = ptx::max3(m2[0], __uint_as_float(r[h][u]), __uint_as_float(r[h][u + 1]));
                  m2[1] = ptx::max3(m2[1], __uint_as_float(r[h][u + 2]), __uint_as_float(r[h][u + 3]));
                }
              } else {  // ragged tile, or scale <= 0 (scale first, then take the max)
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                  const int c = 64 * cp + 32 * h + u;
                  float v = __uint_as_float(r[h][u]);
                  if (!fold) v *= sl;
                  m2[u & 1] = fmaxf(m2[u & 1], c < ncols ? v : -INFINITY);
                }
              }
            }
          }
          float mx = fmaxf(m2[0], m2[1]);
          if (fold) mx *= sl;
          const float m_new = fmaxf(m_run, mx);
          if (j == 0) {
            m_run = m_new;
          } else if (m_new > m_run + 8.0f) {
            alpha = ptx::ex2_approx(m_run - m_new);
            l_run *= alpha;
            m_run = m_new;
            rescale = true;
          }
          const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
          const uint64_t mul2 = ptx::f2_pack(sl, sl);   // scale * log2(e), both lanes
          const uint64_t neg2 = ptx::f2_pack(-m_use, -m_use);
          // pass 2: exponentials, row sum, P (bf16 pairs) over the scores
          uint64_t acc[4] = {0, 0, 0, 0};  // +0.0f pairs
#pragma unroll
          for (int cp = 0; cp < 2; ++cp) {
            if (2 * cp >= nch) break;
            uint32_t r[2][32];
            ptx::tmem_ld32(s_addr + 64 * cp, r[0]);
            if (2 * cp + 1 < nch) ptx::tmem_ld32(s_addr + 64 * cp + 32, r[1]);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (2 * cp + h >= nch) break;
              uint32_t pk[16];
              if (full) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                  const uint64_t x2 = ptx::f2_fma(ptx::f2_pack(__uint_as_float(r[h][2 * u]), __uint_as_float(r[h][2 * u + 1])),
                                                  mul2, neg2);
                  float a, b;
                  ptx::f2_unpack(x2, a, b);
                  a = ptx::ex2_approx(a);
                  b = ptx::ex2_approx(b);
                  acc[u & 3] = ptx::f2_add(acc[u & 3], ptx::f2_pack(a, b));
                  pk[u] = ptx::pack_bf16x2(a, b);
                }
              } else {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                  const int c = 64 * cp + 32 * h + 2 * u;
                  const uint64_t x2 = ptx::f2_fma(ptx::f2_pack(__uint_as_float(r[h][2 * u]), __uint_as_float(r[h][2 * u + 1])),
                                                  mul2, neg2);
                  float a, b;
                  ptx::f2_unpack(x2, a, b);
                  a = c < ncols ? ptx::ex2_approx(a) : 0.0f;
                  b = c + 1 < ncols ? ptx::ex2_approx(b) : 0.0f;
                  acc[u & 3] = ptx::f2_add(acc[u & 3], ptx::f2_pack(a, b));
                  pk[u] = ptx::pack_bf16x2(a, b);
                }
              }
              ptx::tmem_st16(s_addr + 32 * cp + 16 * h, pk);
            }
          }
          const uint64_t acc01 = ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3]));
          float sa, sb;
          ptx::f2_unpack(acc01, sa, sb);
          l_run += sa + sb;
        } else {  // GELU, one pass
#pragma unroll
          for (int cp = 0; cp < 2; ++cp) {
            if (2 * cp >= nch) break;
            uint32_t r[2][32];
            ptx::tmem_ld32(s_addr + 64 * cp, r[0]);
            if (2 * cp + 1 < nch) ptx::tmem_ld32(s_addr + 64 * cp + 32, r[1]);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (2 * cp + h >= nch) break;
              uint32_t pk[16];
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const int c = 64 * cp + 32 * h + 2 * u;
                float a, b;
                gelu_tanh_alu2(__uint_as_float(r[h][2 * u]) * sl, __uint_as_float(r[h][2 * u + 1]) * sl, a, b);
                if (!full) {
                  a = c < ncols ? a : 0.0f;
                  b = c + 1 < ncols ? b : 0.0f;
                }
                pk[u] = ptx::pack_bf16x2(a, b);
              }
              ptx::tmem_st16(s_addr + 32 * cp + 16 * h, pk);
            }
          }
        }
        ptx::tmem_wait_st();
      }
      // O_x += P_x(g-1) V(g-1) was issued before S_x(g) and has landed; the
      // wait is immediate and keeps this thread's view of the phase exact.
      if (gx >= 1) {
        ok = ptx::mbar_wait(&B.o_done[x], (gx - 1) & 1, p.timeout_ns, abort);
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
      ptx::mbar_arrive(&B.p_full[x]);
    }
    if (!ok) break;
    ok = ptx::mbar_wait(&B.o_done[x], (gx - 1) & 1, p.timeout_ns, abort);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    ptx::tc_fence_after();
    const float inv = (ACT == kActSoftmax) ? (l_run > 0.0f ? 1.0f / l_run : 0.0f) : 1.0f / static_cast<float>(t.Lkv);
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
    ptx::mbar_arrive(&B.o_empty[x]);
  }
  if (!ok && lane == 0) report_failure(p, abort, kStatusActivation);
}

// ------------------------------------------------------------------ kernel

template <int D, int ACT>
__global__ void __launch_bounds__(352, 1) gdpa_fwd_pair_kernel(const __grid_constant__ FwdParams p) {
  using C = PairCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* sm = smem_raw + pad;
  PairBars<D>& B = *reinterpret_cast<PairBars<D>*>(sm + C::OFF_BAR);
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
      ptx::mbar_init(&B.p_full[x], 128);
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
    if (lane == 0) pair_producer<D, false>(p, sm, B, ibeg, iend);
  } else if (warp == 10) {
    if (lane == 0) pair_producer<D, true>(p, sm, B, ibeg, iend);
  } else if (warp == 1) {
    if (lane == 0) pair_mma<D>(p, sm, B, tmem, ibeg, iend);
  } else {
    pair_activation<D, ACT>(p, B, tmem, ibeg, iend, warp < 6 ? 0 : 1, warp, lane);
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::TM_COLS);
}

}  // namespace gdpa
