/*
 * gdpa_oracle.c -- plain fp64 CPU oracle for the jagged GDPA forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code with the CUDA library.
 *
 * What it computes (one (sequence b, head h) at a time, every query row i):
 *
 *   s_ij = scale * <q_i, k_j>            over the bf16 inputs widened to fp64
 *
 *   softmax:  o_i = sum_j exp(s_ij - m_i) v_j / sum_j exp(s_ij - m_i),
 *             m_i = max_j s_ij,  o_i = 0 when the key set is empty
 *   GELU:     o_i = (1 / Lkv_b) * sum_j gelu(s_ij) v_j,
 *             gelu(x) = x/2 * (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))),
 *             o_i = 0 when Lkv_b = 0
 *   SiLU:     o_i = (1 / Lkv_b) * sum_j silu(s_ij) v_j,  silu(x) = x / (1 + e^-x)
 *             (the same form with another activation: the remio.ai
 *             commentary's "alternative activations" of GDPA)
 *
 * with j over the key set K(i):
 *   full attention:  every key j < Lkv_b of the same sequence;
 *   sliding window of W tokens (window_blocks = -W < 0): the keys j with
 *                    i - W < j <= i (causal, W tokens wide);
 *   block window W:  blocks of 64 tokens counted from the sequence start,
 *                    beta(t) = floor(t / 64); keys of the W-1 previous blocks
 *                    and keys j <= i of the query's own block.
 *
 * Sources: jagged, unpadded sequences and the three shape classes (self,
 * long-query/short-KV cross, short-query/long-KV pooled) -- techfeed summary
 * of "GEM Training", section on why LLM infrastructure does not carry over,
 * and its JFA section; attention with the softmax replaced by another
 * activation (GELU, evaluated through tanh) -- same page, GDPA section, and
 * the remio.ai commentary, section on model/system co-design; 64-token
 * block-aligned windows, window a whole number of blocks -- techfeed summary,
 * BlockAttention section, and the aigeeknews translation, co-design section.
 * The token-granular sliding window is the causal window the BlockAttention
 * section names as the step before block-aligned attention (techfeed
 * summary); its width W in tokens is this project's parameter.
 * The output normalisation 1/Lkv of the GELU form and the window-of-blocks
 * semantics (own block causal plus the previous W-1 blocks, one softmax over
 * the union) are this project's readings of those passages.
 *
 * The oracle follows that definition literally: it loops over sequences,
 * heads, queries and keys, in fp64, with libm's exp and tanh.  There is no
 * tiling, no online (running-max) rescaling and no reordering.
 *
 * Backward (oracle_gdpa_bwd): the gradients of the same forward for an
 * upstream gradient dO -- the training step the techfeed summary's JFA
 * section measures for this attention (its backward parallelises dQ, dK,
 * dV).  The formulas are the chain rule written out for one query row i,
 * with P_ij the weight of key j in o_i and dP_ij = <dO_i, v_j>:
 *
 *   dv_j  = sum_i P_ij dO_i
 *   softmax:  P_ij = exp(s_ij - lse_i),  lse_i = log sum_j exp(s_ij),
 *             dS_ij = P_ij (dP_ij - sum_j' P_ij' dP_ij')
 *   GELU:     P_ij = gelu(s_ij) / Lkv_b,  dS_ij = gelu'(s_ij) dP_ij / Lkv_b
 *   dq_i  = scale * sum_j dS_ij k_j,   dk_j = scale * sum_i dS_ij q_i
 *
 * It also returns lse_i (natural log; -inf for an empty key set, 0 for GELU
 * rows), which a forward that keeps it for the backward must reproduce.
 *
 * MXFP8 score operands (oracle_gdpa_fwd_mx): q and k arrive as OCP
 * microscaling values -- an e4m3 element per coordinate and one E8M0 scale
 * per 32 consecutive coordinates of a (token, head) row -- and the forward
 * above runs on their values
 *
 *   q_id = e4m3(q8_id) * 2^(qs_i,floor(d/32) - 127)    (k likewise; v stays bf16)
 *
 * e4m3: 1 sign, 4 exponent (bias 7) and 3 mantissa bits, subnormal below
 * exponent 1, no infinities, S.1111.111 is NaN; E8M0: 2^(e - 127), 0xFF NaN.
 * Source: MXFP8 applied to attention -- techfeed summary of "GEM Training",
 * section on MXFP8 ultra-low-precision training, and the aigeeknews
 * translation, section on compute efficiency ("MXFP8 attention").  Which
 * operands are quantised is not stated there; this oracle quantises the two
 * operands of the score product along their contraction (head) dimension.
 *
 * All three inputs in MXFP8 (oracle_gdpa_fwd_mxfp8): q and k as above, and v
 * quantised along the contraction dimension of P V -- the keys -- so it
 * arrives key-major: for each (head h, coordinate d) one row of VT codes,
 * sequence b's keys at columns [P_b, P_b + Lkv_b) with
 *
 *   P_b = 32 * sum_{b' < b} ceil(Lkv_b' / 32),   VT = P_B,
 *
 * and one E8M0 scale per 32 columns of a row, stored column-block major:
 *
 *   v_jd = e4m3(vt8[(h D + d) VT + P_b + j]) * 2^(vt_sf[((P_b + j) / 32) H D + h D + d] - 127)
 *
 * (a block never spans two sequences: each sequence starts a block).  The
 * forward is then the definition above on these values, with the weights
 * P_ij exact; rounding them to e4m3 on the way to the P V product is a
 * precision of the implementation that the tests' error bar accounts for.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_ACT_SOFTMAX 0
#define ORACLE_ACT_GELU_TANH 1
#define ORACLE_ACT_SILU 2
#define ORACLE_BLOCK 64

/* bf16 bit pattern -> exact double (bf16 is the top half of an IEEE float). */
static double bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP e4m3 ("E4M3FN") element code -> exact double. */
double oracle_e4m3_to_double(uint8_t c) {
  const int e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10); /* m/8 * 2^-6, (1 + m/8) 2^(e-7) */
  return (c & 0x80) ? -mag : mag;
}

/* OCP E8M0 scale code -> 2^(c - 127); 0xFF is NaN. */
double oracle_e8m0_to_double(uint8_t c) { return c == 0xFF ? NAN : ldexp(1.0, (int)c - 127); }

double oracle_gelu_tanh(double x) {
  const double c = sqrt(2.0 / M_PI);
  return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

double oracle_silu(double x) { return x / (1.0 + exp(-x)); }

/* d/dx of oracle_silu: sigma(x) (1 + x (1 - sigma(x))). */
double oracle_silu_grad(double x) {
  const double sg = 1.0 / (1.0 + exp(-x));
  return sg * (1.0 + x * (1.0 - sg));
}

/* The elementwise activation of the non-softmax forms and its derivative. */
static double act_value(int act, double x) { return act == ORACLE_ACT_SILU ? oracle_silu(x) : oracle_gelu_tanh(x); }
double oracle_gelu_tanh_grad(double x);
static double act_grad(int act, double x) {
  return act == ORACLE_ACT_SILU ? oracle_silu_grad(x) : oracle_gelu_tanh_grad(x);
}

/* d/dx of oracle_gelu_tanh. */
double oracle_gelu_tanh_grad(double x) {
  const double c = sqrt(2.0 / M_PI);
  const double t = tanh(c * (x + 0.044715 * x * x * x));
  return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * c * (1.0 + 3.0 * 0.044715 * x * x);
}

/* Is key j in the key set of query i (both counted from the sequence start)? */
static int key_in_set(int64_t i, int64_t j, int window_blocks) {
  if (window_blocks < 0) return j <= i && j > i + window_blocks; /* W = -window_blocks tokens */
  if (window_blocks == 0) return 1;
  int64_t bi = i / ORACLE_BLOCK, bj = j / ORACLE_BLOCK;
  if (bj == bi) return j <= i;                        /* own block, causal */
  return bj < bi && bj >= bi - (window_blocks - 1);   /* W-1 previous blocks */
}

typedef struct {
  const uint16_t *q, *k, *v;
  const int32_t *q_off, *kv_off;
  int B, H, D, act, window_blocks;
  double scale;
  double* out;
  int64_t next_task; /* shared counter over (b, h) tasks */
  /* MXFP8 q and k (used instead of q, k when q8 is set): e4m3 codes
   * [T, H, D] and E8M0 scales [T, H, D/32] */
  const uint8_t *q8, *q_sf, *k8, *k_sf;
  /* MXFP8 v, key-major (used instead of v when vt8 is set): codes [H D, VT],
   * scales [VT / 32, H D], sequence b's first column vt_col[b] */
  const uint8_t *vt8, *vt_sf;
  const int64_t* vt_col;
  int64_t VT;
} job_t;

/* Element d of the (token t, head h) row of q or k, as a double. */
static double qk_value(const job_t* J, int is_k, int64_t t, int h, int d) {
  const int64_t e = (t * J->H + h) * J->D + d;
  if (!J->q8) return bf16_to_double(is_k ? J->k[e] : J->q[e]);
  const uint8_t* codes = is_k ? J->k8 : J->q8;
  const uint8_t* sf = is_k ? J->k_sf : J->q_sf;
  return oracle_e4m3_to_double(codes[e]) * oracle_e8m0_to_double(sf[(t * J->H + h) * (J->D / 32) + d / 32]);
}

/* Element d of key j of sequence b, head h, of v, as a double. */
static double v_value(const job_t* J, int b, int64_t j, int h, int d) {
  const int H = J->H, D = J->D;
  if (!J->vt8) return bf16_to_double(J->v[((J->kv_off[b] + j) * H + h) * D + d]);
  const int64_t col = J->vt_col[b] + j, row = (int64_t)h * D + d;
  return oracle_e4m3_to_double(J->vt8[row * J->VT + col]) *
         oracle_e8m0_to_double(J->vt_sf[(col / 32) * ((int64_t)H * D) + row]);
}

static void run_task(const job_t* J, int b, int h, double* kbuf, double* vbuf, double* qrow, double* s) {
  const int H = J->H, D = J->D;
  const int64_t q0 = J->q_off[b], Lq = J->q_off[b + 1] - q0;
  const int64_t k0 = J->kv_off[b], Lkv = J->kv_off[b + 1] - k0;
  for (int64_t j = 0; j < Lkv; ++j)
    for (int d = 0; d < D; ++d) {
      kbuf[j * D + d] = qk_value(J, 1, k0 + j, h, d);
      vbuf[j * D + d] = v_value(J, b, j, h, d);
    }
  for (int64_t i = 0; i < Lq; ++i) {
    double* o = J->out + ((q0 + i) * H + h) * (int64_t)D;
    for (int d = 0; d < D; ++d) {
      qrow[d] = qk_value(J, 0, q0 + i, h, d);
      o[d] = 0.0;
    }
    /* scores over the key set */
    int any = 0;
    double m = -INFINITY;
    for (int64_t j = 0; j < Lkv; ++j) {
      if (!key_in_set(i, j, J->window_blocks)) continue;
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qrow[d] * kbuf[j * D + d];
      s[j] = J->scale * dot;
      if (s[j] > m) m = s[j];
      any = 1;
    }
    if (!any) continue; /* empty key set: output stays 0 */
    if (J->act == ORACLE_ACT_SOFTMAX) {
      double den = 0.0;
      for (int64_t j = 0; j < Lkv; ++j) {
        if (!key_in_set(i, j, J->window_blocks)) continue;
        double w = exp(s[j] - m);
        den += w;
        for (int d = 0; d < D; ++d) o[d] += w * vbuf[j * D + d];
      }
      for (int d = 0; d < D; ++d) o[d] /= den;
    } else {
      for (int64_t j = 0; j < Lkv; ++j) {
        if (!key_in_set(i, j, J->window_blocks)) continue;
        double g = act_value(J->act, s[j]);
        for (int d = 0; d < D; ++d) o[d] += g * vbuf[j * D + d];
      }
      for (int d = 0; d < D; ++d) o[d] /= (double)Lkv;
    }
  }
}

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  int64_t max_kv = 0;
  for (int b = 0; b < J->B; ++b) {
    int64_t L = J->kv_off[b + 1] - J->kv_off[b];
    if (L > max_kv) max_kv = L;
  }
  double* kbuf = (double*)malloc(sizeof(double) * (size_t)(max_kv * J->D + 1));
  double* vbuf = (double*)malloc(sizeof(double) * (size_t)(max_kv * J->D + 1));
  double* qrow = (double*)malloc(sizeof(double) * (size_t)J->D);
  double* s = (double*)malloc(sizeof(double) * (size_t)(max_kv + 1));
  if (!kbuf || !vbuf || !qrow || !s) {
    free(kbuf); free(vbuf); free(qrow); free(s);
    return (void*)1;
  }
  const int64_t ntask = (int64_t)J->B * J->H;
  for (;;) {
    int64_t t = __atomic_fetch_add(&J->next_task, 1, __ATOMIC_RELAXED);
    if (t >= ntask) break;
    run_task(J, (int)(t / J->H), (int)(t % J->H), kbuf, vbuf, qrow, s);
  }
  free(kbuf); free(vbuf); free(qrow); free(s);
  return NULL;
}

int oracle_num_cpus(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/*
 * q: bf16 bits [Tq, H, D]; k, v: bf16 bits [Tkv, H, D]; q_off, kv_off: int32
 * [B+1] prefix sums starting at 0; out: fp64 [Tq, H, D] (fully written).
 * window_blocks != 0 needs q_off == kv_off (> 0: block window of that many
 * 64-token blocks; < 0: sliding window of -window_blocks tokens).  nthreads <= 0 uses every online
 * CPU.  Returns 0 on success, 1 on a bad argument, 2 on allocation failure.
 */
static int run_fwd(job_t* J, int nthreads) {
  const int B = J->B, H = J->H, D = J->D, act = J->act, window_blocks = J->window_blocks;
  const int32_t *q_off = J->q_off, *kv_off = J->kv_off;
  if (B < 0 || H <= 0 || D <= 0 || (act != ORACLE_ACT_SOFTMAX && act != ORACLE_ACT_GELU_TANH && act != ORACLE_ACT_SILU))
    return 1;
  if (!q_off || !kv_off || q_off[0] != 0 || kv_off[0] != 0) return 1;
  for (int b = 0; b < B; ++b) {
    if (q_off[b + 1] < q_off[b] || kv_off[b + 1] < kv_off[b]) return 1;
    if (window_blocks != 0 && q_off[b + 1] != kv_off[b + 1]) return 1;
  }
  if (B == 0 || q_off[B] == 0) return 0;
  const int mx = J->q8 != NULL;
  if (!J->out || (mx ? !J->q_sf : !J->q)) return 1;
  if (kv_off[B] > 0 && (!(J->v || J->vt8) || (mx ? (!J->k8 || !J->k_sf) : !J->k))) return 1;
  if (J->vt8 && kv_off[B] > 0 && !J->vt_sf) return 1;
  if (nthreads <= 0) nthreads = oracle_num_cpus();
  if (nthreads > B * H) nthreads = B * H;
  if (nthreads < 1) nthreads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return 2;
  int started = 0, failed = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, worker, J) != 0) break;
    ++started;
  }
  if (started == 0) { /* no thread could start: run on this one */
    failed = worker(J) != NULL;
  }
  for (int t = 0; t < started; ++t) {
    void* r = NULL;
    pthread_join(th[t], &r);
    if (r) failed = 1;
  }
  free(th);
  return failed ? 2 : 0;
}

/*
 * q: bf16 bits [Tq, H, D]; k, v: bf16 bits [Tkv, H, D]; q_off, kv_off: int32
 * [B+1] prefix sums starting at 0; out: fp64 [Tq, H, D] (fully written).
 * window_blocks != 0 needs q_off == kv_off (> 0: block window of that many
 * 64-token blocks; < 0: sliding window of -window_blocks tokens).  nthreads <= 0 uses every online
 * CPU.  Returns 0 on success, 1 on a bad argument, 2 on allocation failure.
 */
int oracle_gdpa_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* q_off,
                    const int32_t* kv_off, int B, int H, int D, int act, int window_blocks, double scale,
                    double* out, int nthreads) {
  job_t J = {q, k, v, q_off, kv_off, B, H, D, act, window_blocks, scale, out, 0, NULL, NULL, NULL, NULL,
             NULL, NULL, NULL, 0};
  return run_fwd(&J, nthreads);
}

/*
 * The same forward with MXFP8 q and k: q8 / k8 e4m3 codes [T, H, D], q_sf /
 * k_sf E8M0 scales [T, H, D/32] (D a multiple of 32); v bf16 bits.  Full
 * attention or a window exactly as oracle_gdpa_fwd.
 */
int oracle_gdpa_fwd_mx(const uint8_t* q8, const uint8_t* q_sf, const uint8_t* k8, const uint8_t* k_sf,
                       const uint16_t* v, const int32_t* q_off, const int32_t* kv_off, int B, int H, int D, int act,
                       int window_blocks, double scale, double* out, int nthreads) {
  if (!q8 || D % 32 != 0) return 1;
  job_t J = {NULL, NULL, v, q_off, kv_off, B, H, D, act, window_blocks, scale, out, 0, q8, q_sf, k8, k_sf,
             NULL, NULL, NULL, 0};
  return run_fwd(&J, nthreads);
}

/* Columns of the key-major v layout: P_b = 32 sum_{b' < b} ceil(Lkv_b' / 32)
 * into col[0..B] (col[B] = VT).  kv_off must be a valid prefix sum. */
static void vt_columns(const int32_t* kv_off, int B, int64_t* col) {
  col[0] = 0;
  for (int b = 0; b < B; ++b) col[b + 1] = col[b] + 32 * (((int64_t)kv_off[b + 1] - kv_off[b] + 31) / 32);
}

int64_t oracle_vt_columns(const int32_t* kv_off, int B) {
  if (B < 0 || !kv_off) return -1;
  int64_t c = 0;
  for (int b = 0; b < B; ++b) c += 32 * (((int64_t)kv_off[b + 1] - kv_off[b] + 31) / 32);
  return c;
}

/*
 * The forward with q, k and v in MXFP8: q8 / k8 e4m3 codes [T, H, D], q_sf /
 * k_sf E8M0 scales [T, H, D/32]; vt8 e4m3 codes [H D, VT] and vt_sf E8M0
 * scales [VT / 32, H D] in the key-major layout of the header comment (VT
 * must equal oracle_vt_columns).  D a multiple of 32.  Full attention or a
 * window exactly as oracle_gdpa_fwd.
 */
int oracle_gdpa_fwd_mxfp8(const uint8_t* q8, const uint8_t* q_sf, const uint8_t* k8, const uint8_t* k_sf,
                          const uint8_t* vt8, const uint8_t* vt_sf, int64_t VT, const int32_t* q_off,
                          const int32_t* kv_off, int B, int H, int D, int act, int window_blocks, double scale,
                          double* out, int nthreads) {
  if (!q8 || !vt8 || D % 32 != 0 || B < 0 || !kv_off) return 1;
  for (int b = 0; b < B; ++b)
    if (kv_off[b + 1] < kv_off[b]) return 1;
  if (VT != oracle_vt_columns(kv_off, B)) return 1;
  int64_t* col = (int64_t*)malloc(sizeof(int64_t) * ((size_t)B + 1));
  if (!col) return 2;
  vt_columns(kv_off, B, col);
  job_t J = {NULL, NULL, NULL, q_off, kv_off, B, H, D, act, window_blocks, scale, out, 0, q8, q_sf, k8, k_sf,
             vt8, vt_sf, col, VT};
  const int rc = run_fwd(&J, nthreads);
  free(col);
  return rc;
}

/* ------------------------------------------------------------------ backward */

typedef struct {
  const uint16_t *q, *k, *v, *dout;
  const int32_t *q_off, *kv_off;
  int B, H, D, act, window_blocks;
  double scale;
  double *dq, *dk, *dv, *lse;
  int64_t next_task;
} bjob_t;

typedef struct {
  double *kbuf, *vbuf, *qrow, *drow, *s, *p, *dp;
} bscratch_t;

static void run_bwd_task(const bjob_t* J, int b, int h, const bscratch_t* W) {
  const int H = J->H, D = J->D;
  const int64_t q0 = J->q_off[b], Lq = J->q_off[b + 1] - q0;
  const int64_t k0 = J->kv_off[b], Lkv = J->kv_off[b + 1] - k0;
  for (int64_t j = 0; j < Lkv; ++j)
    for (int d = 0; d < D; ++d) {
      W->kbuf[j * D + d] = bf16_to_double(J->k[((k0 + j) * H + h) * D + d]);
      W->vbuf[j * D + d] = bf16_to_double(J->v[((k0 + j) * H + h) * D + d]);
      J->dk[((k0 + j) * H + h) * (int64_t)D + d] = 0.0;
      J->dv[((k0 + j) * H + h) * (int64_t)D + d] = 0.0;
    }
  for (int64_t i = 0; i < Lq; ++i) {
    double* dqi = J->dq + ((q0 + i) * H + h) * (int64_t)D;
    for (int d = 0; d < D; ++d) {
      W->qrow[d] = bf16_to_double(J->q[((q0 + i) * H + h) * D + d]);
      W->drow[d] = bf16_to_double(J->dout[((q0 + i) * H + h) * D + d]);
      dqi[d] = 0.0;
    }
    double* lse_i = J->lse + (q0 + i) * H + h;
    *lse_i = J->act == ORACLE_ACT_SOFTMAX ? -INFINITY : 0.0;
    int any = 0;
    double m = -INFINITY;
    for (int64_t j = 0; j < Lkv; ++j) {
      if (!key_in_set(i, j, J->window_blocks)) continue;
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += W->qrow[d] * W->kbuf[j * D + d];
      W->s[j] = J->scale * dot;
      if (W->s[j] > m) m = W->s[j];
      any = 1;
    }
    if (!any) continue; /* empty key set: no gradient flows */
    /* P_ij and dP_ij = <dO_i, v_j> over the key set */
    double den = 0.0;
    if (J->act == ORACLE_ACT_SOFTMAX) {
      for (int64_t j = 0; j < Lkv; ++j)
        if (key_in_set(i, j, J->window_blocks)) den += exp(W->s[j] - m);
      *lse_i = m + log(den);
    }
    double dsum = 0.0; /* sum_j P_ij dP_ij (softmax) */
    for (int64_t j = 0; j < Lkv; ++j) {
      if (!key_in_set(i, j, J->window_blocks)) continue;
      W->p[j] = J->act == ORACLE_ACT_SOFTMAX ? exp(W->s[j] - *lse_i) : act_value(J->act, W->s[j]) / (double)Lkv;
      double dp = 0.0;
      for (int d = 0; d < D; ++d) dp += W->drow[d] * W->vbuf[j * D + d];
      W->dp[j] = dp;
      dsum += W->p[j] * dp;
    }
    for (int64_t j = 0; j < Lkv; ++j) {
      if (!key_in_set(i, j, J->window_blocks)) continue;
      const double ds = J->act == ORACLE_ACT_SOFTMAX ? W->p[j] * (W->dp[j] - dsum)
                                                     : act_grad(J->act, W->s[j]) * W->dp[j] / (double)Lkv;
      double* dkj = J->dk + ((k0 + j) * H + h) * (int64_t)D;
      double* dvj = J->dv + ((k0 + j) * H + h) * (int64_t)D;
      for (int d = 0; d < D; ++d) {
        dqi[d] += J->scale * ds * W->kbuf[j * D + d];
        dkj[d] += J->scale * ds * W->qrow[d];
        dvj[d] += W->p[j] * W->drow[d];
      }
    }
  }
}

static void* bwd_worker(void* arg) {
  bjob_t* J = (bjob_t*)arg;
  int64_t max_kv = 0;
  for (int b = 0; b < J->B; ++b) {
    int64_t L = J->kv_off[b + 1] - J->kv_off[b];
    if (L > max_kv) max_kv = L;
  }
  bscratch_t W;
  W.kbuf = (double*)malloc(sizeof(double) * (size_t)(max_kv * J->D + 1));
  W.vbuf = (double*)malloc(sizeof(double) * (size_t)(max_kv * J->D + 1));
  W.qrow = (double*)malloc(sizeof(double) * (size_t)J->D);
  W.drow = (double*)malloc(sizeof(double) * (size_t)J->D);
  W.s = (double*)malloc(sizeof(double) * (size_t)(max_kv + 1));
  W.p = (double*)malloc(sizeof(double) * (size_t)(max_kv + 1));
  W.dp = (double*)malloc(sizeof(double) * (size_t)(max_kv + 1));
  void* rc = NULL;
  if (!W.kbuf || !W.vbuf || !W.qrow || !W.drow || !W.s || !W.p || !W.dp) {
    rc = (void*)1;
  } else {
    const int64_t ntask = (int64_t)J->B * J->H;
    for (;;) {
      int64_t t = __atomic_fetch_add(&J->next_task, 1, __ATOMIC_RELAXED);
      if (t >= ntask) break;
      run_bwd_task(J, (int)(t / J->H), (int)(t % J->H), &W);
    }
  }
  free(W.kbuf); free(W.vbuf); free(W.qrow); free(W.drow); free(W.s); free(W.p); free(W.dp);
  return rc;
}

/*
 * Gradients of oracle_gdpa_fwd for the upstream gradient dout (bf16 bits
 * [Tq, H, D]).  dq: fp64 [Tq, H, D]; dk, dv: fp64 [Tkv, H, D]; lse: fp64
 * [Tq, H]; all fully written (keys no query sees get zero gradients).
 * Arguments and return codes as oracle_gdpa_fwd.
 */
int oracle_gdpa_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                    const int32_t* q_off, const int32_t* kv_off, int B, int H, int D, int act, int window_blocks,
                    double scale, double* dq, double* dk, double* dv, double* lse, int nthreads) {
  if (B < 0 || H <= 0 || D <= 0 || (act != ORACLE_ACT_SOFTMAX && act != ORACLE_ACT_GELU_TANH && act != ORACLE_ACT_SILU))
    return 1;
  if (!q_off || !kv_off || q_off[0] != 0 || kv_off[0] != 0) return 1;
  for (int b = 0; b < B; ++b) {
    if (q_off[b + 1] < q_off[b] || kv_off[b + 1] < kv_off[b]) return 1;
    if (window_blocks != 0 && q_off[b + 1] != kv_off[b + 1]) return 1;
  }
  if (B == 0) return 0;
  if ((q_off[B] > 0 && (!q || !dout || !dq || !lse)) || (kv_off[B] > 0 && (!k || !v || !dk || !dv))) return 1;
  bjob_t J = {q, k, v, dout, q_off, kv_off, B, H, D, act, window_blocks, scale, dq, dk, dv, lse, 0};
  if (nthreads <= 0) nthreads = oracle_num_cpus();
  if (nthreads > B * H) nthreads = B * H;
  if (nthreads < 1) nthreads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return 2;
  int started = 0, failed = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, bwd_worker, &J) != 0) break;
    ++started;
  }
  if (started == 0) failed = bwd_worker(&J) != NULL;
  for (int t = 0; t < started; ++t) {
    void* r = NULL;
    pthread_join(th[t], &r);
    if (r) failed = 1;
  }
  free(th);
  return failed ? 2 : 0;
}
