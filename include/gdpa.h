/*
 * gdpa.h -- C ABI of libgdpa: forward and backward passes of jagged
 * Generalized Dot-Product Attention (GDPA) on NVIDIA GB300 (sm_103a).
 *
 * The operation (techfeed summary of "GEM Training", sections "JFA" and
 * "GDPA"; remio.ai commentary, section on model/system co-design): attention
 * over a batch of variable-length, unpadded sequences, where the activation
 * applied to the scores is either a softmax or a GELU (tanh form), and where
 * the self-attention variant may be restricted to 64-token block-aligned
 * windows (techfeed summary, section "BlockAttention"; aigeeknews translation,
 * co-design section).  For sequence b, head h and query row i < Lq_b:
 *
 *   s_ij = scale * <q_i, k_j>                                  j in K(i)
 *   softmax : o_i = sum_j exp(s_ij - max s) v_j / sum_j exp(s_ij - max s)
 *   GELU    : o_i = (1/Lkv_b) * sum_j gelu_tanh(s_ij) v_j
 *   SiLU    : o_i = (1/Lkv_b) * sum_j silu(s_ij) v_j        (GDPA_ACT_SILU)
 *
 *   K(i) = all keys j < Lkv_b of sequence b            (window_blocks == 0)
 *        = keys j <= i with floor(i/64) - floor(j/64) <= window_blocks - 1
 *                                                      (window_blocks  > 0)
 *        = keys i - W < j <= i   (gdpa_fwd_sliding / gdpa_bwd_sliding, W tokens)
 *
 * The training entry points keep the softmax row logsumexp in the forward
 * (gdpa_fwd_lse, gdpa_fwd_sliding) and return dq, dk, dv in the backward
 * (gdpa_bwd, gdpa_bwd_sliding).  gdpa_fwd_mx takes q and k in MXFP8,
 * gdpa_fwd_mxfp8 q, k and v.
 *
 * An empty key set gives o_i = 0.  The GELU's tanh is rewritten as a
 * logistic function, gelu(x) = x sigma(2u), whose sigma takes one of two
 * routes (gdpa_act_route_t): the special-function unit's exp2 and reciprocal
 * (the default), or the ALU-only form of the GDPA section ("ALU-only
 * activation", valid because QK-norm bounds the scores): a range-reduced
 * 6th-order Taylor polynomial of exp and a Newton reciprocal.  Either is
 * within 1e-3 of the exact tanh-GELU for |s| <= 17 and saturates correctly
 * beyond.
 *
 * Data layout (all pointers are device pointers unless named h_*):
 *   q    bf16 [Tq,  H, D]   row-major, contiguous, Tq  = q_offsets[B]
 *   k, v bf16 [Tkv, H, D]   row-major, contiguous, Tkv = kv_offsets[B]
 *   out  bf16 [Tq,  H, D]   every row is written (zeros for empty key sets)
 *   q_offsets, kv_offsets  int32 [B+1], offsets[0] = 0, non-decreasing
 * q, k, v and out must be 16-byte aligned.  D must be 64 or 128 (128 for
 * gdpa_fwd_mx, whose q and k are e4m3 codes with E8M0 scales).  Tq and Tkv
 * must be below 2^31.  Windows (block or sliding) require q_offsets ==
 * kv_offsets and act == GDPA_ACT_SOFTMAX.
 *
 * Ownership: the caller owns every buffer it passes; the library never frees
 * them and keeps no reference after the call returns (the GPU may still be
 * reading them until the stream reaches the end of the launched work).  The
 * library owns its plans and internal per-device work-list buffers (two,
 * used in turn).
 *
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 * stream).  All kernels are enqueued on it; the entry points that plan on
 * every call (gdpa_fwd, gdpa_fwd_async, gdpa_fwd_lse, gdpa_fwd_sliding,
 * gdpa_fwd_mx, gdpa_fwd_mxfp8) copy their work list up on a library-owned
 * stream that `stream` then waits for (on a stream being captured, the copy
 * stays on that stream).  The pair
 * kernels take their work items at run time from a device counter; each
 * launch uses its own counter from a fixed pool of 1024, so launches in
 * flight at the same time on different streams are independent unless more
 * than 1024 are.
 *
 * Errors: every entry point returns a gdpa_status_t and never throws or
 * aborts.  Kernel-side failures (a bounded wait that ran out) are recorded in
 * a device status word; gdpa_device_status() reads and clears it.
 */
#ifndef GDPA_H_
#define GDPA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDPA_ACT_SOFTMAX = 0,    /* online softmax */
  GDPA_ACT_GELU_TANH = 1,  /* (1/Lkv) * sum gelu_tanh(s) v (sigma route: gdpa_act_route_t) */
  GDPA_ACT_SILU = 2        /* (1/Lkv) * sum silu(s) v, silu(x) = x sigma(x), the same sigma
                              (an alternative activation of GDPA: remio.ai commentary,
                              model/system co-design section); no windows */
} gdpa_act_t;

/*
 * How the GELU and SiLU activations evaluate their sigma (process-wide, see
 * gdpa_set_act_route).  Both compute the same function to fp32 level:
 *   GDPA_ROUTE_SFU: sigma(z) = 1 / (1 + 2^(-z log2 e)) with the
 *     special-function unit's ex2.approx and rcp.approx (the default: on
 *     sm_103a it measured faster than the polynomial in every forward kernel);
 *   GDPA_ROUTE_ALU: the ALU-only form of the GDPA section of the techfeed
 *     summary of "GEM Training" (a 6th-order Taylor polynomial of exp after
 *     range reduction, Newton reciprocal), FMA and integer instructions only.
 * The backward follows the same route (value and derivative).
 */
typedef enum {
  GDPA_ROUTE_SFU = 0,
  GDPA_ROUTE_ALU = 1
} gdpa_act_route_t;

typedef enum {
  GDPA_OK = 0,
  GDPA_ERR_INVALID_ARG = 1,    /* bad pointer, size, offsets or combination */
  GDPA_ERR_UNSUPPORTED = 2,    /* valid request the library does not implement */
  GDPA_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
  GDPA_ERR_DEVICE_TIMEOUT = 4, /* a kernel wait ran out of time (device status word) */
  GDPA_ERR_NO_MEMORY = 5       /* host or device allocation failed, or capacity too small */
} gdpa_status_t;

/* One unit of GPU work: query rows [q0, q0+R) of sequence `seq`, head
 * `head` (R = 128, or 256 for full attention over sequences averaging more
 * than 128 queries), against keys from `kv0` (sequence-local) to the end of
 * its key range.  Produced by the host tile planner (GDPA section: valid tiles are
 * precomputed on the CPU, empty ones skipped, and spread over the SMs). */
typedef struct {
  int32_t seq;
  int32_t head;
  int32_t q0;
  int32_t kv0;
} gdpa_work_item_t;

typedef struct gdpa_plan gdpa_plan_t;

/*
 * gdpa_fwd -- the whole forward pass in one call.
 * q_offsets / kv_offsets are DEVICE pointers: the call copies them to the host
 * (this synchronises `stream` once), plans the work list, uploads it to a
 * library-owned device buffer and launches the kernel on `stream`.  `scale`
 * multiplies every score.  Returns GDPA_OK once the kernel is enqueued.
 */
gdpa_status_t gdpa_fwd(const void* q, const void* k, const void* v, const int32_t* q_offsets,
                       const int32_t* kv_offsets, int B, int H, int D, int act, int window_blocks,
                       float scale, void* out, void* stream);

/*
 * gdpa_fwd_async -- the whole forward pass, fully asynchronous: the caller
 * passes the offsets twice, as HOST arrays (h_*, read during the call to plan
 * the work list; the caller may reuse them once the call returns) and as
 * DEVICE arrays (read by the kernel, same values).  Planning runs on the
 * calling thread while earlier work on `stream` is still executing; the work
 * list goes up through a library-owned pinned buffer.  No synchronisation.
 */
gdpa_status_t gdpa_fwd_async(const void* q, const void* k, const void* v, const int32_t* h_q_offsets,
                             const int32_t* h_kv_offsets, const int32_t* q_offsets, const int32_t* kv_offsets,
                             int B, int H, int D, int act, int window_blocks, float scale, void* out,
                             void* stream);

/*
 * gdpa_fwd_lse -- gdpa_fwd_async that also keeps, for the backward pass, the
 * row logsumexp of every softmax query row: lse[t * H + h] =
 * ln sum_j exp(scale <q_t, k_j>) over the row's key set (natural log; -inf
 * for a row whose sequence has no keys).  lse: device fp32 [Tq, H], 4-byte
 * aligned, written in full for softmax and not touched for GELU (may be
 * NULL then).  Every other argument, layout and result as gdpa_fwd_async.
 * The row logsumexp is the quantity the backward needs to rebuild the
 * softmax weights tile by tile (techfeed summary of "GEM Training", JFA
 * section: the forward of a training step feeds its backward).
 */
gdpa_status_t gdpa_fwd_lse(const void* q, const void* k, const void* v, const int32_t* h_q_offsets,
                           const int32_t* h_kv_offsets, const int32_t* q_offsets, const int32_t* kv_offsets, int B,
                           int H, int D, int act, int window_blocks, float scale, void* out, float* lse,
                           void* stream);

/*
 * gdpa_fwd_sliding -- the forward with a causal sliding window of
 * window_tokens tokens instead of block windows: query i of a sequence sees
 * the keys i - window_tokens < j <= i of its own sequence (the token-granular
 * window the BlockAttention section of the techfeed summary of "GEM
 * Training" names as the step before block-aligned attention).  Softmax only
 * (GDPA_ERR_UNSUPPORTED for GELU), self attention (q and kv offsets equal),
 * window_tokens >= 1.  lse: optional (may be NULL) device fp32 [Tq, H], as
 * gdpa_fwd_lse.  Offsets twice (host and device) and everything else as
 * gdpa_fwd_async; asynchronous on `stream`.
 */
gdpa_status_t gdpa_fwd_sliding(const void* q, const void* k, const void* v, const int32_t* h_q_offsets,
                               const int32_t* h_kv_offsets, const int32_t* q_offsets, const int32_t* kv_offsets,
                               int B, int H, int D, int act, int window_tokens, float scale, void* out, float* lse,
                               void* stream);

/*
 * gdpa_fwd_mx -- the forward (full attention) with q and k in MXFP8, the
 * microscaling FP8 format the techfeed summary of "GEM Training" (section on
 * MXFP8 ultra-low-precision training) and the aigeeknews translation
 * (compute-efficiency section, "MXFP8 attention") apply to attention:
 *
 *   q8, k8  uint8 [T, H, D]     OCP e4m3 element codes ("E4M3FN": no
 *                               infinities, S.1111.111 NaN)
 *   q_sf, k_sf uint8 [T, H, D/32]  OCP E8M0 scale codes, 2^(e - 127): code b
 *                               of a (token, head) row scales its elements
 *                               [32 b, 32 b + 32)
 *   q_id = e4m3(q8_id) * 2^(q_sf_i,floor(d/32) - 127), k likewise
 *
 * The score product runs on the block-scaled e4m3 tensor-core MMA with fp32
 * accumulation; v and out stay bf16, and everything after the scores is
 * gdpa_fwd_lse's (softmax, GELU or SiLU; lse optional, may be NULL).  D must
 * be 128 (GDPA_ERR_UNSUPPORTED otherwise), no windows.  q8, k8, v and out
 * 16-byte aligned, q_sf and k_sf 4-byte aligned (each row's four codes are
 * read as one 32-bit word).  Offsets twice (host and device) as
 * gdpa_fwd_async; asynchronous on `stream`.  The buffers stay the caller's.
 */
gdpa_status_t gdpa_fwd_mx(const void* q8, const void* q_sf, const void* k8, const void* k_sf, const void* v,
                          const int32_t* h_q_offsets, const int32_t* h_kv_offsets, const int32_t* q_offsets,
                          const int32_t* kv_offsets, int B, int H, int D, int act, float scale, void* out, float* lse,
                          void* stream);

/*
 * gdpa_fwd_mxfp8 -- the forward (full attention, softmax) with q, k and v
 * all in MXFP8, both products on the block-scaled e4m3 tensor-core MMA (same
 * sources as gdpa_fwd_mx).  q8, q_sf, k8, k_sf as gdpa_fwd_mx; v is
 * quantised along the contraction of the P V product, the keys, so it
 * arrives key-major:
 *
 *   vt8    uint8 [H*D, VT]      e4m3 codes; row h*D + d holds coordinate d
 *                               of head h for every key: sequence b's keys
 *                               at columns [P_b, P_b + Lkv_b),
 *                               P_b = 32 * sum_{b' < b} ceil(Lkv_b' / 32),
 *                               VT = P_B; the columns [P_b + Lkv_b, P_{b+1})
 *                               must hold finite codes (zero)
 *   vt_sf  uint8 [VT/32, H*D]   E8M0 scales: byte [c, h*D + d] scales
 *                               columns [32 c, 32 c + 32) of row h*D + d
 *   v_jd = e4m3(vt8[h*D + d, P_b + j]) * 2^(vt_sf[(P_b + j) / 32, h*D + d] - 127)
 *
 * The weights P_ij (exp2 of the scaled scores less the row's running
 * maximum) are rounded on chip to e4m3 with one E8M0 scale per 32 keys of a
 * row -- the scale puts the block's largest weight just under 448, so no
 * code saturates -- and the row sum takes the unrounded weights.  D must be
 * 128 and act GDPA_ACT_SOFTMAX (GDPA_ERR_UNSUPPORTED otherwise).  q8, k8,
 * vt8 and out 16-byte aligned; q_sf, k_sf 4-byte aligned; vt_sf any.  lse
 * optional (may be NULL).  Offsets twice (host and device) as
 * gdpa_fwd_async; the host copy also fixes VT.  Asynchronous on `stream`;
 * the buffers stay the caller's.
 */
gdpa_status_t gdpa_fwd_mxfp8(const void* q8, const void* q_sf, const void* k8, const void* k_sf, const void* vt8,
                             const void* vt_sf, const int32_t* h_q_offsets, const int32_t* h_kv_offsets,
                             const int32_t* q_offsets, const int32_t* kv_offsets, int B, int H, int D, int act,
                             float scale, void* out, float* lse, void* stream);

/*
 * gdpa_bwd -- gradients of the forward for an upstream gradient dout:
 *   dq = dL/dq, dk = dL/dk, dv = dL/dv for L = sum(dout * out), computed by
 * the chain rule of the forward's definition (techfeed summary of "GEM
 * Training", JFA section: a backward over batch x heads without atomics):
 *   softmax: P_ij = exp(scale <q_i,k_j> - lse_i), dS_ij = P_ij (<dO_i,v_j> - <dO_i,o_i>)
 *   GELU:    P_ij = gelu(scale <q_i,k_j>) / Lkv,  dS_ij = gelu'(...) <dO_i,v_j> / Lkv
 *   dv_j = sum_i P_ij dO_i,  dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i
 * q, k, v, out, dout: device bf16 [tokens, H, D] (out and lse from
 * gdpa_fwd_lse on the same inputs); lse: device fp32 [Tq, H] (softmax only;
 * may be NULL for GELU); offsets twice, host (h_*, read during the call) and
 * device, as gdpa_fwd_async; dq: device bf16 [Tq, H, D]; dk, dv: device bf16
 * [Tkv, H, D]; all written in full (keys no query sees get zero gradients).
 * Tensors 16-byte aligned.  window_blocks > 0 (block windows, softmax, self
 * attention) as in the forward: each query row's gradient runs over its
 * window only.  Asynchronous on `stream`; the library keeps a
 * grow-only device buffer for the work lists and 8 Tq H bytes of scratch.
 * Errors as gdpa_fwd (a wait that runs out shows in gdpa_device_status).
 */
gdpa_status_t gdpa_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                       const float* lse, const int32_t* h_q_offsets, const int32_t* h_kv_offsets,
                       const int32_t* q_offsets, const int32_t* kv_offsets, int B, int H, int D, int act,
                       int window_blocks, float scale, void* dq, void* dk, void* dv, void* stream);

/*
 * gdpa_bwd_sliding -- gdpa_bwd for the causal sliding window of
 * window_tokens tokens (the forward of gdpa_fwd_sliding, whose out and lse
 * it takes).  Softmax only, self attention, window_tokens >= 1; everything
 * else as gdpa_bwd.
 */
gdpa_status_t gdpa_bwd_sliding(const void* q, const void* k, const void* v, const void* out, const void* dout,
                               const float* lse, const int32_t* h_q_offsets, const int32_t* h_kv_offsets,
                               const int32_t* q_offsets, const int32_t* kv_offsets, int B, int H, int D, int act,
                               int window_tokens, float scale, void* dq, void* dk, void* dv, void* stream);

/*
 * gdpa_fwd_noalloc -- gdpa_fwd for callers that must not allocate memory.
 * The pages describe no such entry point; it exists for users of this
 * library.  Some callers cannot allocate where they run attention: a serving
 * process that splits all device memory into a fixed arena at start-up and
 * forbids allocation on its request path, or a framework hook that must not
 * go around its own caching allocator.  This call allocates nothing -- no
 * cudaMalloc, cudaFree, cudaMallocHost or other allocating routine -- on the
 * device or the host: the work list lives in a file-scope device array of
 * 4 MiB and is planned in fixed host arrays by the same planner gdpa_fwd
 * uses.
 * Arguments, layout and results are those of gdpa_fwd (device offsets; every
 * call copies them to the host and synchronises `stream`).  Limits: B <= 65536
 * sequences and at most 261632 work items (query tiles x heads, about 33M
 * query rows x heads); larger requests return GDPA_ERR_NO_MEMORY before any
 * GPU work.
 * First call on a device: it looks up the array's device address (with that
 * device current); make it before any stream capture.  With CUDA's lazy
 * module loading (the default), the driver loads the array and the kernels
 * onto a device the first time they are used there, and that load reserves
 * device memory (the 4 MiB array and the kernels' code); a device holds them
 * from then until the process exits.  A caller that carves device memory
 * into an arena should therefore make one small call per device at start-up,
 * before carving it (or load modules eagerly, CUDA_MODULE_LOADING=EAGER).
 * Every call shares the array and the host arrays: calls are serialised on
 * the host, but two calls whose kernels overlap on the GPU (different
 * streams) race on the work list -- order them on one stream or synchronise
 * between them.  Each call rewrites the whole part of the array its launch
 * reads.
 */
gdpa_status_t gdpa_fwd_noalloc(const void* q, const void* k, const void* v, const int32_t* q_offsets,
                               const int32_t* kv_offsets, int B, int H, int D, int act, int window_blocks,
                               float scale, void* out, void* stream);

/*
 * gdpa_plan_create -- build a reusable plan from HOST offsets (the same
 * arrays the caller will later pass on the device).  Allocates the plan and
 * its device work list; *plan is NULL on failure.  Planning is host work:
 * tile enumeration plus longest-processing-time-first balancing over the SMs
 * of the current device.
 */
gdpa_status_t gdpa_plan_create(const int32_t* h_q_offsets, const int32_t* h_kv_offsets, int B, int H,
                               int D, int act, int window_blocks, gdpa_plan_t** plan);

/*
 * gdpa_plan_create_sliding -- the plan of gdpa_fwd_sliding (causal sliding
 * window of window_tokens >= 1 tokens; self attention: h_q_offsets and
 * h_kv_offsets equal; softmax).  Launch it with gdpa_fwd_planned.
 * GDPA_ERR_INVALID_ARG for window_tokens < 1, unequal offsets or another act.
 */
gdpa_status_t gdpa_plan_create_sliding(const int32_t* h_q_offsets, const int32_t* h_kv_offsets, int B, int H,
                                       int D, int act, int window_tokens, gdpa_plan_t** plan);

/*
 * gdpa_fwd_planned -- launch the forward pass with a plan; fully asynchronous
 * on `stream`.  The device offsets must hold the values the plan was built
 * from.  The kernels clip every work item to the rows of the tensors the plan
 * was built for, so offsets that reach past them never make the launch read
 * or write outside q, k, v or out; such a launch is flagged and
 * gdpa_device_status() then returns GDPA_ERR_INVALID_ARG (its output is
 * undefined).  Offsets that differ from the plan's but stay inside the
 * tensors are not detected: the output is then undefined.
 */
gdpa_status_t gdpa_fwd_planned(const gdpa_plan_t* plan, const void* q, const void* k, const void* v,
                               const int32_t* q_offsets, const int32_t* kv_offsets, float scale,
                               void* out, void* stream);

/* Frees the plan (synchronises the device if its buffers may be in use). */
void gdpa_plan_destroy(gdpa_plan_t* plan);

/* Number of work items / CTAs of a plan (for reporting); -1 on NULL. */
int64_t gdpa_plan_num_items(const gdpa_plan_t* plan);
int gdpa_plan_num_ctas(const gdpa_plan_t* plan);

/*
 * gdpa_fwd_host -- end-to-end call with HOST buffers: copies q, k, v and the
 * offsets to library-owned device buffers on `stream`, runs the forward pass
 * and copies `h_out` back, then synchronises `stream`.  Host buffers should be
 * pinned (page-locked) for full copy bandwidth.
 */
gdpa_status_t gdpa_fwd_host(const void* h_q, const void* h_k, const void* h_v, const int32_t* h_q_offsets,
                            const int32_t* h_kv_offsets, int B, int H, int D, int act, int window_blocks,
                            float scale, void* h_out, void* stream);

/*
 * gdpa_plan_enumerate -- the host planner alone, no GPU needed.  Fills
 * `items` (capacity `capacity`) grouped by CTA and `cta_begin` [num_ctas+1]
 * (items of CTA c are items[cta_begin[c] .. cta_begin[c+1])); `cost` (may be
 * NULL) receives each item's estimated cost; `rows_per_item` (may be NULL)
 * receives R; `kv_tile` (may be NULL) receives the keys per K/V tile the
 * kernel stages (64 for block windows and short key ranges on 256-row
 * items, else 128).  *n_items always receives the required count;
 * GDPA_ERR_NO_MEMORY if it exceeds `capacity`.
 */
gdpa_status_t gdpa_plan_enumerate(const int32_t* h_q_offsets, const int32_t* h_kv_offsets, int B, int H,
                                  int D, int act, int window_blocks, int num_ctas,
                                  gdpa_work_item_t* items, int64_t capacity, int32_t* cta_begin,
                                  int64_t* cost, int64_t* n_items, int32_t* rows_per_item, int32_t* kv_tile);

/*
 * gdpa_act_eval -- evaluates the kernel's device activation elementwise:
 * y[i] = gelu(x[i]) (act = GDPA_ACT_GELU_TANH) or y[i] = silu(x[i])
 * (act = GDPA_ACT_SILU) through the current route (gdpa_set_act_route),
 * or y[i] = 2^x[i] with the exponential the softmax path uses
 * (act = GDPA_ACT_SOFTMAX).  x, y: device fp32 [n].  For accuracy tests;
 * GDPA_ERR_INVALID_ARG for any other act.
 */
gdpa_status_t gdpa_act_eval(int act, const float* x, float* y, int64_t n, void* stream);

/*
 * gdpa_set_act_route -- selects the route (gdpa_act_route_t) every later
 * forward launch and gdpa_act_eval call of this process uses for the GELU and
 * SiLU sigma; launches already enqueued keep theirs.  Thread-safe (an atomic
 * word).  GDPA_ERR_INVALID_ARG for any other value (the route is unchanged).
 * gdpa_get_act_route returns the current one.
 */
gdpa_status_t gdpa_set_act_route(int route);
int gdpa_get_act_route(void);

/*
 * gdpa_device_status -- synchronises `stream`, then reads and clears the
 * device status word of the current device.  Returns GDPA_OK,
 * GDPA_ERR_DEVICE_TIMEOUT (a kernel gave up on a wait; its output is
 * undefined), GDPA_ERR_INVALID_ARG (a forward launch met device offsets past
 * its tensors, see gdpa_fwd_planned; its output is undefined) or
 * GDPA_ERR_CUDA.
 */
gdpa_status_t gdpa_device_status(void* stream);

/*
 * gdpa_wait_selftest -- launches one thread that waits, with the same
 * bounded mbarrier wait every role of the forward kernel uses, on a barrier
 * nothing ever arrives on.  After `timeout_ms` (1..10000) the wait gives up
 * and sets the device status word; gdpa_device_status() then returns
 * GDPA_ERR_DEVICE_TIMEOUT and the context stays usable.  For tests of the
 * failure path: no fault, trap or hang is involved.
 */
gdpa_status_t gdpa_wait_selftest(int timeout_ms, void* stream);

/* Human-readable name of a status code (static string). */
const char* gdpa_status_string(int status);

/* Library version, e.g. "gdpa 0.1 sm_103a". */
const char* gdpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDPA_H_ */
