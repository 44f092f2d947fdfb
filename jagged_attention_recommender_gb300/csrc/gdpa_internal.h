// gdpa_internal.h -- declarations shared by the host side of libgdpa
// (planner, API layer, kernel launchers).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <vector>

#include "../../include/gdpa.h"

namespace gdpa {

constexpr int kBlockM = 128;      // query rows per work item (one tcgen05 M=128 tile)
constexpr int kBlockN = 128;      // keys per K/V tile
constexpr int kWindowBlock = 64;  // block size of the block-aligned window
constexpr int kKeySplitRows = 32; // query rows of a key-split item

inline gdpa_status_t validate_shape(int B, int H, int D, int act, int window_blocks) {
  if (B < 0 || H <= 0 || window_blocks < 0) return GDPA_ERR_INVALID_ARG;
  if (act != GDPA_ACT_SOFTMAX && act != GDPA_ACT_GELU_TANH && act != GDPA_ACT_SILU) return GDPA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return GDPA_ERR_UNSUPPORTED;
  if (window_blocks > 0 && act != GDPA_ACT_SOFTMAX) return GDPA_ERR_UNSUPPORTED;
  if ((int64_t)H * D > (1 << 20)) return GDPA_ERR_UNSUPPORTED;
  return GDPA_OK;
}

gdpa_status_t validate_offsets(const int32_t* q_off, const int32_t* kv_off, int B, int window_blocks,
                               int64_t* Tq, int64_t* Tkv);

// Query rows per work item, chosen per batch:
//   window                                   256 (two 128-row tiles whose
//                                            windows overlap)
//   D = 64, every sequence <= 32 queries     32 (key split: the four
//                                            activation warps share the
//                                            queries and split each tile)
//   sequences average > 128 queries          256 (two 128-row tiles sharing
//                                            every K/V tile)
//   otherwise                                128
int choose_rows_per_item(const int32_t* q_off, int B, int D, int window_blocks);

// Keys per K/V tile for 256-row items: 64 (the scores double-buffered, so
// the next tile's S is computed while the current one is activated; block
// windows, whose 64-key blocks become whole tiles, and key ranges averaging
// at most kShortRange keys) or 128 (long key ranges, where the wider tile
// halves the per-tile overheads).  128 for every other item shape.
constexpr int kShortRange = 256;
int choose_kv_tile(const int32_t* q_off, const int32_t* kv_off, int B, int window_blocks, int rows_per_item);

// First key of the window of a query tile starting at q0: window_blocks > 0
// is a block window of that many 64-token blocks, window_blocks < 0 (internal
// only, gdpa_fwd_sliding) a causal sliding window of -window_blocks tokens,
// whose first key is rounded down to its 64-key tile.
int64_t window_start(int64_t q0, int window_blocks);

// Planner cost of an item (units of key columns of a 128-row tile).
int64_t plan_item_cost(int64_t q0, int64_t Lq, int64_t Lkv, int window_blocks, int rows_per_item);

// Number of work items plan_items will emit.
int64_t count_plan_items(const int32_t* q_off, int B, int H, int rows_per_item);

// Working storage of one planning pass, all of it owned by the caller:
// `cap_items` entries in each per-item array, `cap_buckets` counting-sort
// cursors (the planner falls back to an in-place sort of `keys` when the
// costs need more), and `max_leaves` >= the CTA count rounded up to a power
// of two entries in `load` (2 * max_leaves in `tree`, num_ctas in `count`).
struct PlanStorage {
  gdpa_work_item_t* items;
  int64_t* cost;
  uint32_t* order;
  int32_t* owner;
  uint64_t* keys;
  uint32_t* bucket;
  int64_t* load;
  int32_t* tree;
  int32_t* count;
  int64_t cap_items;
  int64_t cap_buckets;
  int max_leaves;
};

// The planner: enumerates the items, orders them by decreasing cost and
// assigns each to the least-loaded CTA.  Writes *n_out items to items_out
// grouped by CTA (decreasing cost within a CTA), cta_begin[num_ctas + 1] and,
// if cost_out is not null, each item's cost.  Allocates nothing;
// GDPA_ERR_NO_MEMORY if the storage is too small.
gdpa_status_t plan_items_into(const int32_t* q_off, const int32_t* kv_off, int B, int H, int window_blocks,
                              int rows_per_item, int num_ctas, const PlanStorage& st, gdpa_work_item_t* items_out,
                              int32_t* cta_begin, int64_t* cost_out, int64_t* n_out);

// plan_items_into over storage it allocates (std::vector; may throw bad_alloc).
gdpa_status_t plan_items(const int32_t* q_off, const int32_t* kv_off, int B, int H, int window_blocks,
                         int rows_per_item, int num_ctas, std::vector<gdpa_work_item_t>& items,
                         std::vector<int32_t>& cta_begin, std::vector<int64_t>* cost);

// Everything one launch of the forward kernel needs besides the tensor maps.
struct LaunchArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const int32_t* q_off;   // device
  const int32_t* kv_off;  // device
  const gdpa_work_item_t* items;  // device, grouped by CTA
  const int32_t* cta_begin;       // device [num_ctas + 1]
  int num_ctas;
  int rows_per_item;      // 128: one query tile per item; 256: two; 32: key split
  int kv_tile;            // keys per K/V tile (64 or 128, see choose_kv_tile)
  int64_t Tq, Tkv;
  int H, D, act, window_blocks;
  float scale;
  void* stream;
  float* lse = nullptr;   // optional: softmax row logsumexp [Tq, H]
  // MXFP8 Q and K: q, k hold e4m3 codes [T, H, D] and these the E8M0 scale
  // words [T, H] (4 codes each); full attention, D = 128, single-tile items
  const void* q_sf = nullptr;
  const void* k_sf = nullptr;
  // MXFP8 V as well (q_sf, k_sf set too): v holds the key-major codes
  // [H*D, VT], these its scales [VT/32, H*D] and each sequence's first
  // column (device, [B+1]); 256-row items, 64-key tiles, softmax
  const void* vt_sf = nullptr;
  const int32_t* vt_col = nullptr;
  int64_t VT = 0;
};

// Backward launch: work lists of int4 {sequence, head, first row, 0} on the
// device (dq: 128-row query tiles; dkdv: 128-key tiles), scratch [Tq, H]
// fp32 x 2 (log2-domain lse, then Dv).
struct BwdLaunchArgs {
  const void *q, *k, *v, *out, *dout;
  const float* lse;
  const int32_t* q_off;   // device
  const int32_t* kv_off;  // device
  const void* dq_items;
  int64_t n_dq;
  const void* kv_items;
  int64_t n_kv;
  float* scratch;
  void *dq, *dk, *dv;
  int64_t Tq, Tkv;
  int H, D, act;
  int window;             // 0 full; > 0 block window (blocks); < 0 sliding window (-tokens)
  float scale;
  void* stream;
};

// Defined in gdpa_kernels.cu.
gdpa_status_t launch_forward(const LaunchArgs& a);
// Defined in gdpa_bwd.cu.
gdpa_status_t launch_backward(const BwdLaunchArgs& a);
// Backward work lists (host): query tiles ordered by their key count, key
// tiles by their query count, longest first.
void plan_backward(const int32_t* q_off, const int32_t* kv_off, int B, int H, std::vector<int32_t>& dq_items,
                   std::vector<int32_t>& kv_items);
gdpa_status_t launch_act_eval(int act, const float* x, float* y, int64_t n, void* stream);
// The process-wide sigma route of the ALU activations (GDPA_ROUTE_*), read
// by every forward launch and act_eval call.  Defined in gdpa_kernels.cu.
int act_route();
void set_act_route(int route);

// Failure-path tests only: true while the environment variable
// GDPA_FAULT_INJECT names `what` ("alloc": the library's buffer growth fails
// as if the allocator were out of memory; "skip_arrive": in the 128-key pair
// kernel one activation warp of CTA 0 withholds its arrival on the first
// item's O-free barrier, so the MMA warp's bounded wait runs out and the
// launch takes its drain path).  Read on every call, so a test can set and
// clear it between calls; unset, nothing changes.
bool fault_injected(const char* what);
gdpa_status_t read_and_clear_device_status(void* stream);
gdpa_status_t launch_wait_selftest(int timeout_ms, void* stream);

}  // namespace gdpa
