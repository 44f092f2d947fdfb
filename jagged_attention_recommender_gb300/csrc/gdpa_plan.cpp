// gdpa_plan.cpp -- host-side jagged tile planner.
//
// GDPA section of the techfeed summary of "GEM Training" (jagged tile
// scheduling): the valid tiles are worked out on the CPU ahead of the launch,
// empty tiles are never emitted, and the tiles are spread over the SMs so
// that one long sequence cannot leave most SMs idle.  The pages balance with
// a zigzag SM assignment; this planner uses longest-processing-time-first
// (LPT) list scheduling over a min-heap of per-CTA loads, which bounds the
// finish time by 4/3 of optimal and subsumes the zigzag order.
//
// Work unit (chosen per batch by choose_rows_per_item): 32, 128
// or 256 query rows of one (sequence, head) against its key range:
//   full attention : keys [0, Lkv)
//   block window W : keys [64 * max(0, q0/64 - (W-1)), min(L, q0 + rows)),
//                    each 128-row tile of a 256-row item attending to its
//                    own window inside that range
// Items whose key range is empty (Lkv = 0) are still emitted (cheap) because
// their output rows must be zero-filled.
#include "gdpa_internal.h"

#include <algorithm>
#include <climits>
#include <cstring>
#include <vector>

namespace gdpa {

gdpa_status_t validate_offsets(const int32_t* q_off, const int32_t* kv_off, int B, int window_blocks,
                               int64_t* Tq, int64_t* Tkv) {
  if (B < 0) return GDPA_ERR_INVALID_ARG;
  if (B == 0) {
    *Tq = 0;
    *Tkv = 0;
    return GDPA_OK;
  }
  if (!q_off || !kv_off) return GDPA_ERR_INVALID_ARG;
  if (q_off[0] != 0 || kv_off[0] != 0) return GDPA_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    if (q_off[b + 1] < q_off[b] || kv_off[b + 1] < kv_off[b]) return GDPA_ERR_INVALID_ARG;
    if (window_blocks != 0 && (q_off[b + 1] != kv_off[b + 1])) return GDPA_ERR_INVALID_ARG;
  }
  *Tq = q_off[B];
  *Tkv = kv_off[B];
  return GDPA_OK;
}

// Estimated cost of one item, in units of "key columns of a 128-row tile".
// A tile of n key columns costs its MMA + activation work (~n, padded to the
// 16-column MMA granule) plus a fixed part for the query-tile load and the
// epilogue store.
static int64_t item_cost(int64_t kv_len) {
  if (kv_len <= 0) return 8;
  return ((kv_len + 15) / 16) * 16 + 96;
}

int64_t window_start(int64_t q0, int window_blocks) {
  if (window_blocks < 0) {  // sliding window of W tokens, from the 64-key tile holding q0 - W + 1
    const int64_t lo = q0 + window_blocks + 1;
    return lo > 0 ? lo / kWindowBlock * kWindowBlock : 0;
  }
  const int64_t blk = q0 / kWindowBlock - (window_blocks - 1);
  return blk > 0 ? blk * kWindowBlock : 0;
}

// Cost of one item: each of its (one or two) 128-row query tiles pays for
// the keys it attends to -- the whole key range, or its own block window.
int64_t plan_item_cost(int64_t q0, int64_t Lq, int64_t Lkv, int window_blocks, int rows_per_item) {
  const int64_t tiles = std::max<int64_t>(1, std::min<int64_t>(rows_per_item, Lq - q0 + kBlockM - 1) / kBlockM);
  int64_t c = 0;
  for (int64_t x = 0; x < tiles; ++x) {
    const int64_t qt = q0 + kBlockM * x;
    int64_t lo = 0, hi = Lkv;
    if (window_blocks != 0) {
      lo = window_start(qt, window_blocks);
      hi = std::min<int64_t>(Lkv, qt + kBlockM);
    }
    c += item_cost(hi > lo ? hi - lo : 0);
  }
  return c;
}

int choose_rows_per_item(const int32_t* q_off, int B, int D, int window_blocks) {
  if (B <= 0) return kBlockM;
  if (window_blocks != 0) return 2 * kBlockM;  // both tiles share the overlapping windows' keys
  int64_t busy = 0, max_lq = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t lq = q_off[b + 1] - q_off[b];
    busy += lq > 0 ? 1 : 0;
    max_lq = std::max<int64_t>(max_lq, lq);
  }
  if (busy == 0) return kBlockM;
  if (D == 64 && max_lq <= kKeySplitRows) return kKeySplitRows;
  return q_off[B] > (int64_t)kBlockM * busy ? 2 * kBlockM : kBlockM;
}

int choose_kv_tile(const int32_t* q_off, const int32_t* kv_off, int B, int window_blocks, int rows_per_item) {
  if (rows_per_item != 2 * kBlockM) return kBlockN;
  if (window_blocks != 0) return kBlockN / 2;
  int64_t busy = 0, keys = 0;
  for (int b = 0; b < B; ++b)
    if (q_off[b + 1] > q_off[b]) {
      ++busy;
      keys += kv_off[b + 1] - kv_off[b];
    }
  return (busy > 0 && keys <= (int64_t)kShortRange * busy) ? kBlockN / 2 : kBlockN;
}

int64_t count_plan_items(const int32_t* q_off, int B, int H, int rows_per_item) {
  int64_t n = 0;
  for (int b = 0; b < B; ++b) n += (int64_t)((q_off[b + 1] - q_off[b] + rows_per_item - 1) / rows_per_item) * H;
  return n;
}

gdpa_status_t plan_items_into(const int32_t* q_off, const int32_t* kv_off, int B, int H, int window_blocks,
                              int rows_per_item, int num_ctas, const PlanStorage& st, gdpa_work_item_t* items_out,
                              int32_t* cta_begin, int64_t* cost_out, int64_t* n_out) {
  *n_out = 0;
  if (H <= 0 || num_ctas <= 0) return GDPA_ERR_INVALID_ARG;
  const bool ok_rows = rows_per_item == kBlockM || rows_per_item == 2 * kBlockM ||
                       (rows_per_item == kKeySplitRows && window_blocks == 0);
  if (!ok_rows) return GDPA_ERR_INVALID_ARG;
  int leaves = 1;
  while (leaves < num_ctas) leaves <<= 1;
  if (leaves > st.max_leaves) return GDPA_ERR_NO_MEMORY;
  int64_t n = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t Lq = q_off[b + 1] - q_off[b];
    const int64_t Lkv = kv_off[b + 1] - kv_off[b];
    for (int64_t q0 = 0; q0 < Lq; q0 += rows_per_item) {
      const int64_t kv0 = window_blocks != 0 ? window_start(q0, window_blocks) : 0;
      const int64_t c = plan_item_cost(q0, Lq, Lkv, window_blocks, rows_per_item);
      for (int h = 0; h < H; ++h) {
        if (n >= st.cap_items) return GDPA_ERR_NO_MEMORY;
        st.items[n] = gdpa_work_item_t{(int32_t)b, (int32_t)h, (int32_t)q0, (int32_t)kv0};
        st.cost[n] = c;
        ++n;
      }
    }
  }
  // LPT: order by decreasing cost, then give each item to the CTA with the
  // least load so far.  Costs are multiples of 16 (or the small constant of
  // an empty item), so the order is by cost/16, ties in sequence/head/tile
  // order: the tiles of one (sequence, head) land on different CTAs at about
  // the same time and share its K/V through L2.  A counting sort gives that
  // order in O(n) when the cursor array is large enough; otherwise an
  // in-place sort of (bucket, index) keys gives the same order.  The
  // least-loaded CTA comes from a tournament tree (min over a complete
  // binary tree of per-CTA loads), O(log #CTAs) per item.
  int64_t max_bucket = 0;
  for (int64_t i = 0; i < n; ++i) max_bucket = std::max<int64_t>(max_bucket, st.cost[i] >> 4);
  uint32_t* order = st.order;
  if (max_bucket + 2 <= st.cap_buckets) {
    uint32_t* start = st.bucket;
    std::fill(start, start + max_bucket + 2, 0u);
    for (int64_t i = 0; i < n; ++i) start[(size_t)(max_bucket - (st.cost[i] >> 4)) + 1]++;
    for (int64_t b = 1; b < max_bucket + 2; ++b) start[b] += start[b - 1];
    for (int64_t i = 0; i < n; ++i) order[start[(size_t)(max_bucket - (st.cost[i] >> 4))]++] = (uint32_t)i;
  } else {
    for (int64_t i = 0; i < n; ++i) {
      const uint64_t rank = (uint64_t)std::min<int64_t>(max_bucket - (st.cost[i] >> 4), 0x7FFFFFFF);
      st.keys[i] = (rank << 32) | (uint64_t)i;
    }
    std::sort(st.keys, st.keys + n);  // in place, no allocation
    for (int64_t i = 0; i < n; ++i) order[i] = (uint32_t)(st.keys[i] & 0xFFFFFFFFu);
  }
  int32_t* count = st.count;
  for (int c = 0; c < num_ctas; ++c) count[c] = 0;
  int64_t total = 0;
  for (int64_t i = 0; i < n && total < (int64_t(1) << 47); ++i) total += st.cost[i];
  if (n >= 2 * (int64_t)leaves && total < (int64_t(1) << 47)) {
    // Every load fits in 47 bits: node k of the tree holds the key
    // (load << 16 | cta) of the least-loaded CTA below it, so the smallest
    // key is the least load with ties to the lowest index, as in the general
    // form below.  An update walks up from the leaf with the new key in a
    // register and reads only the siblings, whose addresses do not depend on
    // the walk: one min per level on the dependent chain instead of two
    // indirect loads.  (The keys array is free once `order` is built.)
    uint64_t* key = st.keys;
    for (int c = 0; c < leaves; ++c) key[leaves + c] = c < num_ctas ? (uint64_t)c : UINT64_MAX;
    for (int k = leaves - 1; k >= 1; --k) key[k] = std::min(key[2 * k], key[2 * k + 1]);
    uint64_t top = key[1];  // the root, carried from one item to the next
    for (int64_t k = 0; k < n; ++k) {
      const uint32_t idx = order[k];
      const int32_t c = (int32_t)(top & 0xFFFFu);
      st.owner[idx] = c;
      count[c]++;
      uint64_t v = top + ((uint64_t)st.cost[idx] << 16);
      int node = leaves + c;
      key[node] = v;
      for (; node > 1; node >>= 1) {
        v = std::min(v, key[node ^ 1]);
        key[node >> 1] = v;
      }
      top = v;
    }
  } else {
    int64_t* load = st.load;
    int32_t* tree = st.tree;  // tree[k] = CTA with the least load below node k
    for (int c = 0; c < leaves; ++c) load[c] = c < num_ctas ? 0 : INT64_MAX;
    for (int c = 0; c < leaves; ++c) tree[leaves + c] = c;
    for (int k = leaves - 1; k >= 1; --k) {
      const int32_t a = tree[2 * k], b = tree[2 * k + 1];
      tree[k] = load[b] < load[a] ? b : a;
    }
    for (int64_t k = 0; k < n; ++k) {
      const uint32_t idx = order[k];
      const int32_t c = tree[1];
      st.owner[idx] = c;
      count[c]++;
      load[c] += st.cost[idx];
      for (int node = (leaves + c) >> 1; node >= 1; node >>= 1) {
        const int32_t a = tree[2 * node], b = tree[2 * node + 1];
        tree[node] = load[b] < load[a] ? b : a;
      }
    }
  }
  cta_begin[0] = 0;
  for (int c = 0; c < num_ctas; ++c) cta_begin[c + 1] = cta_begin[c] + count[c];
  for (int c = 0; c < num_ctas; ++c) count[c] = cta_begin[c];  // now the fill cursors
  for (int64_t k = 0; k < n; ++k) {  // within a CTA: decreasing cost (LPT order)
    const uint32_t idx = order[k];
    const int32_t pos = count[st.owner[idx]]++;
    items_out[pos] = st.items[idx];
    if (cost_out) cost_out[pos] = st.cost[idx];
  }
  *n_out = n;
  return GDPA_OK;
}

gdpa_status_t plan_items(const int32_t* q_off, const int32_t* kv_off, int B, int H, int window_blocks,
                         int rows_per_item, int num_ctas, std::vector<gdpa_work_item_t>& items_out,
                         std::vector<int32_t>& cta_begin, std::vector<int64_t>* cost_out) {
  if (H <= 0 || num_ctas <= 0) return GDPA_ERR_INVALID_ARG;
  const int64_t n = count_plan_items(q_off, B, H, rows_per_item);
  int leaves = 1;
  while (leaves < num_ctas) leaves <<= 1;
  std::vector<gdpa_work_item_t> items((size_t)n);
  std::vector<int64_t> cost((size_t)n);
  std::vector<uint32_t> order((size_t)n), bucket((size_t)(4 * n + 1026));
  std::vector<int32_t> owner((size_t)n), tree(2 * (size_t)leaves), count((size_t)num_ctas);
  std::vector<uint64_t> keys((size_t)n);
  std::vector<int64_t> load((size_t)leaves);
  PlanStorage st{items.data(), cost.data(), order.data(), owner.data(), keys.data(), bucket.data(),
                 load.data(), tree.data(), count.data(), n, (int64_t)bucket.size(), leaves};
  items_out.resize((size_t)n);
  cta_begin.assign((size_t)num_ctas + 1, 0);
  if (cost_out) cost_out->resize((size_t)n);
  int64_t got = 0;
  const gdpa_status_t r = plan_items_into(q_off, kv_off, B, H, window_blocks, rows_per_item, num_ctas, st,
                                          items_out.data(), cta_begin.data(), cost_out ? cost_out->data() : nullptr,
                                          &got);
  if (r != GDPA_OK) return r;
  return got == n ? GDPA_OK : GDPA_ERR_INVALID_ARG;
}

}  // namespace gdpa

extern "C" gdpa_status_t gdpa_plan_enumerate(const int32_t* h_q_offsets, const int32_t* h_kv_offsets, int B,
                                             int H, int D, int act, int window_blocks, int num_ctas,
                                             gdpa_work_item_t* items, int64_t capacity, int32_t* cta_begin,
                                             int64_t* cost, int64_t* n_items, int32_t* rows_per_item,
                                             int32_t* kv_tile) {
  if (n_items) *n_items = 0;
  gdpa_status_t st = gdpa::validate_shape(B, H, D, act, window_blocks);
  if (st != GDPA_OK) return st;
  if (num_ctas <= 0 || !n_items || (capacity > 0 && !items) || !cta_begin) return GDPA_ERR_INVALID_ARG;
  int64_t Tq = 0, Tkv = 0;
  st = gdpa::validate_offsets(h_q_offsets, h_kv_offsets, B, window_blocks, &Tq, &Tkv);
  if (st != GDPA_OK) return st;
  std::vector<gdpa_work_item_t> v;
  std::vector<int32_t> cb;
  std::vector<int64_t> c;
  const int rpi = gdpa::choose_rows_per_item(h_q_offsets, B, D, window_blocks);
  if (rows_per_item) *rows_per_item = rpi;
  if (kv_tile) *kv_tile = gdpa::choose_kv_tile(h_q_offsets, h_kv_offsets, B, window_blocks, rpi);
  try {
    st = gdpa::plan_items(h_q_offsets, h_kv_offsets, B, H, window_blocks, rpi, num_ctas, v, cb, &c);
  } catch (...) {
    return GDPA_ERR_NO_MEMORY;
  }
  if (st != GDPA_OK) return st;
  *n_items = (int64_t)v.size();
  if ((int64_t)v.size() > capacity) return GDPA_ERR_NO_MEMORY;
  if (!v.empty()) std::memcpy(items, v.data(), v.size() * sizeof(gdpa_work_item_t));
  std::memcpy(cta_begin, cb.data(), cb.size() * sizeof(int32_t));
  if (cost && !c.empty()) std::memcpy(cost, c.data(), c.size() * sizeof(int64_t));
  return GDPA_OK;
}

namespace gdpa {

// Backward work lists: every 128-row query tile (dq) and every 128-key tile
// (dk/dv) of every (sequence, head), as {sequence, head, first row, 0}.  A
// query tile's work grows with its sequence's key count and a key tile's with
// its query count, so each list is ordered longest first (the GPU hands the
// next CTA slot to the next item in order, a greedy longest-first schedule).
void plan_backward(const int32_t* q_off, const int32_t* kv_off, int B, int H, std::vector<int32_t>& dq_items,
                   std::vector<int32_t>& kv_items) {
  std::vector<int> by_keys(B), by_queries(B);
  for (int b = 0; b < B; ++b) by_keys[b] = by_queries[b] = b;
  std::stable_sort(by_keys.begin(), by_keys.end(),
                   [&](int a, int b) { return kv_off[a + 1] - kv_off[a] > kv_off[b + 1] - kv_off[b]; });
  std::stable_sort(by_queries.begin(), by_queries.end(),
                   [&](int a, int b) { return q_off[a + 1] - q_off[a] > q_off[b + 1] - q_off[b]; });
  dq_items.clear();
  kv_items.clear();
  for (int b : by_keys) {
    const int Lq = q_off[b + 1] - q_off[b];
    for (int h = 0; h < H; ++h)
      for (int q0 = 0; q0 < Lq; q0 += kBlockM) dq_items.insert(dq_items.end(), {b, h, q0, 0});
  }
  for (int b : by_queries) {
    const int Lkv = kv_off[b + 1] - kv_off[b];
    for (int h = 0; h < H; ++h)
      for (int k0 = 0; k0 < Lkv; k0 += kBlockN) kv_items.insert(kv_items.end(), {b, h, k0, 0});
  }
}

}  // namespace gdpa
