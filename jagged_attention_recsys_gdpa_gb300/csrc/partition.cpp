// Host-side partitioning of one jagged batch over data-parallel ranks.
//
// Sequences (and heads) are independent problems, so a batch shards by
// sequence with no exchange inside attention. Work per sequence is its
// number of allowed (query, key) pairs, which varies by orders of magnitude
// across a jagged batch; the split balances that cost with the
// longest-processing-time-first greedy rule: sequences in order of
// decreasing cost (ties: lower index first) each go to the rank with the
// least cost so far (ties: lower rank). This is the sort-then-balance idea
// of the "Base Batch Shuffling" takeaway in the GEM training summary (sort
// by total length, pair the heaviest with the lightest) applied to
// attention cost instead of raw length.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/jattn.h"

namespace {

// Allowed pairs of one sequence for one head: the size of every query row's
// visible key interval (bottom-right aligned, delta = lkv - lq). The same
// rules as the kernels' masks: causal j <= i + delta; window W additionally
// i + delta - j < W; block W keeps the keys of the block holding i + delta.
int64_t sequence_pairs(int64_t lq, int64_t lkv, int mask, int64_t window) {
  if (lq <= 0 || lkv <= 0) return 0;
  const bool causal = mask & (JATTN_MASK_CAUSAL | JATTN_MASK_WINDOW);
  const bool win = mask & JATTN_MASK_WINDOW;
  const bool blk = mask & JATTN_MASK_BLOCK;
  const int64_t delta = lkv - lq;
  int64_t total = 0;
  for (int64_t i = 0; i < lq; ++i) {
    const int64_t pos = i + delta;
    int64_t lo = 0, hi = lkv;
    if (causal) hi = std::min(hi, pos + 1);
    if (win) lo = std::max(lo, pos - window + 1);
    if (blk) {
      const int64_t b0 = (pos >= 0 ? pos / window : -((window - 1 - pos) / window)) * window;
      lo = std::max(lo, b0);
      hi = std::min(hi, b0 + window);
    }
    if (hi > lo) total += hi - lo;
  }
  return total;
}

bool valid_offsets(int64_t B, const int64_t* off) {
  if (off[0] != 0) return false;
  for (int64_t b = 0; b < B; ++b)
    if (off[b + 1] < off[b]) return false;
  return true;
}

}  // namespace

extern "C" int jattn_partition(int64_t B, const int64_t* q_off, const int64_t* kv_off, int mask, int window,
                               int n_ranks, int32_t* rank_of, int64_t* rank_pairs) {
  if (B < 1 || B >= (int64_t(1) << 31) || n_ranks < 1 || !q_off || !kv_off || !rank_of || !rank_pairs)
    return JATTN_ERR_INVALID;
  if (mask != JATTN_MASK_NONE && mask != JATTN_MASK_CAUSAL && mask != (JATTN_MASK_CAUSAL | JATTN_MASK_WINDOW) &&
      mask != JATTN_MASK_BLOCK && mask != (JATTN_MASK_CAUSAL | JATTN_MASK_BLOCK))
    return JATTN_ERR_INVALID;
  if ((mask & (JATTN_MASK_WINDOW | JATTN_MASK_BLOCK)) && window < 1) return JATTN_ERR_INVALID;
  if (!valid_offsets(B, q_off) || !valid_offsets(B, kv_off)) return JATTN_ERR_INVALID;
  std::vector<int64_t> cost(B);
  for (int64_t b = 0; b < B; ++b)
    cost[b] = sequence_pairs(q_off[b + 1] - q_off[b], kv_off[b + 1] - kv_off[b], mask, window);
  std::vector<int64_t> order(B);
  for (int64_t b = 0; b < B; ++b) order[b] = b;
  std::stable_sort(order.begin(), order.end(), [&](int64_t x, int64_t y) { return cost[x] > cost[y]; });
  for (int r = 0; r < n_ranks; ++r) rank_pairs[r] = 0;
  for (int64_t b : order) {
    int best = 0;
    for (int r = 1; r < n_ranks; ++r)
      if (rank_pairs[r] < rank_pairs[best]) best = r;
    rank_of[b] = best;
    rank_pairs[best] += cost[b];
  }
  return JATTN_OK;
}
