// Host side of the split schedule: which problems split, into how many
// pieces, and the workspace that takes.  The kernel side (units, partial
// results, the completion counter and the combine) is in attn_fwd.cuh.
#pragma once

#include <cstddef>
#include <mutex>
#include <vector>

#include "../../include/fp8attn.h"
#include "attn_fwd.cuh"

namespace {

// Split schedule: considered for problems with fewer than kSplitMaxWaves * SMs
// items, with a workspace of at most kSplitMaxBytes.
constexpr int kSplitMaxWaves = 4;
constexpr size_t kSplitMaxBytes = 128ull << 20;

// The paths whose codes or roundings allow a split (the others run whole items).
bool split_variant(int variant) {
  return variant == ATTN_VARIANT_LEANP || variant == ATTN_VARIANT_BLOCK_EXACT ||
         variant == ATTN_VARIANT_BF16;
}

// ---------------------------------------------------------------- split plan
struct SplitPlan {
  int split_qb = 0, ns = 1, n_split_items = 0;
  size_t ws_bytes = 0;
};

size_t split_ws_bytes(int n_split_items, int ns) {
  return fa8::split_cnt_bytes(n_split_items) +
         (size_t)n_split_items * ns * 2 * fa8::kSplitSlotFloats * sizeof(float);
}

// The plan model's costs (ns at about 2 GHz): per key tile of both query
// tiles, per unit (the item boundary), and per piece piece0 + piece_ns * ns
// (its partial result written, and the ns partial results read and added up
// by the last piece); and the smallest predicted gain, in percent, for which
// a split is taken.
struct SplitCosts {
  int step, unit, piece0, piece_ns, min_gain_pct;
  bool operator==(const SplitCosts& o) const {
    return step == o.step && unit == o.unit && piece0 == o.piece0 && piece_ns == o.piece_ns &&
           min_gain_pct == o.min_gain_pct;
  }
};

// Least-squares fits to GB300 times of forced plans.  FP8 (Lean-P, and
// block-exact alike): 103 plans on 2 to 16 heads, 2K to 8K keys, head dims 128
// and 192, within 8% of each with 5 us for the launch; the MLA shape's step
// is the head-dim-128 step scaled by its measured throughput.  BF16: 180
// plans on 1 to 16 heads, 1K to 16K keys, causal and not, within 7.4% of each
// with 3 us for the launch.  The model was fitted with the inputs in L2; with
// L2 flushed before every call it predicts too much gain, most at 2K keys.
// The thresholds are the smallest predicted gains above which every plan the
// model chose, over 75 shapes (1 to 16 heads, 1K to 16K keys, causal and
// not, GQA), ran at 99% or more of the whole-item speed with L2 flushed: 15%
// for FP8 (below it, losses of up to 7.5%), 8% for BF16.
SplitCosts split_costs(int variant, int Dqk) {
  if (variant == ATTN_VARIANT_BF16) return {1580, 6640, 5360, 1300, 8};
  return {Dqk == 192 ? 1140 : 950, 5000, 3000, 1000, 15};
}

// Estimated finishing time of the busiest CTA (ns) when the items of query
// block >= sq are split into ns pieces (ns = 1: no split), following the
// kernel's unit order and its alternating round-robin assignment (item_at).
long long split_makespan(int units_bh, int n_qblocks, int n_kv_tiles, int causal,
                         const SplitCosts& c, int sq, int ns, int grid,
                         std::vector<long long>& load) {
  const long long step = c.step, unit_cost = c.unit;
  const long long piece_cost = c.piece0 + (long long)c.piece_ns * ns;
  load.assign(grid, 0);
  long long pos = 0;
  auto place = [&](long long cost) {
    const long long round = pos / grid, k = pos % grid;
    const long long c = (round & 1) ? grid - 1 - k : k;
    load[c] += cost + unit_cost;
    ++pos;
  };
  auto nkv_of = [&](int qb) {
    const int need = 2 * qb + 2;
    return causal && need < n_kv_tiles ? need : n_kv_tiles;
  };
  if (ns > 1)
    for (int qb = n_qblocks - 1; qb >= sq; --qb) {
      const int n = nkv_of(qb);
      for (int u = 0; u < units_bh; ++u)
        for (int s = 0; s < ns; ++s)
          place(((long long)(s + 1) * n / ns - (long long)s * n / ns) * step + piece_cost);
    }
  for (int qb = (ns > 1 ? sq : n_qblocks) - 1; qb >= 0; --qb) {
    const long long n = nkv_of(qb);
    for (int u = 0; u < units_bh; ++u) place(n * step);
  }
  long long m = 0;
  for (long long x : load) m = x > m ? x : m;
  return m;
}

// The split schedule for a problem (none unless the model above predicts at
// least the path's minimum gain: smaller predicted gains are within the
// model's error).  Plans are cached: the search walks every candidate.
SplitPlan split_plan(int units_bh, int S, int causal, const SplitCosts& costs, int sms,
                     size_t limit) {
  SplitPlan best;
  const int n_qblocks = (S + 255) / 256, n_kv_tiles = (S + 127) / 128;
  const long long n_items = (long long)units_bh * n_qblocks;
  if (n_items >= (long long)kSplitMaxWaves * sms) return best;
  struct Entry {
    int units_bh, S, causal;
    SplitCosts costs;
    int sms;
    size_t limit;
    SplitPlan plan;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry& e : cache)
      if (e.units_bh == units_bh && e.S == S && e.causal == causal && e.costs == costs &&
          e.sms == sms && e.limit == limit)
        return e.plan;
  }
  std::vector<long long> load;
  const int grid0 = (int)(n_items < sms ? n_items : sms);
  const long long base =
      split_makespan(units_bh, n_qblocks, n_kv_tiles, causal, costs, 0, 1, grid0, load);
  long long best_t = base;
  for (int ns = 2; ns <= 4; ++ns)
    for (int sq = n_qblocks - 1; sq >= 0; --sq) {
      const int nkv_min = causal && 2 * sq + 2 < n_kv_tiles ? 2 * sq + 2 : n_kv_tiles;
      if (nkv_min < 2 * ns) break;  // every piece needs two key tiles
      const int n_split = units_bh * (n_qblocks - sq);
      const size_t bytes = split_ws_bytes(n_split, ns);
      if (bytes > limit) break;
      const long long n_units = n_items + (long long)n_split * (ns - 1);
      const int grid = (int)(n_units < sms ? n_units : sms);
      const long long t =
          split_makespan(units_bh, n_qblocks, n_kv_tiles, causal, costs, sq, ns, grid, load);
      if (t < best_t) {
        best_t = t;
        best.split_qb = sq;
        best.ns = ns;
        best.n_split_items = n_split;
        best.ws_bytes = bytes;
      }
    }
  if (best.n_split_items > 0 && best_t * (100 + costs.min_gain_pct) > base * 100)
    best = SplitPlan();
  std::lock_guard<std::mutex> lk(mu);
  if (cache.size() >= 64) cache.erase(cache.begin());
  cache.push_back({units_bh, S, causal, costs, sms, limit, best});
  return best;
}

}  // namespace
