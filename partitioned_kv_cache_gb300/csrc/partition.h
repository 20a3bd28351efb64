// partition.h -- how one partitioned-attention launch shares out its work
// (host code only).
//
// "Reflex: Real-Time VLA Control through Streaming Inference", §III "Core
// formulas", Proposition A.1: softmax attention over a key set equals the
// merge of its parts, so the key sequence may be cut into any number of
// slices (splits) whose partials (m, l, O) are merged afterwards.  A launch
// runs (M-tiles x K/V heads) units, each cut into `splits` key slices times
// `dparts` shares of the output columns.  Up to kMaxClusterSplits splits of a
// unit form one thread-block cluster and merge on chip; more are merged by a
// second kernel.
#pragma once

namespace rx {

constexpr int kMaxClusterSplits = 16;   // splits merged on chip through a cluster

// Relative cost of one launch, in units of about 0.7 us on GB300: each key
// tile of the longest split costs 1 + 0.2/dparts (the K tile, the S tile
// and the softmax chain are the same for every column share; only the V
// bytes and the P V product shrink), and a cluster merge costs 3/dparts for
// the partials' exchange through L2 plus 2.5 for its barrier and combine.
// Fitted to timings of 2163- and 8448-key suffixes and the shared-cache batch
// (12 x 2, 16 x 1 and 16 x 1 win there).  Ties go to more splits: the longest
// split is as long, but the average one is shorter (8448 keys: 16 x 1 is
// 0.4 us faster than 15 x 1; the batch: 16 x 1 0.3 us faster than 14 x 1).
inline double split_cost(int t_max, int splits, int dparts) {
  const int tiles = (t_max + splits - 1) / splits;
  double c = tiles * (1.0 + 0.2 / dparts);
  if (splits > 1) c += 3.0 / dparts + 2.5;
  return c;
}

// The same units for more splits than one cluster, merged by a combine
// kernel after the grid: 1.2 a key tile of the longest split plus 7.3 for the
// exchange, the second launch and its combine.  Fitted to 2163-, 4352-,
// 6400- and 8448-key suffixes: the unclustered merge won wherever the
// cluster left 5 or more tiles per split (8448 keys: 13.55 against 15.12 us;
// 4352: 11.04 against 11.42 us) and lost at 3 (c3 and the shared-cache
// batch: 9.09 against 8.82 us, 11.23 against 11.12 us).
inline double split_cost_unclustered(int t_max, int splits) {
  const int tiles = (t_max + splits - 1) / splits;
  return tiles * 1.2 + 7.3;
}

struct PartitionRequest {
  int t_max;           // key tiles (64 keys) of the longest query segment
  int units;           // M-tiles x K/V heads
  int D;               // head dimension (64, 128 or 256)
  int num_sms;
  int max_splits;      // splits the exchange workspace holds
  int forced_splits;   // 0 = automatic
  int forced_dparts;   // 0 = automatic, else 1, 2 or 4
  const int* cap;      // [kMaxClusterSplits + 1]: clusters of c CTAs the device holds at once
};

struct PartitionChoice {
  int splits;
  int dparts;
  bool fused;          // the splits of a unit form one cluster and merge on chip
};

// The automatic choice minimises split_cost over the partitions whose
// clusters all fit on the device at once (one wave), then compares one
// unclustered candidate: the splits that keep the grid within three quarters
// of the SMs, reduced to the fewest with the same longest split.  Forced
// values are kept (splits are clamped to [1, min(t_max, max_splits)]).
// Returns false for a column split that is not 1, 2 or 4 or does not divide D
// into 64-column blocks.
inline bool choose_partition(const PartitionRequest& r, PartitionChoice* out) {
  const int units = r.units > 0 ? r.units : 1;
  // A cluster merge exchanges its partials through the workspace, which
  // holds at most max_splits of them.
  auto fits = [&](int sp, int dp) {
    if (sp == 1) return units * dp <= r.num_sms;
    return sp <= kMaxClusterSplits && sp <= r.max_splits && units * dp <= r.cap[sp];
  };
  int splits = r.forced_splits > 0 ? r.forced_splits : 0;
  int dparts = r.forced_dparts > 0 ? r.forced_dparts : 0;
  if (splits == 0 || dparts == 0) {
    double best = 1e30;
    int bs = 1, bd = 1;
    const int s_hi = r.t_max < kMaxClusterSplits ? r.t_max : kMaxClusterSplits;
    for (int sp = 1; sp <= s_hi; ++sp) {
      if (splits > 0 && sp != splits) continue;
      for (int dp = 1; dp <= 4; dp *= 2) {
        if (dparts > 0 && dp != dparts) continue;
        if (r.D / dp < 64 || !fits(sp, dp)) continue;
        const double c = split_cost(r.t_max, sp, dp);
        if (c < best - 1e-9 || (c < best + 1e-9 && sp > bs)) {
          best = c;
          bs = sp;
          bd = dp;
        }
      }
    }
    int sp_nf = r.t_max < r.max_splits ? r.t_max : r.max_splits;
    const int sp_cap = 3 * r.num_sms / 4 / units;
    sp_nf = sp_nf < sp_cap ? sp_nf : sp_cap;
    // The fewest splits whose longest one is as short: every extra split
    // adds a CTA's Q load and a partial to merge (8448 keys: 27 splits of at
    // most 5 tiles 12.00 us, 28 12.22 us).
    if (sp_nf >= 1) {
      const int longest = (r.t_max + sp_nf - 1) / sp_nf;
      sp_nf = (r.t_max + longest - 1) / longest;
    }
    if (sp_nf > kMaxClusterSplits && (splits == 0 || splits == sp_nf) && dparts <= 1) {
      const double c = split_cost_unclustered(r.t_max, sp_nf);
      if (c < best - 1e-9) {
        best = c;
        bs = sp_nf;
        bd = 1;
      }
    }
    if (splits == 0) splits = bs;
    if (dparts == 0) dparts = bd;
  }
  splits = splits > r.t_max ? r.t_max : splits;
  splits = splits > r.max_splits ? r.max_splits : splits;
  splits = splits < 1 ? 1 : splits;
  if (dparts != 1 && dparts != 2 && dparts != 4) return false;
  if (r.D % (dparts * 64) != 0) return false;
  out->splits = splits;
  out->dparts = dparts;
  out->fused = splits >= 2 && splits <= kMaxClusterSplits && r.cap[splits] >= 1;
  return true;
}

}  // namespace rx
