// Grid-size / tile-width selection by the analytic model of "Stream-K:
// Work-centric Parallel Decomposition for Dense Matrix-Matrix Multiplication
// on the GPU", App. A.1: the run time of a Stream-K launch is the run time
// of its slowest CTA, modelled as
//
//   t_CTA = a + c * (MAC iterations) + e * (tiles it stores)
//             + b * [it stores a partial tile] + d * (peers it accumulates)
//
// a: fixed per-CTA cost (launch, pipeline fill, last epilogue); b: writing
// a partial tile; c: one MAC iteration; d: reading and adding one peer's
// partial tile; e: one more tile epilogue. The page fits {a, b, c, d} per
// architecture, data type and tile by microbenchmark and prints no values;
// the constants below were fitted on a GB300 (152 SMs, bf16, BLK_K = 64)
// from in-kernel %globaltimer spans over 726 (shape, tile, schedule, g)
// launches (median relative error 2 % for BLK_N = 128, 6 % for 256). The
// per-tile term e is an addition to the page's four.
//
// The page uses the model to pick g; here it also picks the schedule (DP,
// basic SK, or two-tile SK + DP) and BLK_N: 256 or 128, and for GEMMs
// without ABFT also 64 (the small-tile configuration: half the operand
// bytes per MAC iteration and per partial tile, twice the tiles), the
// kernel ensemble the page's conclusion suggests for bandwidth-bound and
// small shapes.
#pragma once
#include <stdint.h>

#include <mutex>
#include <unordered_map>

#include "skg_sched.cuh"

namespace skg {

struct CostModel {
  double a, c, e, b, d;  // microseconds
};

// BLK_N = 64 was fitted against the 128-wide constants: in-kernel spans of
// 480 launches of each width (20 small and skinny shapes, three schedules,
// g from 4 to 152, back to back with the L2 flushed), scored by the spans
// of the plans the search then picks. Per MAC iteration it costs about what
// a 128-wide one does (the k-step is latency-bound at these sizes), so it
// wins only where the fixed cost and the tile count decide.
constexpr CostModel kModel64 = {2.15, 0.360, 0.11, 4.50, 0.80};
constexpr CostModel kModel128 = {2.64, 0.334, 0.17, 4.67, 1.03};
constexpr CostModel kModel256 = {3.47, 0.364, 0.00, 8.18, 1.73};

inline const CostModel& model_for(int bn) {
  return bn == 64 ? kModel64 : bn == 128 ? kModel128 : kModel256;
}

// A shared tile also costs each part about this many d-units per covering
// CTA (every part waits for every cover's flag and reads a slice of every
// cover's partial): fitted on the GB300 from deep-k launches split 16 and 32
// ways (9.4 and 13.9 us beyond the MAC iterations).
constexpr double kShareCoverCost = 0.27;

// Whether the tile starting at iteration ti of an evenly split region is
// reduced by its covering CTAs together (see Work::share_parts): at least
// share_min covering CTAs end in it, and its owner's range starts at ti
// unless bank2. Gives the number of those (parts) and of all covering CTAs
// (covers).
inline bool shared_tile(int64_t q, int r, int64_t ti, int64_t I, int share_min, bool bank2,
                        int& parts, int& covers) {
  const int owner = even_cta_of(q, r, ti);
  int64_t ob, oe;
  even_range(q, r, owner, ob, oe);
  if (ob != ti && !bank2) return false;
  const int last = even_cta_of(q, r, ti + I - 1);
  int64_t lb, le;
  even_range(q, r, last, lb, le);
  const int part_last = last - (le > ti + I ? 1 : 0);
  parts = part_last - owner + 1;
  covers = last - owner + 1;
  return parts >= share_min;
}

// Segment counts of CTA x in an evenly split region of `total` iterations;
// `fix` counts the partial tiles' worth of fixup reads. With `share`
// (launches without ABFT) a shared tile costs each of its parts one partial
// store and covers / parts partial tiles of reads instead of the owner
// reading every peer.
inline void region_counts(int64_t q, int r, int64_t total, int64_t I, int x, bool share,
                          int share_min, bool bank2, int64_t& iters, int64_t& tiles,
                          int64_t& partial, double& fix) {
  if (total <= 0) return;
  int64_t b, e;
  even_range(q, r, x, b, e);
  if (e <= b) return;
  iters += e - b;
  if (b % I != 0) partial += 1;
  const int64_t first = (b % I == 0) ? b : (b / I + 1) * I;
  int parts = 0, covers = 0;
  if (first < e) {
    const int64_t started = (e - 1 - first) / I + 1;
    tiles += started;
    const int64_t last = first + (started - 1) * I;
    if (last + I > e) {  // owns an unfinished tile
      if (share && shared_tile(q, r, last, I, share_min, bank2, parts, covers)) {
        partial += 1;
        fix += (double)covers / parts + kShareCoverCost * covers;
      } else {
        fix += even_cta_of(q, r, last + I - 1) - x;
      }
    }
  } else if (share && shared_tile(q, r, (b / I) * I, I, share_min, bank2, parts, covers)) {
    // The whole range lies inside a tile another CTA started and owns.
    fix += (double)covers / parts + kShareCoverCost * covers;
  }
}

// Predicted time (us) of one launch with schedule s: max over CTAs. O(g).
// Side-tile iterations (fused checksum GEMMs) are costed like output ones.
// `share`: the launch reduces shared tiles together (no ABFT).
inline double predict_us(const Schedule& s, const CostModel& M, bool share) {
  if (s.t == 0 || s.ipt == 0) return 0.0;
  const int64_t I = s.ipt;
  double worst = 0.0;
  for (int x = 0; x < s.g; ++x) {
    int64_t iters = 0, tiles = 0, partial = 0;
    double fix = 0.0;
    if (x < s.t_dp) {
      const int64_t nd = (s.t_dp - 1 - x) / s.g + 1;
      iters += nd * I;
      tiles += nd;
    }
    region_counts(s.sk_q, s.sk_r, s.sk_total, I, x, share, s.share_min, s.share_bank2 != 0, iters,
                  tiles, partial, fix);
    if (s.g_ck == 0)
      region_counts(s.ck_q, s.ck_r, s.ck_total, I, x, false, kShareMin, false, iters, tiles,
                    partial, fix);
    const double tx = M.a + M.c * (double)iters + M.e * (double)tiles + M.b * (double)partial +
                      M.d * fix;
    if (tx > worst) worst = tx;
  }
  for (int x = 0; x < s.g_ckt; ++x) {  // dedicated side CTAs: the side region split over them
    int64_t iters = 0, tiles = 0, partial = 0;
    double fix = 0.0;
    region_counts(s.ck_q, s.ck_r, s.ck_total, I, x, false, kShareMin, false, iters, tiles,
                  partial, fix);
    const double tx = M.a + M.c * (double)iters + M.e * (double)tiles + M.b * (double)partial +
                      M.d * fix;
    if (tx > worst) worst = tx;
  }
  return worst;
}

struct Plan {
  int bn, sched, grid;
  double us;
  int grid_ck;  // dedicated side CTAs launched after the grid ones
};

// Best (BLK_N, schedule, g) for an m x n x k launch on `sms` SMs. Fixed
// choices (want_* != 0 / >= 0) are kept; the rest are searched (BLK_N = 64
// only with `small_tiles`).
inline Plan search_plan(int64_t m, int64_t n, int64_t k, int want_bn, int want_sched,
                        int want_grid, int sms, int t_ck, bool side_ctas, bool share,
                        bool small_tiles) {
  static const int kCands[] = {1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 76, 96, 112, 128, 144};
  Plan best{want_bn ? want_bn : 256, want_sched >= 0 ? want_sched : kSchedSK2DP,
            want_grid ? want_grid : sms, 1e300, 0};
  for (int bn = 64; bn <= 256; bn *= 2) {
    if (want_bn ? bn != want_bn : (bn == 64 && !small_tiles)) continue;
    const CostModel& M = model_for(bn);
    const int64_t t = ((m + kTileM - 1) / kTileM) * ((n + bn - 1) / bn) + t_ck;
    int cands[64];
    int nc = 0;
    if (want_grid) {
      cands[nc++] = want_grid;
    } else {
      for (int c : kCands)
        if (c <= sms) cands[nc++] = c;
      cands[nc++] = sms;
      for (int w = 1; w <= 8 && nc < 64; ++w) {
        const int64_t g = (t + w - 1) / w;
        if (g >= 1 && g <= sms) cands[nc++] = (int)g;
      }
    }
    int scheds[3] = {kSchedDP, kSchedSK, kSchedSK2DP};
    int ns = 3;
    if (want_sched >= 0) {
      scheds[0] = want_sched;
      ns = 1;
    }
    for (int si = 0; si < ns; ++si) {
      const int sched = scheds[si];
      for (int i = 0; i < nc; ++i) {
        // Basic Stream-K keeps its tile-processing skew for the whole
        // launch, which costs cache reuse the model does not see (§5.2);
        // with two or more full waves the hybrids exist to bound it, so the
        // automatic choice does not take basic SK there. Measured on GB300,
        // the skew also loses from one full wave on when tiles are deep
        // (8192 x 1024 x 8192 on 76 clusters: basic SK 115 us, DP + one-tile
        // SK 92 us; at k = 4096 basic SK was still ahead by 3-4 %).
        const int64_t ipt = (k + kTileK - 1) / kTileK;
        if (want_sched < 0 && sched == kSchedSK &&
            (t >= 2 * (int64_t)cands[i] || (t >= cands[i] && ipt >= 128)))
          continue;
        // Side tiles split over the grid, or (automatic grid only) one each
        // on SMs the grid leaves idle: every verification waits for all side
        // tiles, so they must end with the output CTAs' first tiles.
        const int spare = (want_grid || !side_ctas) ? 0 : sms - cands[i];
        const int gck_opts[2] = {0, t_ck <= spare ? t_ck : 0};
        for (int oi = 0; oi < (gck_opts[1] > 0 ? 2 : 1); ++oi) {
          const int gck = gck_opts[oi];
          const Schedule s =
              make_schedule(m, n, k, kTileM, bn, kTileK, cands[i], sched, t_ck, gck);
          const double us = predict_us(s, M, share);
          // Prefer fewer CTAs on ties (less fixup storage and traffic).
          if (us < best.us - 1e-9 ||
              (us < best.us + 1e-9 && cands[i] + gck < best.grid + best.grid_ck)) {
            best = Plan{bn, sched, cands[i], us, gck};
          }
        }
      }
    }
  }
  return best;
}

// search_plan behind a small cache: the search walks up to ~150 candidate
// schedules of up to `sms` CTAs each, far more host time than a launch.
inline Plan choose_plan(int64_t m, int64_t n, int64_t k, int want_bn, int want_sched,
                        int want_grid, int sms, int t_ck = 0, bool side_ctas = true,
                        bool share = true, bool small_tiles = false) {
  struct Key {
    int64_t m, n, k;
    int bn, sched, grid, sms, t_ck, side, share, small;
    bool operator==(const Key& o) const {
      return m == o.m && n == o.n && k == o.k && bn == o.bn && sched == o.sched &&
             grid == o.grid && sms == o.sms && t_ck == o.t_ck && side == o.side &&
             share == o.share && small == o.small;
    }
  };
  struct Hash {
    size_t operator()(const Key& x) const {
      uint64_t h = 1469598103934665603ull;
      const int64_t v[11] = {x.m,    x.n,    x.k,    x.bn,    x.sched,
                             x.grid, x.sms,  x.t_ck, x.side, x.share, x.small};
      for (int64_t e : v) h = (h ^ (uint64_t)e) * 1099511628211ull;
      return (size_t)h;
    }
  };
  static std::mutex mu;
  static std::unordered_map<Key, Plan, Hash> cache;
  const Key key{m, n, k, want_bn, want_sched, want_grid, sms, t_ck, side_ctas ? 1 : 0,
                share ? 1 : 0, small_tiles ? 1 : 0};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const Plan p =
      search_plan(m, n, k, want_bn, want_sched, want_grid, sms, t_ck, side_ctas, share, small_tiles);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache.emplace(key, p);
  return p;
}

}  // namespace skg
