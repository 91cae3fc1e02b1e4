// Stream-K schedule arithmetic, shared by the host-side schedule query and
// the persistent kernel (every role warp walks the same list).
//
// "Stream-K: Work-centric Parallel Decomposition for Dense Matrix-Matrix
// Multiplication on the GPU":
//   - Algorithm 5 (§4): the MAC iterations of all tiles form one linear
//     m -> n -> k space split over g CTAs; a CTA's range is cut at tile
//     boundaries into segments; tile_started / tile_ended give the role.
//   - §A1: iterations are split evenly, CTA counts differing by one at most: CTA x gets
//     q + [x < r] iterations starting at x*q + min(x, r), (q, r) = divmod(T, g).
//   - §5.2: "DP + one-tile SK" keeps w = floor(t/g) full DP waves; "two-tile
//     SK + DP" gives one of them up when w >= 2 so every Stream-K CTA holds
//     between one and two tiles of iterations. DP tiles are the first t_dp
//     output tiles, walked x, x+g, ...; the Stream-K region is the rest.
//   - Algorithm 3 (tile coordinates): the page numbers tiles row-major,
//     tile = tm * tiles_n + tn. Its conclusion names cache-aware tile orders
//     as future work; here tile indices are walked in bands of `band` tile
//     columns, row by row inside a band, so the CTAs of one wave share a few
//     columns of B and rows of A in L2. band >= tiles_n is the page's
//     row-major order. Only the index -> (tm, tn) map changes; the schedule
//     (which CTA runs which tile index and k-range) does not.
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define SKG_HD __host__ __device__ __forceinline__
#else
#define SKG_HD inline
#endif

namespace skg {

enum : int { kSchedDP = 0, kSchedSK = 1, kSchedDPSK1 = 2, kSchedSK2DP = 3, kSchedAuto = 4 };

// CTA tile rows (BLK_M) and MAC-iteration depth (BLK_K) of the kernel.
constexpr int kTileM = 128;
constexpr int kTileK = 64;
enum : int { kRoleFull = 0, kRoleOwner = 1, kRolePeer = 2 };

// Tiles of an output Stream-K region that this many covering CTAs end their
// ranges in, the k = 0 CTA's range starting at the tile, are reduced by all
// of those together in launches without ABFT (Work::share_parts): the
// default of Schedule::share_min.
constexpr int kShareMin = 8;

struct Schedule {
  int tiles_m, tiles_n;
  int ipt;            // MAC iterations per tile, ceil(k / BLK_K)
  int t;              // tiles (t_ck + tiles_m * tiles_n)
  int t_ck;           // leading tiles of fused side GEMMs (0 for a plain GEMM)
  int t_dp;           // data-parallel output tiles [t_ck, t_ck + t_dp)
  int g;              // persistent CTAs
  int64_t sk_total;   // Stream-K iterations of the output tiles after the DP ones
  int64_t sk_q;       // floor(sk_total / g)
  int sk_r;           // sk_total mod g
  int64_t ck_total;   // side-tile iterations, split over the g CTAs or, with
                      // g_ck > 0, over the first g_ckt dedicated side CTAs
  int64_t ck_q;       // floor(ck_total / (g_ck ? g_ckt : g))
  int ck_r;           // ck_total mod (g_ck ? g_ckt : g)
  int g_ck;           // dedicated side CTAs g .. g + g_ck - 1 (0: none)
  int g_ckt;          // of those, the ones that run side tiles (the others
                      // only take part in the in-kernel encode pass)
  int band;           // tile columns per raster band (tiles_n = row-major)
  // Shared reduction (launches without ABFT): a Stream-K tile that at least
  // share_min covering CTAs end their ranges in is reduced by all of those.
  // With share_bank2 the owner may also be a CTA whose range began in an
  // earlier tile (it already holds a partial there): its partial of the
  // shared tile and its flag then live in a second bank (the storage of the
  // otherwise unused second region).
  int share_min;
  int share_bank2;
  // Split reduction (launches without ABFT): a Stream-K tile that 2 ..
  // split_max covering CTAs end their ranges in (fewer than share_min) is
  // finished by those CTAs together, each owning a range of the tile's
  // columns: every one stores its partial, then folds the other covering
  // CTAs' partials of its columns into its own accumulator and stores them
  // (0 = off; needs share_bank2 when an owner began in an earlier tile).
  int split_max;
};

// Output-tile coordinates of tile index `tile` (>= t_ck) under the banded
// raster.
SKG_HD void tile_coords(const Schedule& s, int tile, int& tm, int& tn) {
  tile -= s.t_ck;
  const int per_band = s.band * s.tiles_m;
  const int b = tile / per_band;
  const int within = tile - b * per_band;
  const int rest = s.tiles_n - b * s.band;
  const int bw = rest < s.band ? rest : s.band;
  tm = within / bw;
  tn = b * s.band + within % bw;
}

SKG_HD int dp_tiles(int t, int g, int mode) {
  if (mode == kSchedDP) return t;
  if (mode == kSchedSK) return 0;
  const int w = t / g;
  if (t % g == 0) return t;
  if (mode == kSchedSK2DP && w >= 2) return (w - 1) * g;
  return w * g;  // DP + one-tile SK, and the two-tile hybrid when w < 2
}

// The page's schedule over the output tiles (DP tiles first, then the
// Stream-K region) on g CTAs, plus `t_ck` full-k side tiles (the fused ABFT
// checksum GEMMs) in a Stream-K region of their own (own partial slots and
// flags), its iterations split evenly either
//   - g_ck == 0: over the g CTAs, so every CTA starts with the same small
//     share of side work, whatever the schedule of the output tiles; or
//   - g_ck > 0: over g_ckt <= g_ck more CTAs that run nothing else, for
//     launches that leave SMs idle (g_ckt = t_ck gives one whole side tile
//     each); g_ckt < 0 means all g_ck.
SKG_HD Schedule make_schedule(int64_t m, int64_t n, int64_t k, int bm, int bn, int bk, int g,
                              int mode, int t_ck = 0, int g_ck = 0, int g_ckt = -1) {
  Schedule s;
  s.tiles_m = (int)((m + bm - 1) / bm);
  s.tiles_n = (int)((n + bn - 1) / bn);
  s.ipt = (int)((k + bk - 1) / bk);
  const int t_out = s.tiles_m * s.tiles_n;
  s.t_ck = t_out > 0 ? t_ck : 0;
  s.t = s.t_ck + t_out;
  s.g = g;
  s.t_dp = (t_out == 0 || s.ipt == 0) ? t_out : dp_tiles(t_out, g, mode);
  s.sk_total = (int64_t)(t_out - s.t_dp) * s.ipt;
  s.sk_q = s.sk_total / g;
  s.sk_r = (int)(s.sk_total % g);
  s.g_ck = s.t_ck > 0 ? g_ck : 0;
  s.g_ckt = (g_ckt < 0 || g_ckt > s.g_ck) ? s.g_ck : g_ckt;
  s.ck_total = (int64_t)s.t_ck * s.ipt;
  const int ck_ctas = s.g_ck > 0 ? s.g_ckt : g;
  s.ck_q = s.ck_total / ck_ctas;
  s.ck_r = (int)(s.ck_total % ck_ctas);
  s.band = s.tiles_n > 0 ? s.tiles_n : 1;
  s.share_min = kShareMin;
  s.share_bank2 = 0;
  s.split_max = 0;
  return s;
}

// [begin, end) of CTA x in an iteration space split evenly over the CTAs
// (q, r) = divmod(total, g).
SKG_HD void even_range(int64_t q, int r, int x, int64_t& begin, int64_t& end) {
  begin = (int64_t)x * q + (x < r ? x : r);
  end = begin + q + (x < r ? 1 : 0);
}

// CTA whose range holds iteration `it` of such a split.
SKG_HD int even_cta_of(int64_t q, int r, int64_t it) {
  const int64_t big = (int64_t)r * (q + 1);
  if (it < big) return (int)(it / (q + 1));
  return r + (int)((it - big) / q);
}

// [begin, end) of CTA x in the Stream-K iteration space (even split).
SKG_HD void sk_range(const Schedule& s, int x, int64_t& begin, int64_t& end) {
  even_range(s.sk_q, s.sk_r, x, begin, end);
}

// CTA whose Stream-K range holds iteration `it` (0 <= it < sk_total).
SKG_HD int sk_cta_of(const Schedule& s, int64_t it) { return even_cta_of(s.sk_q, s.sk_r, it); }

struct Work {
  int tile;
  int kb_begin, kb_end;  // MAC iterations within the tile
  int role;
  int peer_last;         // OWNER: last peer CTA (peers are cta+1 .. peer_last)
  int region;            // 0: output tiles, 1: side tiles (own partial slots and flags)
  // CTAs covering the tile: owner .. contrib_last; those up to part_last
  // end their ranges inside it (the tile is their last work in the region);
  // share_parts = part_last - owner + 1 of them. owner_bank2: the owner's
  // range began in an earlier tile, so it holds another partial in the
  // region (a shared reduction keeps its partial of this tile in bank 2).
  int owner, contrib_last, part_last, share_parts, owner_bank2;
};

// Walks one CTA's segments in execution order: its share of the side
// tiles, its DP tiles, then its Stream-K range; the split regions are cut
// at tile boundaries. A dedicated side CTA (x >= g) walks whole side tiles.
struct Cursor {
  int x;
  int next_dp;
  int ck_base;  // first CTA of the split side region (g for dedicated side CTAs)
  int64_t ck_it, ck_end;
  int64_t it, it_end;

  SKG_HD void init(const Schedule& s, int cta) {
    x = cta;
    next_dp = cta;
    ck_base = 0;
    it = it_end = ck_it = ck_end = 0;
    if (cta >= s.g) {
      // Dedicated side CTA: its share of the side region (the first g_ckt
      // of them), nothing else.
      next_dp = s.t_dp;
      ck_base = s.g;
      if (s.ck_total > 0 && cta - s.g < s.g_ckt)
        even_range(s.ck_q, s.ck_r, cta - s.g, ck_it, ck_end);
      return;
    }
    if (s.sk_total > 0) sk_range(s, cta, it, it_end);
    if (s.ck_total > 0 && s.g_ck == 0) even_range(s.ck_q, s.ck_r, cta, ck_it, ck_end);
  }

  // Next segment of a split region whose tiles start at `base`.
  // CTA indices of the split are cta_base + (index within the split).
  SKG_HD static void cut(const Schedule& s, int64_t q, int r, int base, int region, int x,
                         int cta_base, int64_t& pos, int64_t end, Work& w) {
    const int64_t tile_rel = pos / s.ipt;
    const int64_t tile_iter = tile_rel * s.ipt;
    const int64_t tile_iter_end = tile_iter + s.ipt;
    const bool started = (pos == tile_iter);
    const bool ended = (end >= tile_iter_end);
    w.tile = (int)(tile_rel + base);
    w.kb_begin = (int)(pos - tile_iter);
    w.kb_end = (int)((end < tile_iter_end ? end : tile_iter_end) - tile_iter);
    w.role = !started ? kRolePeer : (ended ? kRoleFull : kRoleOwner);
    const int last_rel = even_cta_of(q, r, tile_iter_end - 1);
    int64_t last_b, last_e;
    even_range(q, r, last_rel, last_b, last_e);
    const int owner_rel = even_cta_of(q, r, tile_iter);
    int64_t owner_b, owner_e;
    even_range(q, r, owner_rel, owner_b, owner_e);
    w.owner = cta_base + owner_rel;
    w.contrib_last = cta_base + last_rel;
    w.part_last = w.contrib_last - (last_e > tile_iter_end ? 1 : 0);
    w.share_parts = w.part_last - w.owner + 1;
    w.owner_bank2 = owner_b != tile_iter ? 1 : 0;
    w.peer_last = (w.role == kRoleOwner) ? w.contrib_last : x;
    w.region = region;
    pos = tile_iter_end;
  }

  // Whether segment w's tile is reduced by its parts together (launches
  // without ABFT; the caller also checks that it is one of the parts).
  SKG_HD static bool shared(const Schedule& s, const Work& w) {
    return w.region == 0 && w.role != kRoleFull && w.share_parts >= s.share_min &&
           (!w.owner_bank2 || s.share_bank2);
  }
  // Whether segment w's tile is finished by a split reduction (see
  // Schedule::split_max; the caller also checks that it is one of the parts).
  SKG_HD static bool split(const Schedule& s, const Work& w) {
    return w.region == 0 && w.role != kRoleFull && w.share_parts >= 2 &&
           w.share_parts <= s.split_max && w.share_parts < s.share_min &&
           (!w.owner_bank2 || s.share_bank2);
  }

  SKG_HD bool next(const Schedule& s, Work& w) {
    if (ck_it < ck_end) {
      cut(s, s.ck_q, s.ck_r, 0, 1, x, ck_base, ck_it, ck_end, w);
      return true;
    }
    if (next_dp < s.t_dp) {
      w.tile = s.t_ck + next_dp;
      w.kb_begin = 0;
      w.kb_end = s.ipt;
      w.role = kRoleFull;
      w.peer_last = x;
      w.region = 0;
      w.owner = w.contrib_last = w.part_last = x;
      w.share_parts = 0;
      w.owner_bank2 = 0;
      next_dp += s.g;
      return true;
    }
    if (it < it_end) {
      cut(s, s.sk_q, s.sk_r, s.t_ck + s.t_dp, 0, x, 0, it, it_end, w);
      return true;
    }
    return false;
  }
};

}  // namespace skg
