// Stream-K schedule arithmetic, shared by the host-side schedule query and
// the persistent kernel (every role warp walks the same list).
//
// "Stream-K: Work-centric Parallel Decomposition for Dense Matrix-Matrix
// Multiplication on the GPU":
//   - Algorithm 5 (§4): the MAC iterations of all tiles form one linear
//     m -> n -> k space split over g CTAs; a CTA's range is cut at tile
//     boundaries into segments; tile_started / tile_ended give the role.
//   - §A1: iterations are split evenly "to within one iteration": CTA x gets
//     q + [x < r] iterations starting at x*q + min(x, r), (q, r) = divmod(T, g).
//   - §5.2: "DP + one-tile SK" keeps w = floor(t/g) full DP waves; "two-tile
//     SK + DP" gives one of them up when w >= 2 so every Stream-K CTA holds
//     between one and two tiles of iterations. DP tiles are the first t_dp
//     tile indices, walked x, x+g, ...; the Stream-K region is the rest.
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

struct Schedule {
  int tiles_m, tiles_n;
  int ipt;            // MAC iterations per tile, ceil(k / BLK_K)
  int t;              // tiles (t_ck + tiles_m * tiles_n)
  int t_ck;           // leading tiles of fused side GEMMs (0 for a plain GEMM)
  int t_dp;           // data-parallel tiles [0, t_dp)
  int g;              // persistent CTAs
  int64_t sk_total;   // Stream-K iterations (t - t_dp) * ipt
  int64_t sk_q;       // floor(sk_total / g)
  int sk_r;           // sk_total mod g
  int band;           // tile columns per raster band (tiles_n = row-major)
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

// `t_ck` extra full-k tiles are placed in front of the output tiles (the
// fused ABFT checksum GEMMs); the schedule treats every tile alike.
SKG_HD Schedule make_schedule(int64_t m, int64_t n, int64_t k, int bm, int bn, int bk, int g,
                              int mode, int t_ck = 0) {
  Schedule s;
  s.tiles_m = (int)((m + bm - 1) / bm);
  s.tiles_n = (int)((n + bn - 1) / bn);
  s.ipt = (int)((k + bk - 1) / bk);
  s.t_ck = (s.tiles_m * s.tiles_n > 0) ? t_ck : 0;
  s.t = s.t_ck + s.tiles_m * s.tiles_n;
  s.g = g;
  s.t_dp = (s.t == 0 || s.ipt == 0) ? s.t : dp_tiles(s.t, g, mode);
  s.sk_total = (int64_t)(s.t - s.t_dp) * s.ipt;
  s.sk_q = s.sk_total / g;
  s.sk_r = (int)(s.sk_total % g);
  s.band = s.tiles_n > 0 ? s.tiles_n : 1;
  return s;
}

// [begin, end) of CTA x in the Stream-K iteration space (even split).
SKG_HD void sk_range(const Schedule& s, int x, int64_t& begin, int64_t& end) {
  begin = (int64_t)x * s.sk_q + (x < s.sk_r ? x : s.sk_r);
  end = begin + s.sk_q + (x < s.sk_r ? 1 : 0);
}

// CTA whose Stream-K range holds iteration `it` (0 <= it < sk_total).
SKG_HD int sk_cta_of(const Schedule& s, int64_t it) {
  const int64_t big = (int64_t)s.sk_r * (s.sk_q + 1);
  if (it < big) return (int)(it / (s.sk_q + 1));
  return s.sk_r + (int)((it - big) / s.sk_q);
}

struct Work {
  int tile;
  int kb_begin, kb_end;  // MAC iterations within the tile
  int role;
  int peer_last;         // OWNER: last peer CTA (peers are cta+1 .. peer_last)
};

// Walks one CTA's segments in execution order: DP tiles, then its
// Stream-K range cut at tile boundaries.
struct Cursor {
  int x;
  int next_dp;
  int64_t it, it_end;

  SKG_HD void init(const Schedule& s, int cta) {
    x = cta;
    next_dp = cta;
    if (s.sk_total > 0) {
      sk_range(s, cta, it, it_end);
    } else {
      it = it_end = 0;
    }
  }

  SKG_HD bool next(const Schedule& s, Work& w) {
    if (next_dp < s.t_dp) {
      w.tile = next_dp;
      w.kb_begin = 0;
      w.kb_end = s.ipt;
      w.role = kRoleFull;
      w.peer_last = x;
      next_dp += s.g;
      return true;
    }
    if (it >= it_end) return false;
    const int64_t tile_sk = it / s.ipt;
    const int64_t tile_iter = tile_sk * s.ipt;
    const int64_t tile_iter_end = tile_iter + s.ipt;
    const bool started = (it == tile_iter);
    const bool ended = (it_end >= tile_iter_end);
    w.tile = (int)(tile_sk + s.t_dp);
    w.kb_begin = (int)(it - tile_iter);
    w.kb_end = (int)((it_end < tile_iter_end ? it_end : tile_iter_end) - tile_iter);
    w.role = !started ? kRolePeer : (ended ? kRoleFull : kRoleOwner);
    w.peer_last = (w.role == kRoleOwner) ? sk_cta_of(s, tile_iter_end - 1) : x;
    it = tile_iter_end;
    return true;
  }
};

}  // namespace skg
