"""Stream-K schedule simulator (test infrastructure, CPU only).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. It shares no code with the CUDA path and imports nothing from it.

Written from "Stream-K: Work-centric Parallel Decomposition for Dense
Matrix-Matrix Multiplication on the GPU":

* Algorithm 2 (§3.2, data-parallel), Algorithm 4 (§3.3, fixed-split) and
  Algorithm 5 (§4, Stream-K) give the per-CTA iteration ranges;
* §5.2 gives the two hybrids ("data-parallel + one-tile Stream-K" and
  "two-tile Stream-K + data-parallel");
* §A1 / Figs. 1-2 and §5.2 / Fig. 3 give the worked examples the tests pin.

Readings where the page is silent or garbled (each is also listed in the
design notes):

* R1 even split. §A1 says the MAC iterations are split evenly "to within one
  iteration"; Algorithm 5 instead gives every CTA ``ceil(T/g)``.  The GPU
  schedule uses the even split: CTA x gets ``q + [x < r]`` iterations starting
  at ``x*q + min(x, r)`` with ``q, r = divmod(T, g)``.  The printed ceil
  variant is kept as ``split="ceil"`` (with its end clamped at T).
* R2 tile coordinates. Algorithm 3 divides by ``ceil(m/BLK_M)`` on both lines;
  tiles are numbered row-major: ``tile = tm * tiles_n + tn``.
* R3 peers. Algorithm 5's peer loop is garbled; the peers of a tile's owner
  are every later CTA whose range meets the tile, accumulated in ascending
  CTA order.
* R4 hybrid placement (Fig. 3b/3c bodies are missing). The data-parallel
  tiles are tile indices ``[0, t_dp)`` and the Stream-K region is the last
  ``t - t_dp`` tiles. Persistent CTA x runs DP tiles ``x, x+g, ...`` first,
  then its Stream-K range.
* R5 hybrid sizes (§5.2): ``w = t // g`` full waves. If ``t % g == 0`` the
  schedule is pure DP. "DP + one-tile SK": ``t_dp = w*g``. "Two-tile SK + DP":
  if ``w >= 2``, ``t_dp = (w-1)*g``, else as "DP + one-tile SK".
"""
from __future__ import annotations

from dataclasses import dataclass
from math import ceil
from typing import Dict, List, Tuple

# Roles of a segment, as defined by Algorithm 5's tile_started / tile_ended.
FULL = 0    # started and ended: this CTA computes the whole tile and stores it
OWNER = 1   # started, not ended: waits for peers, accumulates, stores
PEER = 2    # not started: stores partials and signals

MODES = ("dp", "sk", "dp_sk1", "sk2_dp")


@dataclass(frozen=True)
class Segment:
    cta: int
    tile: int
    k_iter_begin: int   # local MAC-iteration index within the tile
    k_iter_end: int     # exclusive
    role: int


def tile_grid(m: int, n: int, k: int, bm: int, bn: int, bk: int) -> Tuple[int, int, int]:
    """(ceil(m/BLK_M), ceil(n/BLK_N), iters_per_tile = ceil(k/BLK_K)) -- Alg. 2 line 2."""
    return ceil(m / bm), ceil(n / bn), ceil(k / bk)


def tile_coords(tile: int, tiles_n: int) -> Tuple[int, int]:
    """Row-major tile numbering (reading R2 of Algorithm 3)."""
    return tile // tiles_n, tile % tiles_n


# --------------------------------------------------------------------------
# Algorithm 2 / Figure 1: data-parallel, one CTA per tile
# --------------------------------------------------------------------------
def dp_utilization(num_ctas: int, sms: int) -> float:
    """Upper bound on processor utilisation when `num_ctas` equal CTAs run on
    `sms` SMs in waves (Fig. 1a: 9 CTAs on 4 SMs -> 75 %)."""
    waves = ceil(num_ctas / sms)
    return num_ctas / (sms * waves)


def data_parallel_ranges(m, n, k, bm, bn, bk):
    """Algorithm 2: CTA x owns tile x and runs iterations [0, iters_per_tile)."""
    tm, tn, ipt = tile_grid(m, n, k, bm, bn, bk)
    return [(x, 0, ipt) for x in range(tm * tn)]


# --------------------------------------------------------------------------
# Algorithm 4 / Figure 2a: fixed split
# --------------------------------------------------------------------------
def fixed_split_ranges(m, n, k, bm, bn, bk, s):
    """Algorithm 4: CTA (x, y) runs [y*ips, min(ipt, y*ips + ips)) of tile x,
    with ips = ceil(ipt / s). Returns a list of (tile, split, begin, end)."""
    tm, tn, ipt = tile_grid(m, n, k, bm, bn, bk)
    ips = ceil(ipt / s)
    out = []
    for x in range(tm * tn):
        for y in range(s):
            it = y * ips
            it_end = min(ipt, it + ips)
            out.append((x, y, it, it_end))
    return out


# --------------------------------------------------------------------------
# Algorithm 5: Stream-K range of one CTA
# --------------------------------------------------------------------------
def sk_range(x: int, total_iters: int, g: int, split: str = "even") -> Tuple[int, int]:
    """[iter, iter_end) of CTA x over `total_iters` MAC iterations."""
    if split == "even":                       # reading R1
        q, r = divmod(total_iters, g)
        begin = x * q + min(x, r)
        return begin, begin + q + (1 if x < r else 0)
    if split == "ceil":                       # Alg. 5 lines 4, 7, 8 (+ clamp)
        ipc = ceil(total_iters / g)
        begin = min(x * ipc, total_iters)
        return begin, min(begin + ipc, total_iters)
    raise ValueError(split)


def walk_range(x: int, it: int, it_end: int, ipt: int, tile_offset: int = 0) -> List[Segment]:
    """Algorithm 5, lines 10-38: cut [it, it_end) at tile boundaries and label
    each piece with its role. `tile_offset` shifts tile numbers (used by the
    hybrids, whose Stream-K region starts at tile t_dp)."""
    segs = []
    while it < it_end:
        tile = it // ipt
        tile_iter = tile * ipt
        tile_iter_end = tile_iter + ipt
        local_begin = it - tile_iter
        local_end = min(it_end, tile_iter_end) - tile_iter
        started = it == tile_iter
        ended = it_end >= tile_iter_end
        if not started:
            role = PEER
        elif ended:
            role = FULL
        else:
            role = OWNER
        segs.append(Segment(x, tile + tile_offset, local_begin, local_end, role))
        it = tile_iter_end
    return segs


# --------------------------------------------------------------------------
# The persistent schedule the GPU runs (modes of §4 and §5.2)
# --------------------------------------------------------------------------
def dp_tile_count(t: int, g: int, mode: str) -> int:
    """Number of data-parallel tiles t_dp for each mode (reading R5)."""
    if mode == "dp":
        return t
    if mode == "sk":
        return 0
    w = t // g
    if t % g == 0:
        return t
    if mode == "dp_sk1":
        return w * g
    if mode == "sk2_dp":
        return (w - 1) * g if w >= 2 else w * g
    raise ValueError(mode)


def schedule(m, n, k, bm, bn, bk, g, mode="sk2_dp", split="even") -> List[List[Segment]]:
    """Per-CTA ordered segment lists of the persistent schedule.

    CTA x first runs DP tiles x, x+g, ... below t_dp (each FULL), then its
    Stream-K range over the iteration space of tiles [t_dp, t)."""
    if g < 1:
        raise ValueError("g must be >= 1")
    tm, tn, ipt = tile_grid(m, n, k, bm, bn, bk)
    t = tm * tn
    out: List[List[Segment]] = [[] for _ in range(g)]
    if t == 0 or ipt == 0:
        return out
    t_dp = dp_tile_count(t, g, mode)
    for x in range(g):
        for tile in range(x, t_dp, g):
            out[x].append(Segment(x, tile, 0, ipt, FULL))
    sk_total = (t - t_dp) * ipt
    if sk_total:
        for x in range(g):
            b, e = sk_range(x, sk_total, g, split)
            out[x].extend(walk_range(x, b, e, ipt, tile_offset=t_dp))
    return out


# --------------------------------------------------------------------------
# Derived quantities
# --------------------------------------------------------------------------
def iters_per_cta(sched: List[List[Segment]]) -> List[int]:
    return [sum(s.k_iter_end - s.k_iter_begin for s in segs) for segs in sched]


def utilization(sched: List[List[Segment]]) -> float:
    """Total MAC iterations / (g * the busiest CTA's iterations)."""
    per = iters_per_cta(sched)
    busiest = max(per) if per else 0
    return sum(per) / (len(per) * busiest) if busiest else 0.0


def first_k_offsets(sched: List[List[Segment]], bk: int) -> List[int]:
    """k offset of each CTA's first MAC iteration (Fig. 3a: 0, 32, 64, 96)."""
    return [segs[0].k_iter_begin * bk if segs else -1 for segs in sched]


def owners_and_peers(sched: List[List[Segment]]) -> Dict[int, Tuple[int, List[int]]]:
    """tile -> (storing CTA, ascending list of peer CTAs) (reading R3)."""
    owner: Dict[int, int] = {}
    peers: Dict[int, List[int]] = {}
    for segs in sched:
        for s in segs:
            if s.role in (FULL, OWNER):
                if s.tile in owner:
                    raise AssertionError(f"tile {s.tile} has two owners")
                owner[s.tile] = s.cta
            else:
                peers.setdefault(s.tile, []).append(s.cta)
    return {tile: (o, sorted(peers.get(tile, []))) for tile, o in owner.items()}


def coverage(sched: List[List[Segment]], t: int, ipt: int) -> List[List[int]]:
    """How many times each (tile, k-iteration) is assigned (must be all 1)."""
    cov = [[0] * ipt for _ in range(t)]
    for segs in sched:
        for s in segs:
            for it in range(s.k_iter_begin, s.k_iter_end):
                cov[s.tile][it] += 1
    return cov


def flatten(sched: List[List[Segment]]) -> List[Tuple[int, int, int, int, int]]:
    """(cta, tile, k_iter_begin, k_iter_end, role) rows in CTA-then-order."""
    return [(s.cta, s.tile, s.k_iter_begin, s.k_iter_end, s.role)
            for segs in sched for s in segs]
