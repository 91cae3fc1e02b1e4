"""Pins of the Stream-K schedule simulator against what the Stream-K page fixes.

Worked examples come from tests/golden/streamk_worked_examples.json (each
entry cites its section and figure); invariants are checked by brute force.
"""
import json
import os
import random

import pytest

from oracle import schedule_sim as ss

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "streamk_worked_examples.json")))


def test_dp_75_percent_fig1a():
    g = GOLD["dp_384_tiles_128x128"]
    ranges = ss.data_parallel_ranges(g["m"], g["n"], g["k"], g["bm"], g["bn"], 128)
    assert len(ranges) == g["ctas"]
    assert ss.dp_utilization(len(ranges), g["sms"]) == pytest.approx(g["utilization"], abs=0)


def test_dp_90_percent_fig1b():
    g = GOLD["dp_384_tiles_128x64"]
    ranges = ss.data_parallel_ranges(g["m"], g["n"], g["k"], g["bm"], g["bn"], 128)
    assert len(ranges) == g["ctas"]
    assert ss.dp_utilization(len(ranges), g["sms"]) == pytest.approx(g["utilization"], abs=1e-15)


def test_fixed_split_90_percent_fig2a():
    g = GOLD["fixed_split_384_s2"]
    r = ss.fixed_split_ranges(g["m"], g["n"], g["k"], g["bm"], g["bn"], g["bk"], g["s"])
    assert len(r) == g["ctas"]
    # each CTA does a 128x128x64 piece: one MAC iteration of BLK_K = 64
    assert all(e - b == 1 for (_, _, b, e) in r)
    assert ss.dp_utilization(len(r), g["sms"]) == pytest.approx(g["utilization"], abs=1e-15)


def test_basic_streamk_100_percent_fig2b():
    g = GOLD["basic_sk_384_g4"]
    sch = ss.schedule(g["m"], g["n"], g["k"], g["bm"], g["bn"], g["bk"], g["g"], mode="sk")
    per = ss.iters_per_cta(sch)
    assert per == [g["iters_per_cta"]] * g["g"]
    assert per[0] * g["bk"] == g["cta_k_extent"]
    assert ss.utilization(sch) == g["utilization"]
    # the printed ceil split agrees here (288 divides evenly by 4)
    sch_c = ss.schedule(g["m"], g["n"], g["k"], g["bm"], g["bn"], g["bk"], g["g"], mode="sk",
                        split="ceil")
    assert ss.flatten(sch_c) == ss.flatten(sch)


def test_bk64_gives_90_percent_not_100():
    # Reading recorded with the worked example: the page's 100 % needs BLK_K=4;
    # at BLK_K=64 the same problem has 18 iterations -> 5,5,4,4 -> 90 %.
    sch = ss.schedule(384, 384, 128, 128, 128, 64, 4, mode="sk")
    assert ss.iters_per_cta(sch) == [5, 5, 4, 4]
    assert ss.utilization(sch) == pytest.approx(0.9, abs=1e-15)


def test_iteration_is_32x_smaller_and_32way_split_is_perfect():
    g = GOLD["iteration_vs_tile_ratio"]
    ipt = ss.tile_grid(128, 128, g["k"], g["bm"], g["bn"], g["bk"])[2]
    assert ipt == g["ratio"]
    r = ss.fixed_split_ranges(384, 384, 128, 128, 128, g["bk"], g["fixed_split_ways"])
    assert ss.dp_utilization(len(r), 4) == g["fixed_split_utilization"]


def test_skew_k_offsets_fig3a():
    g = GOLD["basic_sk_896_g4_skew"]
    sch = ss.schedule(g["m"], g["n"], g["k"], g["bm"], g["bn"], g["bk"], g["g"], mode="sk")
    assert ss.first_k_offsets(sch, g["bk"]) == g["first_k_offsets"]


def test_single_tile_deep_k_fig9():
    g = GOLD["single_tile_deep_k"]
    dp = ss.schedule(g["m"], g["n"], g["k"], g["bm"], g["bn"], g["bk"], g["g"], mode="dp")
    sk = ss.schedule(g["m"], g["n"], g["k"], g["bm"], g["bn"], g["bk"], g["g"], mode="sk")
    assert sum(1 for s in dp if s) == g["dp_ctas_with_work"]
    assert sum(1 for s in sk if s) == g["sk_ctas_with_work"]
    assert [len(s) for s in sk] == [1, 1, 1, 1]
    assert sk[0][0].role == ss.OWNER and all(s[0].role == ss.PEER for s in sk[1:])
    assert ss.owners_and_peers(sk) == {0: (0, [1, 2, 3])}


@pytest.mark.parametrize("shape", [(384, 384, 128), (896, 384, 128), (640, 1280, 512)])
def test_g_equals_t_is_data_parallel(shape):
    # §4 (generality): with g equal to the number of tiles Stream-K is DP.
    m, n, k = shape
    tm, tn, ipt = ss.tile_grid(m, n, k, 128, 128, 32)
    t = tm * tn
    sk = ss.schedule(m, n, k, 128, 128, 32, t, mode="sk")
    assert [[(s.tile, s.k_iter_begin, s.k_iter_end, s.role) for s in segs] for segs in sk] == \
        [[(x, 0, ipt, ss.FULL)] for x, _, _ in ss.data_parallel_ranges(m, n, k, 128, 128, 32)]


@pytest.mark.parametrize("s", [2, 4, 8])
def test_g_multiple_of_t_is_fixed_split(s):
    # §4 (generality): g = s * t gives the fixed-split schedule of Algorithm 4.
    m, n, k, bk = 384, 256, 1024, 32
    tm, tn, ipt = ss.tile_grid(m, n, k, 128, 128, bk)
    t = tm * tn
    sk = ss.schedule(m, n, k, 128, 128, bk, s * t, mode="sk")
    fs = ss.fixed_split_ranges(m, n, k, 128, 128, bk, s)
    got = [(segs[0].tile, segs[0].k_iter_begin, segs[0].k_iter_end) for segs in sk]
    want = [(x, b, e) for (x, y, b, e) in fs]
    assert got == want
    for segs, (x, y, b, e) in zip(sk, fs):
        assert segs[0].role == (ss.OWNER if y == 0 else ss.PEER)


def _check_invariants(m, n, k, bm, bn, bk, g, mode):
    tm, tn, ipt = ss.tile_grid(m, n, k, bm, bn, bk)
    t = tm * tn
    sch = ss.schedule(m, n, k, bm, bn, bk, g, mode=mode)
    # every (tile, k-iteration) exactly once
    cov = ss.coverage(sch, t, ipt)
    assert all(c == 1 for row in cov for c in row)
    # exactly one storing CTA per tile; peers are later CTAs
    op = ss.owners_and_peers(sch)
    assert sorted(op) == list(range(t))
    for tile, (o, peers) in op.items():
        assert all(p > o for p in peers)
    t_dp = ss.dp_tile_count(t, g, mode)
    # Stream-K region: per-CTA iteration counts differ by at most one
    sk_counts = [sum(s.k_iter_end - s.k_iter_begin for s in segs if s.tile >= t_dp)
                 for segs in sch]
    if t_dp < t:
        assert max(sk_counts) - min(sk_counts) <= 1
    # segments are contiguous in the m -> n -> k linear order of the SK region
    for segs in sch:
        lin = [(s.tile * ipt + s.k_iter_begin, s.tile * ipt + s.k_iter_end)
               for s in segs if s.tile >= t_dp]
        for (b0, e0), (b1, e1) in zip(lin, lin[1:]):
            assert e0 == b1
        # a CTA's only non-started segment is its first Stream-K segment
        sk_roles = [s.role for s in segs if s.tile >= t_dp]
        assert ss.PEER not in sk_roles[1:]
    return sch, op, t, t_dp


def test_invariants_brute_force():
    rnd = random.Random(12345)
    for _ in range(400):
        m = rnd.randint(1, 1500)
        n = rnd.randint(1, 1500)
        k = rnd.randint(1, 2000)
        bm = 128
        bn = rnd.choice([64, 128, 256])
        bk = rnd.choice([16, 32, 64])
        g = rnd.randint(1, 40)
        mode = rnd.choice(ss.MODES)
        _check_invariants(m, n, k, bm, bn, bk, g, mode)


def test_two_tile_hybrid_one_peer_per_owner():
    # §5.2: with w >= 2 full waves, each accumulating CTA receives partial
    # sums from only one other CTA.
    rnd = random.Random(7)
    checked = 0
    for _ in range(300):
        g = rnd.randint(2, 150)
        tm = rnd.randint(1, 40)
        tn = rnd.randint(1, 40)
        t = tm * tn
        if t // g < 2 or t % g == 0:
            continue
        k = 64 * rnd.randint(1, 64)
        sch, op, t, t_dp = _check_invariants(128 * tm, 128 * tn, k, 128, 128, 64, g, "sk2_dp")
        assert t_dp == (t // g - 1) * g
        assert all(len(peers) <= 1 for (_, peers) in op.values())
        # each SK CTA holds between one and two tiles' worth of iterations
        # (the even split may round one CTA up to exactly two)
        ipt = k // 64
        for segs in sch:
            it = sum(s.k_iter_end - s.k_iter_begin for s in segs if s.tile >= t_dp)
            assert ipt <= it <= 2 * ipt
        checked += 1
    assert checked > 50


def test_hybrid_sizes():
    # 169 tiles on 148 CTAs: one full wave (w=1) -> DP + one-tile SK tail.
    assert ss.dp_tile_count(169, 148, "sk2_dp") == 148
    assert ss.dp_tile_count(169, 148, "dp_sk1") == 148
    # 380 tiles: w=2 -> two-tile hybrid gives up one DP wave.
    assert ss.dp_tile_count(380, 148, "sk2_dp") == 148
    assert ss.dp_tile_count(380, 148, "dp_sk1") == 296
    # exact multiple -> pure DP
    assert ss.dp_tile_count(296, 148, "sk2_dp") == 296
    assert ss.dp_tile_count(4, 148, "sk2_dp") == 0


def test_ceil_split_can_leave_short_ctas():
    # Algorithm 5 as printed: T=18, g=4 -> 5,5,5,3 (differs by more than one)
    sch = ss.schedule(384, 384, 128, 128, 128, 64, 4, mode="sk", split="ceil")
    assert ss.iters_per_cta(sch) == [5, 5, 5, 3]
    sch = ss.schedule(384, 384, 128, 128, 128, 64, 4, mode="sk", split="even")
    assert ss.iters_per_cta(sch) == [5, 5, 4, 4]


def test_sk_range_even_and_ceil_hand_computed():
    # T = 18 MAC iterations on g = 4 CTAs. The even split of the Stream-K
    # page's appendix A1 (counts differ by one at most) gives 5, 5, 4, 4
    # contiguous ranges; Algorithm 5's ceil(T / g) = 5 per CTA gives 5, 5, 5, 3
    # once clamped at T.
    assert [ss.sk_range(x, 18, 4) for x in range(4)] == [(0, 5), (5, 10), (10, 14), (14, 18)]
    assert [ss.sk_range(x, 18, 4, "ceil") for x in range(4)] == \
        [(0, 5), (5, 10), (10, 15), (15, 18)]
    # More CTAs than iterations: the last CTAs get empty ranges at T.
    assert [ss.sk_range(x, 3, 5) for x in range(5)] == [(0, 1), (1, 2), (2, 3), (3, 3), (3, 3)]
    assert [ss.sk_range(x, 3, 5, "ceil") for x in range(5)] == \
        [(0, 1), (1, 2), (2, 3), (3, 3), (3, 3)]
    with pytest.raises(ValueError):
        ss.sk_range(0, 3, 5, "other")


def test_walk_range_roles_hand_computed():
    # Algorithm 5 cuts a CTA's range at tile boundaries (8 iterations per
    # tile here): a segment that does not start its tile is a PEER, one that
    # starts and ends it FULL, one that starts it and stops inside it the
    # OWNER.
    def cut(x, b, e, off=0):
        return [(s.cta, s.tile, s.k_iter_begin, s.k_iter_end, s.role)
                for s in ss.walk_range(x, b, e, 8, tile_offset=off)]
    assert cut(1, 5, 20) == [(1, 0, 5, 8, ss.PEER), (1, 1, 0, 8, ss.FULL),
                             (1, 2, 0, 4, ss.OWNER)]
    assert cut(0, 3, 6) == [(0, 0, 3, 6, ss.PEER)]     # inside one tile, not its start
    assert cut(0, 0, 3) == [(0, 0, 0, 3, ss.OWNER)]    # starts the tile, stops inside
    assert cut(0, 8, 16) == [(0, 1, 0, 8, ss.FULL)]
    assert cut(0, 7, 7) == []
    # the hybrids' Stream-K region is numbered from tile t_dp on
    assert [(t, role) for (_, t, _, _, role) in cut(2, 5, 20, off=10)] == \
        [(10, ss.PEER), (11, ss.FULL), (12, ss.OWNER)]


def test_tile_coords_row_major():
    # Reading R2 of Algorithm 3: tile = tm * tiles_n + tn.
    assert [ss.tile_coords(t, 3) for t in range(7)] == \
        [(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 2), (2, 0)]
    assert ss.tile_coords(5, 1) == (5, 0)
