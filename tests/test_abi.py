"""CPU-only checks of the C-ABI library: it loads without a GPU, exports every
symbol include/skgemm.h declares, its host schedule query equals the oracle's
schedule simulator bit-exactly, and argument errors are returned
synchronously (nothing reaches the device)."""
import ctypes
import os
import random
import re

import pytest

from oracle import schedule_sim as ss
from stream_decomposition_abft_gb300 import _build, skgemm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return skgemm.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "skgemm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(skg_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), f"libskgemm.so does not export {name}"
    assert set(skgemm.SYMBOLS) == set(names)


def test_struct_sizes_match_header():
    # Sizes fixed by the header's field lists (x86-64 and aarch64 ABIs agree).
    assert ctypes.sizeof(skgemm.Opts) == 112
    assert ctypes.sizeof(skgemm.Segment) == 20
    assert ctypes.sizeof(skgemm.FaultRecord) == 64
    assert ctypes.sizeof(skgemm.Report) == 64 + 64 * 64
    assert ctypes.sizeof(skgemm.Plan) == 44


def test_defaults(lib):
    o = skgemm.opts_default()
    assert o.sched == skgemm.SCHED_AUTO and o.inject_tile == -1 and o.abft == 0
    assert o.inject2_tile == -1 and o.inject_kstep == -1 and o.stagger == 0
    assert skgemm.status_string(0) == "ok"
    assert "timed out" in skgemm.status_string(skgemm.ERR_FIXUP_TIMEOUT)


MODES = {"dp": skgemm.SCHED_DP, "sk": skgemm.SCHED_SK, "dp_sk1": skgemm.SCHED_DP_SK1,
         "sk2_dp": skgemm.SCHED_SK2_DP}


@pytest.mark.parametrize("mode", list(MODES))
def test_schedule_query_matches_simulator_configs(lib, mode):
    # The workloads' shapes with the kernel's tiles, on 148 CTAs and on the
    # page's hypothetical 4-SM GPU.
    shapes = [(384, 384, 128), (1664, 1664, 8192), (2560, 2432, 4096), (256, 256, 65536),
              (128, 19072, 2048), (4096, 4096, 4096), (8192, 1024, 8192)]
    for (m, n, k) in shapes:
        for bn in (128, 256):
            for g in (4, 148):
                got = skgemm.schedule_query(m, n, k, 128, bn, 64, g, MODES[mode])
                want = ss.flatten(ss.schedule(m, n, k, 128, bn, 64, g, mode=mode))
                assert got == want, (m, n, k, bn, g, mode)


def test_schedule_query_matches_simulator_random(lib):
    rnd = random.Random(2024)
    for _ in range(300):
        m, n, k = rnd.randint(1, 3000), rnd.randint(1, 3000), rnd.randint(1, 5000)
        bn = rnd.choice([128, 256])
        bk = rnd.choice([4, 32, 64])
        g = rnd.randint(1, 160)
        mode = rnd.choice(list(MODES))
        got = skgemm.schedule_query(m, n, k, 128, bn, bk, g, MODES[mode])
        want = ss.flatten(ss.schedule(m, n, k, 128, bn, bk, g, mode=mode))
        assert got == want, (m, n, k, bn, bk, g, mode)


def test_schedule_query_matches_simulator_f64_tiles(lib):
    # The fp64 kernel's 64 x 64 x 16 tiles run the same schedule code: the
    # query for those tiles equals the simulator, bit for bit.
    rnd = random.Random(64)
    for _ in range(150):
        m, n, k = rnd.randint(1, 1500), rnd.randint(1, 1500), rnd.randint(1, 4200)
        g = rnd.randint(1, 160)
        mode = rnd.choice(list(MODES))
        got = skgemm.schedule_query(m, n, k, 64, 64, 16, g, MODES[mode])
        want = ss.flatten(ss.schedule(m, n, k, 64, 64, 16, g, mode=mode))
        assert got == want, (m, n, k, g, mode)


def test_schedule_query_page_example(lib):
    # Stream-K page, Fig. 2b: 384x384x128, BLK_K = 4, g = 4 -> 72 iterations each.
    rows = skgemm.schedule_query(384, 384, 128, 128, 128, 4, 4, skgemm.SCHED_SK)
    per = [0, 0, 0, 0]
    for (cta, tile, b, e, role) in rows:
        per[cta] += e - b
    assert per == [72, 72, 72, 72]


def test_argument_errors_are_synchronous(lib):
    o = skgemm.opts_default()
    args = dict(alpha=1.0, beta=0.0, in_dtype=skgemm.IN_BF16, out_dtype=skgemm.OUT_BF16,
                a_layout=0, b_layout=0, opts=o, ws_ptr=None, ws_bytes=0, stream=None)

    def call(m, n, k, A=16, lda=64, B=16, ldb=64, C=16, ldc=64, **kw):
        a = dict(args)
        a.update(kw)
        return skgemm.gemm(m, n, k, a["alpha"], A, lda, B, ldb, a["beta"], C, ldc,
                           a["in_dtype"], a["out_dtype"], a["a_layout"], a["b_layout"],
                           a["opts"], a["ws_ptr"], a["ws_bytes"], a["stream"])

    assert call(-1, 4, 4) == skgemm.ERR_ARG
    assert call(4, 4, 4, in_dtype=7) == skgemm.ERR_ARG
    assert call(4, 4, 4, out_dtype=9) == skgemm.ERR_ARG
    assert call(4, 4, 4, a_layout=2) == skgemm.ERR_ARG      # unknown layouts
    assert call(4, 4, 4, b_layout=-1) == skgemm.ERR_ARG
    # MN-major operands: the leading dimension spans m (A) or n (B).
    assert call(128, 4, 4, a_layout=skgemm.A_COL, lda=64) == skgemm.ERR_ARG
    assert call(4, 128, 4, b_layout=skgemm.B_NMAJOR, ldb=64) == skgemm.ERR_ARG
    assert call(48, 4, 4, a_layout=skgemm.A_COL, lda=60) == skgemm.ERR_UNSUPPORTED  # 120 bytes
    assert call(0, 4, 4) == skgemm.OK                 # empty output: nothing to do
    assert call(4, 4, 4, C=None) == skgemm.ERR_ARG
    assert call(4, 64, 4, ldc=32) == skgemm.ERR_ARG     # ldc < n
    assert call(4, 4, 4, C=24) == skgemm.ERR_UNSUPPORTED  # C not 16-byte aligned
    assert call(4, 4, 4, ldc=5) == skgemm.ERR_UNSUPPORTED  # ldc * 2 bytes not a multiple of 16
    assert call(4, 4, 64, lda=32) == skgemm.ERR_ARG    # lda < k
    assert call(4, 4, 60, lda=60, ldb=64) == skgemm.ERR_UNSUPPORTED  # lda * 2 % 16 != 0
    assert call(4, 4, 4, A=None) == skgemm.ERR_ARG


def test_workspace_size_scales_with_grid_not_problem(lib):
    # Stream-K page, §4 / conclusion: the fixup storage grows with g, not with
    # the problem size.
    o = skgemm.opts_default(grid=148, tile_n=128)
    small = skgemm.workspace_size(1024, 1024, 1024, o)
    big = skgemm.workspace_size(8192, 8192, 8192, o)
    assert small == big
    o2 = skgemm.opts_default(grid=74, tile_n=128)
    assert skgemm.workspace_size(1024, 1024, 1024, o2) < small
    oa = skgemm.opts_default(grid=148, tile_n=128, abft=1)
    assert skgemm.workspace_size(1024, 1024, 1024, oa) > small


def test_workspace_size_layout(lib):
    # MN-major operands are read in place (with or without ABFT): no extra
    # bytes. Only the in-CTA ABFT references need K-major copies (checked on
    # the GPU, where the library can pick that mode). Unknown layouts: 0.
    for extra in (dict(), dict(abft=1)):
        o = skgemm.opts_default(grid=148, tile_n=128, **extra)
        for al, bl in ((0, 0), (1, 0), (0, 1), (1, 1)):
            assert skgemm.workspace_size_layout(1000, 700, 333, al, bl, o) == \
                skgemm.workspace_size(1000, 700, 333, o)
        assert skgemm.workspace_size_layout(1000, 700, 333, 2, 0, o) == 0


def test_host_staging_size_and_argument_errors(lib):
    # Packed device copies of A and B as stored and of C, rows rounded up to
    # 16 bytes, each region aligned to 256 bytes.
    r256 = lambda x: (x + 255) // 256 * 256
    m, n, k = 100, 60, 33
    want = r256(m * 40 * 2) + r256(n * 40 * 2) + r256(m * 60 * 4)
    assert skgemm.host_staging_size(m, n, k, skgemm.IN_BF16, skgemm.OUT_F32) == want
    want_mn = r256(k * 104 * 2) + r256(k * 64 * 2) + r256(m * 64 * 2)
    assert skgemm.host_staging_size(m, n, k, skgemm.IN_F16, skgemm.OUT_BF16, skgemm.A_COL,
                                    skgemm.B_NMAJOR) == want_mn
    assert skgemm.host_staging_size(m, n, k, 5, skgemm.OUT_F32) == 0
    assert skgemm.host_staging_size(m, n, k, skgemm.IN_F16, skgemm.OUT_F32, 3, 0) == 0
    # Argument errors come back before any copy is issued.
    o = skgemm.opts_default()
    call = lambda **kw: skgemm.gemm_host(
        kw.get("m", m), n, k, 1.0, kw.get("A", 64), kw.get("lda", k), 64, k, 0.0, 64,
        kw.get("ldc", n), skgemm.IN_BF16, skgemm.OUT_F32, 0, 0, o, kw.get("staging", None),
        kw.get("staging_bytes", 0), None, 0, None)
    assert call(m=-1) == skgemm.ERR_ARG
    assert call(lda=k - 1) == skgemm.ERR_ARG
    assert call(ldc=n - 1) == skgemm.ERR_ARG
    assert call(A=None) == skgemm.ERR_ARG
    assert call() == skgemm.ERR_WORKSPACE           # no staging buffer
    assert call(staging=16, staging_bytes=want - 1) == skgemm.ERR_WORKSPACE


def test_f64_workspace_and_argument_errors(lib):
    # One 64 x 64 fp64 slot (32 KB) per CTA after a fixed header, the report
    # and a fixed flag array (1024 flags), whatever the grid.
    a = skgemm.workspace_size_f64(1000, 1000, 1000, skgemm.opts_default(grid=1))
    b = skgemm.workspace_size_f64(1000, 1000, 1000, skgemm.opts_default(grid=148))
    assert b - a == 147 * 32768
    assert a % 256 == 0 and a > 4096 + 32768
    assert skgemm.workspace_size_f64(64, 64, 64, skgemm.opts_default(grid=148)) == b
    o = skgemm.opts_default()
    call = lambda m=64, n=64, k=64, lda=64, ldb=64, ldc=64, A=16, grid=0: skgemm.gemm_f64(
        m, n, k, 1.0, A, lda, 16, ldb, 0.0, 16, ldc, skgemm.opts_default(grid=grid), None, 0,
        None)
    assert call(m=-1) == skgemm.ERR_ARG
    assert call(lda=63) == skgemm.ERR_ARG
    assert call(ldc=32) == skgemm.ERR_ARG
    assert call(A=None) == skgemm.ERR_ARG
    assert call(grid=-3) == skgemm.ERR_ARG
    assert call(m=0) == skgemm.OK


# ----------------------------------------------------------------------------
# Grid-size model (Stream-K page, App. A.1)
# ----------------------------------------------------------------------------
# Model constants (a, c, e, b, d) in microseconds, as fitted for each BLK_N.
MODEL = {64: (2.15, 0.360, 0.11, 4.50, 0.80), 128: (2.64, 0.334, 0.17, 4.67, 1.03),
         256: (3.47, 0.364, 0.00, 8.18, 1.73)}


def brute_force_cost(m, n, k, bn, g, mode):
    """The model evaluated on the simulator's explicit segment lists.

    A launch without ABFT reduces a tile with its covering CTAs together when
    the owner's Stream-K work begins with the tile and at least eight covering
    CTAs end their work in it: each of those stores a partial (the owner too)
    and pays covers / parts + 0.27 * covers peer reads; otherwise the owner
    reads every peer's partial."""
    a, c, e, b, d = MODEL[bn]
    sch = ss.schedule(m, n, k, 128, bn, 64, g, mode=mode)
    op = ss.owners_and_peers(sch)
    tm, tn, _ = ss.tile_grid(m, n, k, 128, bn, 64)
    t_dp = ss.dp_tile_count(tm * tn, g, mode)
    shared = {}
    for tile, (owner, peers) in op.items():
        if not peers:
            continue
        sk = [s for s in sch[owner] if s.tile >= t_dp]
        if sk[0].tile != tile:
            continue
        parts = {x for x in [owner] + list(peers) if sch[x][-1].tile == tile}
        if len(parts) >= 8:
            shared[tile] = (len(parts), 1 + len(peers), parts)
    worst = 0.0
    for x, segs in enumerate(sch):
        iters = sum(s.k_iter_end - s.k_iter_begin for s in segs)
        tiles = sum(1 for s in segs if s.role != ss.PEER)
        partial = sum(1 for s in segs if s.role == ss.PEER)
        fix = 0.0
        for s in segs:
            if s.tile in shared and x in shared[s.tile][2]:
                nparts, covers, _ = shared[s.tile]
                fix += covers / nparts + 0.27 * covers
                partial += 1 if s.role == ss.OWNER else 0
            elif s.role == ss.OWNER:
                fix += len(op[s.tile][1])
        worst = max(worst, a + c * iters + e * tiles + b * partial + d * fix)
    return worst


def test_model_cost_matches_segment_walk(lib):
    rnd = random.Random(99)
    for _ in range(200):
        m, n, k = rnd.randint(1, 4000), rnd.randint(1, 4000), rnd.randint(1, 9000)
        bn = rnd.choice([64, 128, 256])
        g = rnd.randint(1, 152)
        mode = rnd.choice(["dp", "sk", "sk2_dp", "dp_sk1"])
        got = skgemm.schedule_cost(m, n, k, 128, bn, 64, g, MODES[mode])
        want = brute_force_cost(m, n, k, bn, g, mode)
        assert abs(got - want) <= 1e-9 * max(1.0, want), (m, n, k, bn, g, mode, got, want)


def test_plan_honours_explicit_options_and_picks_minimum(lib):
    o = skgemm.opts_default(sched="sk", grid=40, tile_n=128)
    assert skgemm.launch_shape(2048, 2048, 2048, o) == (128, 40, skgemm.SCHED_SK)
    sms = skgemm.device_sm_count() or 256   # without a device the plan assumes 256 SMs
    o = skgemm.opts_default(sched="dp")     # fixed schedule, grid 0 -> every SM
    tn, g, sc = skgemm.launch_shape(2048, 2048, 2048, o)
    assert sc == skgemm.SCHED_DP and g == sms
    # automatic choice is never worse than the page's default (2-tile hybrid on all SMs)
    for (m, n, k) in [(1024, 1024, 1024), (4096, 4096, 4096), (256, 256, 65536),
                      (128, 19072, 2048), (8192, 1024, 8192)]:
        tn, g, sc = skgemm.launch_shape(m, n, k, skgemm.opts_default())
        best = skgemm.schedule_cost(m, n, k, 128, tn, 64, g, sc)
        for bn in (64, 128, 256):
            assert best <= skgemm.schedule_cost(m, n, k, 128, bn, 64, sms, skgemm.SCHED_SK2_DP) + 1e-9


def test_small_tiles_only_without_abft(lib):
    # BLK_N = 64: GEMMs without ABFT on single CTAs; the model may choose it
    # by itself only for those.
    for kw in (dict(tile_n=64, abft=1), dict(tile_n=64, cta_pair=2), dict(tile_n=96)):
        o = skgemm.opts_default(**kw)
        assert skgemm.lib().skg_launch_plan(512, 512, 512, ctypes.byref(o),
                                            ctypes.byref(skgemm.Plan())) == skgemm.ERR_UNSUPPORTED
        assert skgemm.workspace_size(512, 512, 512, o) == 0
    pl = skgemm.launch_plan(256, 256, 384, skgemm.opts_default(tile_n=64, sched="sk", grid=9))
    assert (pl.tile_n, pl.ctas, pl.sched, pl.cta_pair) == (64, 9, skgemm.SCHED_SK, 1)
    for (m, n, k) in [(256, 256, 384), (640, 640, 256), (128, 128, 8192), (4096, 4096, 4096)]:
        assert skgemm.launch_plan(m, n, k, skgemm.opts_default(abft=1)).tile_n != 64
    # a tiny GEMM: fewer MAC iterations per CTA and a cheaper fixed cost
    assert skgemm.launch_plan(256, 256, 384, skgemm.opts_default()).tile_n == 64
    assert skgemm.launch_plan(4096, 4096, 4096, skgemm.opts_default()).tile_n != 64
    assert skgemm.schedule_cost(256, 256, 384, 128, 64, 64, 8, skgemm.SCHED_DP) < \
        skgemm.schedule_cost(256, 256, 384, 128, 128, 64, 4, skgemm.SCHED_DP)


def test_launch_plan_agrees_with_launch_shape(lib):
    for (m, n, k, kw) in [(1024, 1024, 1024, {}), (4096, 4096, 4096, dict(abft=1)),
                          (8192, 1024, 8192, dict(tile_n=128)),
                          (2048, 2048, 2048, dict(cta_pair=2, abft=1)),
                          (512, 512, 512, dict(cta_pair=1, sched="sk", grid=40))]:
        o = skgemm.opts_default(**kw)
        pl = skgemm.launch_plan(m, n, k, o)
        tn, g, sc = skgemm.launch_shape(m, n, k, o)
        assert (pl.tile_n, pl.ctas + pl.side_ctas, pl.sched) == (tn, g, sc)
        assert pl.tile_m == (256 if pl.cta_pair == 2 else 128)
        if kw.get("cta_pair") == 2:
            assert pl.cta_pair == 2 and pl.ctas % 2 == 0 and pl.tile_n == 256
            assert pl.fused_checksums == 1 and pl.side_ctas == 0
    assert skgemm.lib().skg_launch_plan(4, 4, 4, None, None) == skgemm.ERR_ARG
    bad = skgemm.opts_default(cta_pair=3)
    assert skgemm.lib().skg_launch_plan(4, 4, 4, ctypes.byref(bad),
                                        ctypes.byref(skgemm.Plan())) == skgemm.ERR_ARG
