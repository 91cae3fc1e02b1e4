"""GPU ABFT decisions against the oracle, decision by decision.

The kernel's verify step ("Anatomy of High-Performance GEMM with Online
Fault Tolerance on GPUs", thread-level FT, Fig. 3: locate a fault by the
mismatching row and column checksums, correct it from the row checksum) must
reach the same outcome as ``oracle.abft_ref.verify_tile`` on the same
accumulator: the status (clean / corrected / uncorrectable), the number of
mismatching rows and columns, the located row and column and the corrected
value.

On integer-valued inputs every product, row sum, column sum and reference
checksum is exact in fp32, on the GPU as in the fp64 oracle, so the GPU's
pre-fault accumulator IS the oracle's product and the comparison is exact.
Faults are planted through the library's two injection slots, so one tile
can get two flips (the pattern the single-fault rule cannot correct) and two
tiles one flip each; a flip whose change lies between the column threshold
and the row threshold (128 x 256 tiles: tau_row uses sqrt(256), tau_col
sqrt(128)) gives the grey-band pattern of one bad column and no bad row.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from oracle import abft_ref as ab
from oracle import schedule_sim as ss
from stream_decomposition_abft_gb300 import _build, inputs, skgemm

from gpu_util import check_full, draw_must_detect, reference, run

pytestmark = pytest.mark.gpu

STATUS = {ab.CORRECTED: skgemm.ABFT_CORRECTED, ab.UNCORRECTABLE: skgemm.ABFT_UNCORRECTABLE}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    skgemm.lib()


def sms():
    return skgemm.device_sm_count()


# --------------------------------------------------------------------------- helpers
M, N, K = 512, 768, 1536     # every tile full; k puts 1.0 in the grey band at 128 x 256


def integer_problem(seed):
    # entries in [-3, 3]: |acc| <= 9 k = 13824 and every row / column sum of
    # a 128 x 256 tile stays below 2^22, so fp32 holds them exactly
    return inputs.make_problem(M, N, K, seed=seed, in_dtype="bf16", out_dtype="f32",
                               law_a="integer", law_b="integer")


def oracle_outcomes(p, C_exact, bn, flips):
    """Oracle decision for every tile that gets a flip.

    flips: list of (tile, row, col, bit) applied to the exact product (the
    GPU's own pre-fault accumulator on integer data). Returns {tile: result
    of verify_tile} for those tiles."""
    A = p.A.double().numpy()                 # stored m x k
    Bs = p.B.double().numpy()                # stored n x k
    tiles_n = N // bn
    out = {}
    for tile in sorted({f[0] for f in flips}):
        tm, tn = divmod(tile, tiles_n)
        acc = C_exact[tm * 128:(tm + 1) * 128, tn * bn:(tn + 1) * bn].copy()
        for (t, r, c, bit) in flips:
            if t == tile:
                acc[r, c] = ab.flip_f32(acc[r, c], bit)
        cc, cr = ab.tile_reference(A, Bs.T, tm, tn, 128, bn)
        ma, mb = ab.tile_maxima(A, Bs, tm, tn, 128, bn)
        tau_r = ab.default_tau(K, bn, ma, mb)
        tau_c = ab.default_tau(K, 128, ma, mb)
        out[tile] = ab.verify_tile(acc, cr, cc, tau_r, tau_c)
    return out


def gpu_records(rep):
    return {int(r.tile): r for r in rep.records[:min(rep.n_records, skgemm.MAX_RECORDS)]}


def assert_same_decisions(rep, expect, n_tiles, C_exact=None, bn=None):
    assert rep.tiles_checked == n_tiles
    bad = {t: e for t, e in expect.items() if e["status"] != ab.CLEAN}
    assert rep.detected == len(bad)
    assert rep.corrected == sum(e["status"] == ab.CORRECTED for e in bad.values())
    assert rep.uncorrectable == sum(e["status"] == ab.UNCORRECTABLE for e in bad.values())
    recs = gpu_records(rep)
    assert set(recs) == set(bad), (sorted(recs), sorted(bad))
    for t, e in bad.items():
        r = recs[t]
        assert r.status == STATUS[e["status"]]
        assert (r.n_bad_rows, r.n_bad_cols) == (len(e["bad_rows"]), len(e["bad_cols"]))
        want_row = e["bad_rows"][0] if len(e["bad_rows"]) == 1 else -1
        want_col = e["bad_cols"][0] if len(e["bad_cols"]) == 1 else -1
        assert (r.row, r.col) == (want_row, want_col)
        assert r.injected == 1
        if e["status"] == ab.CORRECTED:
            assert r.after == e["value"]        # exact: integers
            tn = t % (N // bn)
            tm = t // (N // bn)
            assert e["value"] == C_exact[tm * 128 + r.row, tn * bn + r.col]


def pick(C_exact, bn, tile, lo, hi, rng, exclude_rows=(), exclude_cols=()):
    """(row, col) in `tile` whose exact value has lo <= |v| < hi."""
    tiles_n = N // bn
    tm, tn = divmod(tile, tiles_n)
    block = np.abs(C_exact[tm * 128:(tm + 1) * 128, tn * bn:(tn + 1) * bn])
    cand = np.argwhere((block >= lo) & (block < hi))
    cand = [(int(a), int(b)) for a, b in cand if a not in exclude_rows and b not in exclude_cols]
    assert cand, "no candidate entry"
    return cand[int(rng.integers(0, len(cand)))]


def grey_bit(v):
    """Mantissa bit of fp32 v whose flip changes v by exactly 1.0."""
    e = math.frexp(abs(v))[1] - 1          # |v| in [2^e, 2^(e+1))
    return 23 - e


def scenario(name, C_exact, bn, rng):
    """Flips (tile, row, col, bit) of one named mismatch pattern."""
    tiles = (M // 128) * (N // bn)
    t1 = int(rng.integers(0, tiles))
    if name == "single_exponent":
        r, c = pick(C_exact, bn, t1, 16, 1e9, rng)
        return [(t1, r, c, 27)]
    if name == "single_to_inf":
        r, c = pick(C_exact, bn, t1, 1, 2, rng)            # |v| = 1: bit 30 -> Inf
        return [(t1, r, c, 30)]
    if name == "two_in_tile":
        r1, c1 = pick(C_exact, bn, t1, 16, 1e9, rng)
        r2, c2 = pick(C_exact, bn, t1, 16, 1e9, rng, exclude_rows=(r1,), exclude_cols=(c1,))
        return [(t1, r1, c1, 26), (t1, r2, c2, 28)]
    if name == "two_in_row":
        r1, c1 = pick(C_exact, bn, t1, 16, 1e9, rng)
        tm, tn = divmod(t1, N // bn)
        row = C_exact[tm * 128 + r1, tn * bn:(tn + 1) * bn]
        c2 = int(next(j for j in range(bn) if j != c1 and abs(row[j]) >= 16))
        return [(t1, r1, c1, 26), (t1, r1, c2, 27)]
    if name == "two_in_col":
        r1, c1 = pick(C_exact, bn, t1, 16, 1e9, rng)
        tm, tn = divmod(t1, N // bn)
        col = C_exact[tm * 128:(tm + 1) * 128, tn * bn + c1]
        r2 = int(next(i for i in range(128) if i != r1 and abs(col[i]) >= 16))
        return [(t1, r1, c1, 29), (t1, r2, c1, 26)]
    if name == "two_tiles":
        t2 = (t1 + 1 + int(rng.integers(0, tiles - 1))) % tiles
        r1, c1 = pick(C_exact, bn, t1, 16, 1e9, rng)
        r2, c2 = pick(C_exact, bn, t2, 16, 1e9, rng)
        return [(t1, r1, c1, 27), (t2, r2, c2, 31)]
    if name == "grey_band":
        r, c = pick(C_exact, bn, t1, 16, 32, rng)
        tm, tn = divmod(t1, N // bn)
        return [(t1, r, c, grey_bit(C_exact[tm * 128 + r, tn * bn + c]))]
    if name == "harmless":
        r, c = pick(C_exact, bn, t1, 16, 32, rng)
        return [(t1, r, c, 0)]                             # 2^-19: below every threshold
    raise ValueError(name)


SCENARIOS = ["single_exponent", "single_to_inf", "two_in_tile", "two_in_row", "two_in_col",
             "two_tiles", "grey_band", "harmless"]
PLANS = {
    "dp_128": dict(tile_n=128, sched="dp", cta_pair=1),
    "sk_128": dict(tile_n=128, sched="sk", cta_pair=1, grid=37),
    "sk2dp_256": dict(tile_n=256, sched="sk2_dp", cta_pair=1, grid=19),
    "pairs_256": dict(tile_n=256, cta_pair=2, sched="sk", grid=12),
    # the library's own plan: idle SMs run the encode pass in the launch and
    # the checksum tiles, split over them, add their segments into the
    # references they zeroed
    "inkernel_128": dict(tile_n=128, cta_pair=1),
    # reference checksums accumulated in the mainloop, several tiles per CTA
    "inloop_128": dict(tile_n=128, cta_pair=1, abft_inloop=2, grid=5),
    "inloop_pairs": dict(tile_n=256, cta_pair=2, abft_inloop=2, grid=4),
}


def _opts(plan, flips):
    kw = dict(PLANS[plan])
    if "grid" in kw:
        kw["grid"] = min(kw["grid"], sms() - sms() % 2)
    o = skgemm.opts_default(abft=1, **kw)
    t, r, c, b = flips[0]
    o.inject_tile, o.inject_row, o.inject_col, o.inject_bit = t, r, c, b
    if len(flips) > 1:
        t, r, c, b = flips[1]
        o.inject2_tile, o.inject2_row, o.inject2_col, o.inject2_bit = t, r, c, b
    return o


# The grey band needs tau_row > tau_col: 128 x 256 tiles only.
CASES = [(plan, name) for plan in PLANS for name in SCENARIOS
         if not (name == "grey_band" and PLANS[plan]["tile_n"] != 256)]


@pytest.mark.parametrize("plan,name", CASES)
def test_decisions_match_oracle(plan, name):
    bn = PLANS[plan]["tile_n"]
    p = integer_problem(seed=7)
    C_exact = reference(p)                   # exact: integer data
    rng = np.random.default_rng(zlib.crc32(f"{plan}/{name}".encode()))
    flips = scenario(name, C_exact, bn, rng)
    expect = oracle_outcomes(p, C_exact, bn, flips)
    if name == "grey_band":
        e = next(iter(expect.values()))
        assert (e["bad_rows"], len(e["bad_cols"]), e["status"]) == ([], 1, ab.UNCORRECTABLE)
    if name in ("two_in_tile", "two_in_row", "two_in_col"):
        assert next(iter(expect.values()))["status"] == ab.UNCORRECTABLE
    opts = _opts(plan, flips)
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    rep = ws.report()
    assert_same_decisions(rep, expect, (M // 128) * (N // bn), C_exact, bn)
    # Corrected and untouched tiles are exact; an uncorrectable tile keeps
    # its faulty values (and is reported) -- compare everything else.
    got = C.cpu().double().numpy()
    tiles_n = N // bn
    mask = np.ones_like(got, dtype=bool)
    for t, e in expect.items():
        if e["status"] == ab.UNCORRECTABLE:
            tm, tn = divmod(t, tiles_n)
            mask[tm * 128:(tm + 1) * 128, tn * bn:(tn + 1) * bn] = False
    if name == "harmless":
        (t, r, c, b), = flips
        tm, tn = divmod(t, tiles_n)
        mask[tm * 128 + r, tn * bn + c] = False
        v = C_exact[tm * 128 + r, tn * bn + c]
        assert got[tm * 128 + r, tn * bn + c] == ab.flip_f32(v, b)
    assert np.array_equal(got[mask], C_exact[mask])


def test_inkernel_plan_is_the_in_launch_encode():
    pl = skgemm.launch_plan(M, N, K, skgemm.opts_default(abft=1, **PLANS["inkernel_128"]))
    assert pl.encode_in_kernel == 1 and pl.side_ctas > 0
    assert pl.side_checksum_ctas == pl.side_ctas   # checksum tiles split over all of them


def test_clean_run_checks_every_tile_with_no_record():
    p = integer_problem(seed=8)
    for plan in PLANS:
        kw = dict(PLANS[plan])
        if "grid" in kw:
            kw["grid"] = min(kw["grid"], sms() - sms() % 2)
        C, ws, st = run(p, skgemm.opts_default(abft=1, **kw))
        assert st == skgemm.OK
        rep = ws.report()
        bn = kw["tile_n"]
        assert rep.tiles_checked == (M // 128) * (N // bn)
        assert rep.detected == 0 and rep.n_records == 0 and rep.status_bits == 0
        # integer data: the checksums match exactly
        assert rep.max_ratio_row == 0.0 and rep.max_ratio_col == 0.0
        assert np.array_equal(C.cpu().double().numpy(), reference(p))


# --------------------------------------------------------------------------- mid-mainloop flips
@pytest.mark.parametrize("plan", ["dp_128", "pairs_256"])
def test_mid_mainloop_flip_exact(plan):
    # The flip lands in TMEM after MAC iteration j of a data-parallel tile,
    # so later iterations add onto the faulty partial sum; the check after
    # the mainloop locates it and restores the exact value.
    p = integer_problem(seed=9)
    C_exact = reference(p)
    bn = PLANS[plan]["tile_n"]
    kw = dict(PLANS[plan])
    kw["sched"] = "dp"
    kw.pop("grid", None)
    rng = np.random.default_rng(3)
    tiles_n = N // bn
    tile = int(rng.integers(0, (M // 128) * tiles_n))
    tm, tn = divmod(tile, tiles_n)
    j = 9                                         # after k = 0 .. 639
    A = p.A.double().numpy()
    Bs = p.B.double().numpy()
    part = A[tm * 128:(tm + 1) * 128, :64 * (j + 1)] @ Bs[tn * bn:(tn + 1) * bn, :64 * (j + 1)].T
    cand = np.argwhere(np.abs(part) >= 64)
    r, c = (int(x) for x in cand[int(rng.integers(0, len(cand)))])
    # exponent bit 24 of |v| in [64, 2^14): the value is multiplied or divided
    # by 4, a change of at least 48, far above both thresholds
    o = skgemm.opts_default(abft=1, inject_tile=tile, inject_row=r, inject_col=c, inject_bit=24,
                            inject_kstep=j, **kw)
    C, ws, st = run(p, o)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.mid_injected == 1
    assert rep.mid_before == part[r, c]           # the partial sum after iteration j
    assert rep.mid_after == ab.flip_f32(part[r, c], 24)
    assert rep.detected == 1 and rep.corrected == 1 and rep.uncorrectable == 0
    rec = gpu_records(rep)[tile]
    assert (rec.row, rec.col, rec.n_bad_rows, rec.n_bad_cols) == (r, c, 1, 1)
    assert rec.after == C_exact[tm * 128 + r, tn * bn + c]
    assert np.array_equal(C.cpu().double().numpy(), C_exact)


def test_mid_mainloop_flip_in_a_peer_partial():
    # Basic Stream-K on few CTAs: the chosen iteration lies in a PEER
    # segment, so the flipped value travels through the partial-tile fixup
    # before the owner's check finds and corrects it.
    m, n, k = 512, 640, 2048
    p = inputs.make_problem(m, n, k, seed=79, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", scale_b=0.02)
    ref = reference(p)
    g = min(7, sms())
    segs = skgemm.schedule_query(m, n, k, 128, 128, 64, g, "sk")
    peer = next(s for s in segs if s[4] == skgemm.ROLE_PEER)
    _, tile, kb0, kb1, _ = peer
    j = (kb0 + kb1) // 2
    tiles_n = (n + 127) // 128
    tm, tn = divmod(tile, tiles_n)
    rng = np.random.default_rng(5)
    r, c = int(rng.integers(0, 128)), int(rng.integers(0, 128))
    # bit 30 of any partial sum: |v| >= 2 drops to ~0, |v| < 2 jumps past 2
    o = skgemm.opts_default(abft=1, tile_n=128, sched="sk", grid=g, cta_pair=1,
                            raster_band=tiles_n, inject_tile=tile, inject_row=r, inject_col=c,
                            inject_bit=30, inject_kstep=j)
    C, ws, st = run(p, o)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.mid_injected == 1
    assert rep.detected == 1 and rep.corrected == 1
    rec = gpu_records(rep)[tile]
    assert (rec.row, rec.col) == (r, c)
    check_full(p, C, ref)


def test_mid_mainloop_argument_checks():
    # An iteration past the tile's last one is an argument error; in-CTA
    # references (whose epilogue warps read every stage while the MMAs run)
    # cannot take a mid-mainloop flip. Both are refused before any launch.
    p = integer_problem(seed=10)
    ws = skgemm.Workspace(skgemm.workspace_size(M, N, K, skgemm.opts_default(abft=1)), "cuda")
    o = skgemm.opts_default(abft=1, inject_tile=0, inject_row=0, inject_col=0, inject_bit=30,
                            inject_kstep=(K + 63) // 64)
    assert skgemm.workspace_size(M, N, K, o) == 0
    C, ws, st = run(p, o, ws=ws)
    assert st == skgemm.ERR_ARG
    o.inject_kstep = 0
    o.abft_local = 2
    small = inputs.make_problem(256, 256, 256, seed=1, in_dtype="bf16", out_dtype="f32",
                                law_a="integer", law_b="integer")
    C, ws, st = run(small, o, ws=ws)
    assert st == skgemm.ERR_UNSUPPORTED


# --------------------------------------------------------------------------- campaign
def test_fault_campaign_1024x1024x8192():
    # The transformer-MLP campaign logic at a reduced size: seeded flips,
    # each drawn until the fault model calls it must-detect, every one
    # detected, located and corrected to within the parity tolerance, and
    # clean launches in between report nothing.
    m, n, k = 1024, 1024, 8192
    p = inputs.make_problem(m, n, k, seed=4, in_dtype="bf16", out_dtype="bf16",
                            law_a="normal", law_b="normal", scale_b=0.02)
    ref = reference(p)
    o = skgemm.opts_default(abft=1)
    bn = skgemm.launch_shape(m, n, k, o)[0]
    A, B = p.A.cuda(), p.B.cuda()
    C = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    ws = skgemm.Workspace(skgemm.workspace_size(m, n, k, o), "cuda")
    sh = torch.cuda.current_stream().cuda_stream
    ref_t = torch.as_tensor(ref, device="cuda")
    base = 1e-3 * math.sqrt(k) * float(p.A.abs().max()) * float(p.B.abs().max())
    tol = base + 2.0 ** -8 * ref_t.abs()

    def launch(opts):
        assert skgemm.gemm(m, n, k, 1.0, A.data_ptr(), k, B.data_ptr(), k, 0.0, C.data_ptr(), n,
                           skgemm.IN_BF16, skgemm.OUT_BF16, 0, 0, opts, ws.ptr, ws.nbytes,
                           sh) == skgemm.OK
        return ws.report(reset=True)

    rng = np.random.default_rng(2024)
    Akm, Bkm = p.A.double().numpy(), p.B.double().numpy()
    must = 0
    for i in range(24):
        bit = int(rng.integers(23, 32))           # exponent and sign bits
        tile, row, col = draw_must_detect(ref, Akm, Bkm, 1.0, k, m, n, bn, bit,
                                          seed=int(rng.integers(0, 2 ** 31)))
        oi = skgemm.opts_default(abft=1, inject_tile=tile, inject_row=row, inject_col=col,
                                 inject_bit=bit)
        rep = launch(oi)
        must += 1
        assert rep.detected == 1 and rep.corrected == 1 and rep.uncorrectable == 0, i
        rec = gpu_records(rep)[tile]
        assert (rec.row, rec.col, rec.injected) == (row, col, 1)
        assert bool(((C.double() - ref_t).abs() <= tol).all())
        rep = launch(o)                            # a clean launch after each fault
        assert rep.detected == 0 and rep.status_bits == 0
        assert bool(((C.double() - ref_t).abs() <= tol).all())
    assert must >= 20


# --------------------------------------------------------------------------- device trace
def _trace(p, opts, ctas):
    trace = torch.zeros(ctas * skgemm.TRACE_STRIDE, dtype=torch.int32, device="cuda")
    opts.trace = trace.data_ptr()
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    torch.cuda.synchronize()
    tr = trace.cpu().numpy().reshape(ctas, skgemm.TRACE_STRIDE)
    out = []
    for x in range(ctas):
        cnt = int(tr[x, 0])
        out.append([tuple(int(v) for v in tr[x, 1 + 4 * i: 5 + 4 * i]) for i in range(cnt)])
    return out, C, ws


def _expected(m, n, k, bm, bn, g, mode, t_ck=0, g_ck=0, g_ckt=None):
    """Per schedule CTA: the side-tile region (t_ck full-k tiles split evenly
    over the g CTAs, or over the first g_ckt of g_ck extra CTAs), then the
    output schedule, as the simulator gives them; side tiles carry the
    numbers -t_ck .. -1."""
    ipt = -(-k // 64)
    out = [[] for _ in range(g + g_ck)]
    if t_ck:
        total = t_ck * ipt
        split = (g_ckt if g_ckt is not None else g_ck) if g_ck else g
        base = g if g_ck else 0
        for x in range(split):
            b, e = ss.sk_range(x, total, split)
            out[base + x] += [(s.tile, s.k_iter_begin, s.k_iter_end, s.role)
                              for s in ss.walk_range(base + x, b, e, ipt, tile_offset=-t_ck)]
    sched = ss.schedule(m, n, k, bm, bn, 64, g, mode)
    for x in range(g):
        out[x] += [(s.tile, s.k_iter_begin, s.k_iter_end, s.role) for s in sched[x]]
    return out


@pytest.mark.parametrize("mode", ["sk", "sk2_dp", "dp_sk1"])
def test_trace_cta_pairs(mode):
    # CTA pairs run the page's schedule over 256-row tiles with one schedule
    # slot per cluster: both CTAs of cluster u walk slot u's segments.
    m, n, k = 1000, 1300, 520
    p = inputs.make_problem(m, n, k, seed=41, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal")
    g = min(10, sms() // 2)
    got, C, _ = _trace(p, skgemm.opts_default(cta_pair=2, tile_n=256, sched=mode, grid=2 * g,
                                              raster_band=1000), 2 * g)
    want = _expected(-(-m // 256) * 256, n, k, 256, 256, g, mode)
    for x in range(2 * g):
        assert got[x] == want[x // 2], x
    check_full(p, C)


@pytest.mark.parametrize("pair", [1, 2])
def test_trace_abft_side_tiles_split(pair):
    # ABFT with fused checksum tiles on a fixed grid: every CTA first runs
    # its even share of the side-tile region, then its output schedule.
    m, n, k = 640, 896, 704
    p = inputs.make_problem(m, n, k, seed=42, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal")
    g = min(12, sms() // 2)
    ctas = g * pair
    kw = dict(abft=1, sched="sk", grid=ctas, raster_band=1000)
    if pair == 2:
        kw.update(cta_pair=2, tile_n=256)
        t_ck = (-(-m // 128) + 1) // 2 + (-(-n // 128) + 1) // 2
        want = _expected(-(-m // 256) * 256, n, k, 256, 256, g, "sk", t_ck)
    else:
        kw.update(cta_pair=1, tile_n=128)
        t_ck = -(-m // 128) + -(-n // 128)
        want = _expected(m, n, k, 128, 128, g, "sk", t_ck)
    plan = skgemm.launch_plan(m, n, k, skgemm.opts_default(**kw))
    assert plan.fused_checksums == 1 and plan.side_ctas == 0
    got, C, ws = _trace(p, skgemm.opts_default(**kw), ctas)
    for x in range(ctas):
        assert got[x] == want[x // pair], x
    check_full(p, C)
    assert ws.report().detected == 0


def test_trace_abft_dedicated_side_ctas():
    # A small bf16 ABFT call leaves SMs idle: extra CTAs run the side tiles
    # (after the in-kernel encode pass), split evenly over them.
    m = n = k = 1024
    p = inputs.make_problem(m, n, k, seed=43, in_dtype="bf16", out_dtype="bf16",
                            law_a="normal", law_b="normal")
    o = skgemm.opts_default(abft=1)
    plan = skgemm.launch_plan(m, n, k, o)
    assert plan.side_ctas > 0 and plan.cta_pair == 1 and plan.encode_in_kernel == 1
    ctas = plan.ctas + plan.side_ctas
    got, C, ws = _trace(p, o, ctas)
    t_ck = m // 128 + n // 128
    names = {v: kk for kk, v in skgemm.SCHED_NAMES.items()}
    # the output schedule's raster is banded; the trace holds schedule tile
    # indices, so the simulator's row-major numbering applies to them
    want = _expected(m, n, k, 128, plan.tile_n, plan.ctas, names[plan.sched], t_ck,
                     plan.side_ctas, plan.side_checksum_ctas)
    assert got == want
    check_full(p, C)
    assert ws.report().detected == 0


# --------------------------------------------------------------------------- workspace reuse
HEADER_BYTES = 16384   # workspace header, report and flags: the part that must start at zero


def _sequence():
    """Calls of different shapes, input types and options, in a row."""
    return [
        (inputs.make_problem(2048, 2048, 1024, seed=51, in_dtype="bf16", out_dtype="bf16",
                             law_a="normal", law_b="normal"), dict()),
        (inputs.make_problem(700, 900, 520, seed=52, in_dtype="f16", out_dtype="f16",
                             law_a="uniform", law_b="uniform", alpha=1.5, beta=0.5),
         dict(abft=1, grid=16, tile_n=128)),
        (inputs.make_problem(1000, 1300, 520, seed=53, in_dtype="bf16", out_dtype="f32",
                             law_a="normal", law_b="normal"), dict(abft=1, cta_pair=2)),
        (inputs.make_problem(1536, 640, 2048, seed=54, in_dtype="f16", out_dtype="f32",
                             law_a="normal", law_b="normal"), dict(abft=1)),
        (inputs.make_problem(384, 4096, 704, seed=55, in_dtype="bf16", out_dtype="bf16",
                             law_a="normal", law_b="normal"), dict(sched="sk", tile_n=256)),
        # split reductions whose owners keep their partial in bank 2 (the
        # storage the ABFT calls use for their checksum tiles), 256 and 64 wide
        (inputs.make_problem(640, 512, 8192, seed=56, in_dtype="f16", out_dtype="f16",
                             law_a="uniform", law_b="uniform", alpha=1.5, beta=0.5),
         dict(sched="sk", tile_n=256, grid=17)),
        (inputs.make_problem(1536, 640, 2048, seed=57, in_dtype="bf16", out_dtype="f32",
                             law_a="normal", law_b="normal"), dict(abft=1, tile_n=128)),
        (inputs.make_problem(640, 512, 8192, seed=58, in_dtype="bf16", out_dtype="f32",
                             law_a="normal", law_b="normal"), dict(sched="sk", tile_n=64, grid=70)),
        (inputs.make_problem(2048, 2048, 1024, seed=51, in_dtype="bf16", out_dtype="bf16",
                             law_a="normal", law_b="normal"), dict()),
    ]


def test_workspace_reused_across_shapes_and_options():
    # One workspace serves a sequence of calls whose layouts differ (grid,
    # tile width, ABFT regions, CTA pairs, input type). Before every call the
    # part after the fixed header is overwritten with small integers -- the
    # values a stale flag, counter or tile scale would hold -- so nothing may
    # depend on what an earlier call left there.
    seq = _sequence()
    sizes = [skgemm.workspace_size(p.m, p.n, p.k, skgemm.opts_default(**kw)) for p, kw in seq]
    ws = skgemm.Workspace(max(sizes), "cuda")
    words = (ws.nbytes - HEADER_BYTES) // 4
    junk = (torch.arange(words, device="cuda", dtype=torch.int32) % 7) + 1
    for i, (p, kw) in enumerate(seq):
        ws.buf[HEADER_BYTES:HEADER_BYTES + 4 * words].view(torch.int32).copy_(junk)
        junk = junk.roll(1)
        opts = skgemm.opts_default(**kw)
        C, ws, st = run(p, opts, ws=ws)
        assert st == skgemm.OK, i
        rep = ws.report(reset=True)
        assert rep.status_bits == 0 and rep.detected == 0, (i, rep.status_bits)
        if kw.get("abft"):
            assert rep.tiles_checked > 0 and rep.max_ratio_row < 0.1 and rep.max_ratio_col < 0.1
        if p.m * p.n * p.k <= 2 ** 31:
            check_full(p, C)
        else:
            from gpu_util import check_sampled
            check_sampled(p, C, seed=i)


# --------------------------------------------------------------------------- in-loop checksums
@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("shape", [(300, 200, 200), (1000, 1300, 520), (1024, 1024, 1024),
                                   (129, 3000, 4104), (2048, 2048, 2048)])
def test_inloop_checksums_clean(shape, dtype, pair):
    # The checksum MMAs run in the output tiles' mainloop: every tile
    # verified, no false positive, ragged m, n and k, fp16 encodings scaled
    # per tile, one or several tiles per CTA.
    m, n, k = shape
    p = inputs.make_problem(m, n, k, seed=m + n + k, in_dtype=dtype, out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=0.75, beta=0.5)
    bn = 256 if pair == 2 else 128
    for grid in (0, 4):
        o = skgemm.opts_default(abft=1, abft_inloop=2, cta_pair=pair, tile_n=bn, grid=grid)
        plan = skgemm.launch_plan(m, n, k, o)
        assert plan.inloop_checksums == 1 and plan.fused_checksums == 0
        assert plan.sched == skgemm.SCHED_DP and plan.side_ctas == 0
        ws = None
        for _ in range(2):
            C, ws, st = run(p, o, ws=ws)
            assert st == skgemm.OK
            check_full(p, C)
            rep = ws.report(reset=True)
            assert rep.detected == 0 and rep.status_bits == 0
            assert rep.tiles_checked == -(-m // 128) * -(-n // bn)
            assert rep.max_ratio_row < 0.1 and rep.max_ratio_col < 0.1


def test_inloop_mid_mainloop_flip():
    # A flip inside the mainloop of an in-loop-checksum launch: the checksum
    # MMAs see the clean operands, the accumulator the faulty partial sum.
    p = integer_problem(seed=11)
    C_exact = reference(p)
    for kw in (PLANS["inloop_128"], PLANS["inloop_pairs"]):
        bn = kw["tile_n"]
        tiles_n = N // bn
        tile = 5
        tm, tn = divmod(tile, tiles_n)
        r, c, j = 77, 100, 3
        o = skgemm.opts_default(abft=1, inject_tile=tile, inject_row=r, inject_col=c,
                                inject_bit=30, inject_kstep=j, **kw)
        C, ws, st = run(p, o)
        assert st == skgemm.OK
        rep = ws.report()
        assert rep.mid_injected == 1 and rep.detected == 1 and rep.corrected == 1
        rec = gpu_records(rep)[tile]
        assert (rec.row, rec.col) == (r, c)
        assert rec.after == C_exact[tm * 128 + r, tn * bn + c]
        assert np.array_equal(C.cpu().double().numpy(), C_exact)
