"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Floating point is compared under the parity tolerance of gpu_util; the
schedule (device trace) and ABFT decisions are compared exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import abft_ref as ab
from oracle import schedule_sim as ss
from stream_decomposition_abft_gb300 import _build, inputs, skgemm

from gpu_util import (check_full, check_sampled, check_checksum_probe, draw_must_detect,
                      reference, run)

pytestmark = pytest.mark.gpu

MODES = ["dp", "sk", "dp_sk1", "sk2_dp"]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    skgemm.lib()


def sms():
    return skgemm.device_sm_count()


def device_trace(p, opts_kw, g):
    trace = torch.zeros(g * skgemm.TRACE_STRIDE, dtype=torch.int32, device="cuda")
    opts = skgemm.opts_default(grid=g, trace=trace.data_ptr(), **opts_kw)
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    torch.cuda.synchronize()
    tr = trace.cpu().numpy().reshape(g, skgemm.TRACE_STRIDE)
    rows = []
    for x in range(g):
        cnt = int(tr[x, 0])
        for i in range(cnt):
            t, b, e, role = tr[x, 1 + 4 * i: 5 + 4 * i]
            rows.append((x, int(t), int(b), int(e), int(role)))
    return rows, C, ws


# --------------------------------------------------------------------------- example
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("g", [4, 148])
def test_example_384_parity_and_trace(mode, g):
    g = min(g, sms())
    p = inputs.example_384()
    ref = reference(p)
    for tile_n in (64, 128, 256):
        rows, C, ws = device_trace(p, dict(sched=mode, tile_n=tile_n), g)
        check_full(p, C, ref)
        want = ss.flatten(ss.schedule(384, 384, 128, 128, tile_n, 64, g, mode=mode))
        assert rows == want
        rep = ws.report()
        assert rep.status_bits == 0 and rep.launches == 1


# --------------------------------------------------------------------------- shapes
SMALL = [
    (300, 500, 200, "bf16", "bf16"),
    (129, 257, 64, "f16", "f32"),
    (128, 128, 64, "bf16", "f32"),
    (1, 1, 8, "f16", "f16"),
    (17, 33, 1000, "bf16", "bf16"),
    (640, 768, 1536, "f16", "f16"),
    (1000, 1300, 520, "bf16", "f32"),
]


@pytest.mark.parametrize("shape", SMALL)
@pytest.mark.parametrize("mode", MODES)
def test_small_shapes(shape, mode):
    m, n, k, dt_in, dt_out = shape
    p = inputs.make_problem(m, n, k, seed=m * 7 + n, in_dtype=dt_in, out_dtype=dt_out,
                            law_a="normal", law_b="uniform", alpha=0.75, beta=-0.5)
    ref = reference(p)
    for tile_n in (64, 128, 256):
        for g in (7, sms()):
            C, ws, st = run(p, skgemm.opts_default(sched=mode, tile_n=tile_n, grid=g))
            assert st == skgemm.OK
            check_full(p, C, ref)


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("tile_n,pair", [(64, 1), (128, 1), (256, 1), (256, 2)])
def test_beta_chunks_of_earlier_tiles(out, tile_n, pair):
    # beta != 0 on tiles that are not a CTA's last (few CTAs, several tiles
    # each): every staging chunk's C0 rows are fetched one chunk ahead, and
    # chunks that lie wholly past n (n = 300: the second column tile of a
    # 256-wide tile keeps 44 of its columns) are neither fetched nor stored.
    p = inputs.make_problem(300, 300, 192, seed=95 + tile_n, in_dtype="bf16", out_dtype=out,
                            law_a="normal", law_b="uniform", alpha=-1.25, beta=0.75)
    ref = reference(p)
    for mode, g in (("dp", 2 * pair), ("sk", 2 * pair), ("sk2_dp", 3 * pair)):
        C, ws, st = run(p, skgemm.opts_default(sched=mode, tile_n=tile_n, cta_pair=pair,
                                               grid=g))
        assert st == skgemm.OK
        check_full(p, C, ref)
        assert ws.report().status_bits == 0


@pytest.mark.parametrize("k", [1, 7, 65, 100, 129])
def test_ragged_k_with_padded_ld(k):
    # k not a multiple of 8 needs a padded row stride (TMA stride rule);
    # the tail of the last MAC iteration is zero-filled by the TMA engine.
    ld = (k + 7) // 8 * 8
    p = inputs.make_problem(200, 300, k, seed=k, in_dtype="f16", out_dtype="f32",
                            law_a="uniform", law_b="uniform")
    ref = reference(p)
    C, ws, st = run(p, skgemm.opts_default(sched="sk", grid=min(40, sms())), lda=ld, ldb=ld)
    assert st == skgemm.OK
    check_full(p, C, ref)
    if k % 8:
        _, _, st = run(p, skgemm.opts_default())
        assert st == skgemm.ERR_UNSUPPORTED


def test_k_zero_scales_c():
    p = inputs.make_problem(100, 60, 0, seed=3, in_dtype="bf16", out_dtype="f32", beta=2.0)
    C, ws, st = run(p, skgemm.opts_default())
    assert st == skgemm.OK
    assert torch.equal(C.cpu(), (2.0 * p.C0.float()))


def test_integer_inputs_exact():
    # Integer-valued inputs: every product and partial sum is exact in fp32,
    # so the GPU must equal the oracle exactly, on every schedule.
    p = inputs.make_problem(512, 640, 768, seed=21, in_dtype="bf16", out_dtype="f32",
                            law_a="integer", law_b="integer")
    ref = reference(p)
    for mode in MODES:
        C, ws, st = run(p, skgemm.opts_default(sched=mode, grid=min(37, sms())))
        assert st == skgemm.OK
        assert np.array_equal(C.cpu().double().numpy(), ref), mode


# --------------------------------------------------------------------------- Stream-K fixup
@pytest.mark.parametrize("g", [2, 3, 16, 64, 148])
def test_many_peers_per_tile(g):
    # Basic Stream-K on few tiles and many CTAs: each owner accumulates
    # several peers (the page's Fig. 9 case: one tile, deep k).
    g = min(g, sms())
    p = inputs.make_problem(256, 256, 8192, seed=g, in_dtype="f16", out_dtype="f32",
                            law_a="uniform", law_b="uniform", alpha=1.5, beta=0.5)
    ref = reference(p)
    rows, C, ws = device_trace(p, dict(sched="sk", tile_n=128), g)
    check_full(p, C, ref)
    assert rows == ss.flatten(ss.schedule(256, 256, 8192, 128, 128, 64, g, mode="sk"))


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("pair", [1, 2])
def test_shared_tile_reduction(out, pair):
    # Deep-k tiles split over many CTAs that all end their ranges in them
    # (grids that divide the iterations evenly, so every owner's range starts
    # at its tile): each of those CTAs stores its partial and reduces a share
    # of the tile (plain stores of C, alpha / beta with C0, ragged m and n, a
    # CTA-pair half past m).
    g = 128 if pair == 2 else 48
    if g > sms():
        pytest.skip("needs more SMs")
    p = inputs.make_problem(300, 200, 16384, seed=11 + pair, in_dtype="f16", out_dtype=out,
                            law_a="uniform", law_b="uniform", alpha=1.5, beta=0.5)
    opts = skgemm.opts_default(sched="sk", tile_n=256 if pair == 2 else 128, grid=g,
                               cta_pair=pair)
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    check_full(p, C)
    assert ws.report().status_bits == 0


# Split reduction (no ABFT, single CTAs): a Stream-K tile that 2 .. BLK_N /
# (staging chunk) CTAs end their ranges in is finished by those CTAs
# together, each folding the others' partials into its own columns; owners
# whose range began in an earlier tile keep that partial in bank 2.
SPLIT_CASES = [(256, 17, "sk"), (128, 37, "sk"), (64, 70, "sk"), (256, 8, "dp_sk1"),
               (128, 13, "sk2_dp")]


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("case", SPLIT_CASES)
def test_split_reduction(out, case):
    tile_n, g, mode = case
    g = min(g, sms())
    for (m, n, k) in ((640, 512, 8192), (600, 500, 8000)):
        p = inputs.make_problem(m, n, k, seed=60 + g, in_dtype="f16", out_dtype=out,
                                law_a="uniform", law_b="uniform", alpha=1.5, beta=0.5)
        ref = reference(p)
        rows, C, ws = device_trace(p, dict(sched=mode, tile_n=tile_n), g)
        check_full(p, C, ref)
        assert rows == ss.flatten(ss.schedule(m, n, k, 128, tile_n, 64, g, mode=mode))
        assert ws.report().status_bits == 0


@pytest.mark.parametrize("a_layout,b_layout", [(1, 1), (0, 1)])
def test_split_reduction_mn_major(a_layout, b_layout):
    p = inputs.make_problem(640, 512, 8192, seed=71, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=1.5, beta=0.5,
                            a_layout=a_layout, b_layout=b_layout)
    C, ws, st = run(p, skgemm.opts_default(sched="sk", tile_n=256, grid=min(17, sms())))
    assert st == skgemm.OK
    check_full(p, C)


def test_split_reduction_injection():
    # A flip in a column that the second part of a split tile stores reaches
    # C at that element only.
    p = inputs.make_problem(640, 512, 8192, seed=72, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal")
    ref = reference(p)
    g = min(17, sms())
    sch = ss.schedule(640, 512, 8192, 128, 256, 64, g, mode="sk")
    op = ss.owners_and_peers(sch)
    # a tile covered by three CTAs: the owner and the middle one end in it
    tile = next(t for t, (o, peers) in sorted(op.items()) if len(peers) == 2)
    col = 200  # in the last quarter: the middle part's columns
    opts = skgemm.opts_default(sched="sk", tile_n=256, grid=g, inject_tile=tile, inject_row=5,
                               inject_col=col, inject_bit=30)
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    got = C.cpu().double().numpy()
    tm, tn = divmod(tile, 2)
    bad = (tm * 128 + 5, tn * 256 + col)
    diff = np.abs(got - ref)
    assert not (diff[bad] < 1e-3)
    diff[bad] = 0
    assert diff.max() < 1e-2


def test_split_reduction_timeout_reports_and_returns():
    # The middle part of a split tile skips its Signal: the owner part's
    # bounded wait runs out, the launch records SKG_ERR_FIXUP_TIMEOUT, and
    # the device stays usable.
    p = inputs.make_problem(640, 512, 8192, seed=73, in_dtype="bf16", out_dtype="f32")
    g = min(17, sms())
    sch = ss.schedule(640, 512, 8192, 128, 256, 64, g, mode="sk")
    op = ss.owners_and_peers(sch)
    middle = next(peers[0] for t, (o, peers) in sorted(op.items()) if len(peers) == 2)
    opts = skgemm.opts_default(sched="sk", grid=g, tile_n=256, timeout_ns=50_000_000,
                               test_drop_signal=middle + 1)
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.status_bits & (1 << skgemm.ERR_FIXUP_TIMEOUT)
    assert rep.timeouts >= 1
    p2 = inputs.make_problem(640, 512, 8192, seed=74, in_dtype="bf16", out_dtype="f32")
    C2, ws2, st2 = run(p2, skgemm.opts_default(sched="sk", grid=g, tile_n=256))
    assert st2 == skgemm.OK
    check_full(p2, C2)
    assert ws2.report().status_bits == 0


def test_shared_tile_reduction_timeout_reports_and_returns():
    # One CTA of a shared-reduction tile skips its Signal: every other CTA of
    # the tile runs out its bounded flag wait; the launch records
    # SKG_ERR_FIXUP_TIMEOUT and the device stays usable.
    p = inputs.make_problem(256, 256, 16384, seed=22, in_dtype="bf16", out_dtype="f32")
    g = min(64, sms())
    rows = ss.flatten(ss.schedule(256, 256, 16384, 128, 128, 64, g, mode="sk"))
    peer = next(r[0] for r in rows if r[4] == ss.PEER)
    opts = skgemm.opts_default(sched="sk", grid=g, tile_n=128, timeout_ns=50_000_000,
                               test_drop_signal=peer + 1)
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.status_bits & (1 << skgemm.ERR_FIXUP_TIMEOUT)
    assert rep.timeouts >= 1
    p2 = inputs.make_problem(256, 256, 16384, seed=23, in_dtype="bf16", out_dtype="f32")
    C2, ws2, st2 = run(p2, skgemm.opts_default(sched="sk", grid=g, tile_n=128))
    assert st2 == skgemm.OK
    check_full(p2, C2)
    assert ws2.report().status_bits == 0


def test_shared_tile_reduction_injection():
    # A bit flipped in one accumulator of a shared-reduction tile reaches C
    # at that element only (no ABFT).
    p = inputs.make_problem(256, 256, 16384, seed=21, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal")
    ref = reference(p)
    opts = skgemm.opts_default(sched="sk", tile_n=128, grid=min(64, sms()), inject_tile=2,
                               inject_row=37, inject_col=101, inject_bit=30)
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    got = C.cpu().double().numpy()
    bad = (128 + 37, 101)
    diff = np.abs(got - ref)
    assert not (diff[bad] < 1e-3)
    diff[bad] = 0
    assert diff.max() < 1e-2


def test_workspace_reuse_across_launches():
    # Flags carry the launch epoch: back-to-back launches on one workspace
    # never read a stale partial.
    opts = skgemm.opts_default(sched="sk", grid=sms(), tile_n=128)
    ws = None
    for i in range(6):
        p = inputs.make_problem(384, 512, 2048, seed=100 + i, in_dtype="bf16", out_dtype="f32",
                                law_a="normal", law_b="normal")
        C, ws, st = run(p, opts, ws=ws)
        assert st == skgemm.OK
        check_full(p, C)
    assert ws.report().launches == 6


def test_fixup_timeout_reports_and_returns():
    # A CTA skips its Signal, so its owner's bounded wait runs out: the
    # launch must end with SKG_ERR_FIXUP_TIMEOUT recorded, and the context
    # stay usable.
    p = inputs.make_problem(256, 256, 4096, seed=5, in_dtype="bf16", out_dtype="f32")
    rows = ss.flatten(ss.schedule(256, 256, 4096, 128, 128, 64, 8, mode="sk"))
    peer = next(r[0] for r in rows if r[4] == ss.PEER)
    opts = skgemm.opts_default(sched="sk", grid=8, tile_n=128, timeout_ns=50_000_000,
                               test_drop_signal=peer + 1)
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.status_bits & (1 << skgemm.ERR_FIXUP_TIMEOUT)
    assert rep.timeouts >= 1
    # the device still works
    p2 = inputs.make_problem(128, 128, 128, seed=6, in_dtype="bf16", out_dtype="f32")
    C2, ws2, st2 = run(p2, skgemm.opts_default())
    assert st2 == skgemm.OK
    check_full(p2, C2)
    assert ws2.report().status_bits == 0


# --------------------------------------------------------------------------- 64-wide tiles
# The small-tile configuration (BLK_N = 64, GEMMs without ABFT): the same
# persistent kernel and schedule with 128 x 64 tiles.
@pytest.mark.parametrize("g", [3, 16, 148])
def test_small_tiles_many_peers(g):
    g = min(g, sms())
    p = inputs.make_problem(256, 200, 8192, seed=30 + g, in_dtype="bf16", out_dtype="f32",
                            law_a="uniform", law_b="uniform", alpha=1.5, beta=0.5)
    ref = reference(p)
    for mode in MODES:
        rows, C, ws = device_trace(p, dict(sched=mode, tile_n=64), g)
        check_full(p, C, ref)
        assert rows == ss.flatten(ss.schedule(256, 200, 8192, 128, 64, 64, g, mode=mode))
        assert ws.report().status_bits == 0


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
def test_small_tiles_shared_reduction(out):
    # Deep-k 128 x 64 tiles split evenly over many CTAs: the shared
    # reduction (every covering CTA reduces a share of the tile).
    g = min(96, sms())
    p = inputs.make_problem(300, 130, 16384, seed=41, in_dtype="f16", out_dtype=out,
                            law_a="uniform", law_b="uniform", alpha=1.5, beta=0.5)
    C, ws, st = run(p, skgemm.opts_default(sched="sk", tile_n=64, grid=g))
    assert st == skgemm.OK
    check_full(p, C)
    assert ws.report().status_bits == 0


@pytest.mark.parametrize("a_layout,b_layout", [(1, 0), (0, 1), (1, 1)])
def test_small_tiles_mn_major(a_layout, b_layout):
    p = inputs.make_problem(384, 200, 1000, seed=42, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", a_layout=a_layout,
                            b_layout=b_layout)
    ref = reference(p)
    for mode, g in (("dp", 12), ("sk", 40), ("sk2_dp", 7)):
        C, ws, st = run(p, skgemm.opts_default(sched=mode, tile_n=64, grid=min(g, sms())))
        assert st == skgemm.OK
        check_full(p, C, ref)


def test_small_tiles_workspace_shared_with_wider_tiles():
    # One workspace for 64-, 128- and 256-wide Stream-K launches of several
    # shapes in a row (the flags sit at fixed offsets and carry the epoch).
    shapes = [(256, 256, 4096), (384, 200, 2048), (128, 520, 3000)]
    size = max(skgemm.workspace_size(m, n, k, skgemm.opts_default(sched="sk", tile_n=t, grid=g))
               for (m, n, k) in shapes for t in (64, 128, 256) for g in (37, sms()))
    ws = skgemm.Workspace(size, "cuda")
    launches = 0
    for i, (m, n, k) in enumerate(shapes):
        for t in (64, 128, 256, 64):
            p = inputs.make_problem(m, n, k, seed=50 + 7 * i + t, in_dtype="bf16", out_dtype="f32",
                                    law_a="normal", law_b="normal")
            g = 37 if t != 256 else sms()
            C, _, st = run(p, skgemm.opts_default(sched="sk", tile_n=t, grid=g), ws=ws)
            assert st == skgemm.OK
            check_full(p, C)
            launches += 1
    rep = ws.report()
    assert rep.status_bits == 0 and rep.launches == launches


def test_small_tiles_chosen_for_tiny_shapes():
    # The grid-size model takes 64-wide tiles for small GEMMs without ABFT,
    # never with ABFT, and keeps wide tiles for large ones.
    assert skgemm.launch_plan(256, 256, 384, skgemm.opts_default()).tile_n == 64
    assert skgemm.launch_plan(256, 256, 384, skgemm.opts_default(abft=1)).tile_n != 64
    assert skgemm.launch_plan(4096, 4096, 4096, skgemm.opts_default()).tile_n != 64
    p = inputs.make_problem(256, 256, 384, seed=43, in_dtype="f16", out_dtype="f16",
                            law_a="normal", law_b="normal")
    C, ws, st = run(p, skgemm.opts_default())
    assert st == skgemm.OK
    check_full(p, C)


# --------------------------------------------------------------------------- workloads
def test_hostile_shapes():
    for i, (m, n, k) in enumerate(inputs.HOSTILE_SHAPES):
        p = inputs.hostile(m, n, k)
        for tile_n in (128, 256):
            C, ws, st = run(p, skgemm.opts_default(tile_n=tile_n))
            assert st == skgemm.OK
            if m * n * k <= 2 ** 33:
                check_full(p, C)
            else:
                check_sampled(p, C, seed=i)
            check_checksum_probe(p, C)
            assert ws.report().status_bits == 0


@pytest.mark.parametrize("size", inputs.SQUARE_SIZES)
def test_square_sweep_abft(size):
    p = inputs.square(size)
    C, ws, st = run(p, skgemm.opts_default(abft=1))
    assert st == skgemm.OK
    check_sampled(p, C, seed=size)
    check_checksum_probe(p, C)
    rep = ws.report()
    tile_n, _, _ = skgemm.launch_shape(size, size, size, skgemm.opts_default(abft=1))
    tiles = ((size + 127) // 128) * ((size + tile_n - 1) // tile_n)
    assert rep.detected == 0 and rep.status_bits == 0, "false positive on a clean run"
    assert rep.tiles_checked == tiles
    assert rep.max_ratio_row < 0.1 and rep.max_ratio_col < 0.1, \
        (rep.max_ratio_row, rep.max_ratio_col)


@pytest.mark.parametrize("shape", inputs.MLP_SHAPES)
def test_mlp_shapes_abft(shape):
    p = inputs.mlp(*shape)
    C, ws, st = run(p, skgemm.opts_default(abft=1))
    assert st == skgemm.OK
    check_sampled(p, C, seed=sum(shape), count=512, rows=4, cols=4)
    rep = ws.report()
    assert rep.detected == 0 and rep.status_bits == 0
    assert rep.max_ratio_row < 0.1 and rep.max_ratio_col < 0.1


def test_random_shapes_subset():
    shapes = inputs.random_shapes(1000)
    for idx in range(0, 1000, 50):
        m, n, k = shapes[idx]
        p = inputs.random_problem(m, n, k, idx)
        C, ws, st = run(p, skgemm.opts_default())
        assert st == skgemm.OK
        check_sampled(p, C, seed=idx, count=128, rows=2, cols=2)


# --------------------------------------------------------------------------- ABFT faults
def _inject(p, opts_kw, tile, row, col, bit):
    opts = skgemm.opts_default(abft=1, inject_tile=tile, inject_row=row, inject_col=col,
                               inject_bit=bit, **opts_kw)
    return run(p, opts)


@pytest.mark.parametrize("mode", ["dp", "sk", "sk2_dp"])
@pytest.mark.parametrize("bit", [30, 29, 26, 23, 31])
def test_injected_fault_detected_located_corrected(mode, bit):
    p = inputs.make_problem(512, 640, 1024, seed=77, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", scale_b=0.02)
    ref = reference(p)
    # A position where this bit is must-detect (seeded draw: never skips).
    tile, row, col = draw_must_detect(ref, p.A.double().numpy(), p.B.double().numpy(), p.alpha,
                                      p.k, 512, 640, 128, bit, seed=bit)
    C, ws, st = _inject(p, dict(sched=mode, tile_n=128, grid=min(64, sms())), tile, row, col, bit)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.detected == 1 and rep.corrected == 1 and rep.uncorrectable == 0
    rec = rep.records[0]
    assert (rec.tile, rec.row, rec.col, rec.injected) == (tile, row, col, 1)
    # the flip is exactly one bit of the GPU's own pre-fault value
    assert ab.flip_f32(rec.clean_value, bit) == rec.before or \
        (np.isnan(rec.before) and np.isnan(ab.flip_f32(rec.clean_value, bit)))
    check_full(p, C, ref)   # corrected output is within parity tolerance


@pytest.mark.parametrize("shape", [(300, 200, 200), (1000, 1300, 520), (1024, 1024, 1024),
                                   (129, 3000, 4104)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_abft_local_matches_fused(shape, dtype):
    # Reference checksums formed inside the CTAs (abft_local = 2) against the
    # encode pass + checksum GEMMs (abft_local = 1): the same output bits (the
    # same MMAs and epilogue), no false positive, every tile checked, ragged
    # m, n and k.
    m, n, k = shape
    tiles = ((m + 127) // 128) * ((n + 127) // 128)
    if tiles > sms():
        pytest.skip("more tiles than SMs")
    p = inputs.make_problem(m, n, k, seed=m + k, in_dtype=dtype, out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=0.5, beta=1.5)
    local = skgemm.opts_default(abft=1, abft_local=2)
    assert skgemm.launch_plan(m, n, k, local).local_checksums == 1
    ws = None
    for _ in range(2):
        C1, ws, st = run(p, local, ws=ws)
        assert st == skgemm.OK
        check_full(p, C1)
        rep = ws.report(reset=True)
        assert rep.detected == 0 and rep.status_bits == 0
        assert rep.tiles_checked == tiles
        assert rep.max_ratio_row < 0.1 and rep.max_ratio_col < 0.1
    C2, ws2, st2 = run(p, skgemm.opts_default(abft=1, abft_local=1, tile_n=128, sched="dp"))
    assert st2 == skgemm.OK and ws2.report().detected == 0
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("bit", [30, 28])
def test_abft_local_injection(dtype, bit):
    # A flipped accumulator bit under in-CTA references is detected, located
    # and corrected as under the fused checksum path.
    p = inputs.make_problem(512, 640, 1024, seed=78, in_dtype=dtype, out_dtype="f32",
                            law_a="normal", law_b="normal", scale_b=0.02)
    ref = reference(p)
    tile, row, col = draw_must_detect(ref, p.A.double().numpy(), p.B.double().numpy(), p.alpha,
                                      p.k, 512, 640, 128, bit, seed=100 + bit)
    assert skgemm.launch_plan(512, 640, 1024,
                              skgemm.opts_default(abft=1, abft_local=2)).local_checksums == 1
    C, ws, st = _inject(p, dict(abft_local=2), tile, row, col, bit)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.detected == 1 and rep.corrected == 1 and rep.uncorrectable == 0
    rec = rep.records[0]
    assert (rec.tile, rec.row, rec.col, rec.injected) == (tile, row, col, 1)
    check_full(p, C, ref)


def test_injection_without_abft_corrupts_output():
    p = inputs.make_problem(256, 256, 256, seed=9, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal")
    ref = reference(p)
    opts = skgemm.opts_default(inject_tile=1, inject_row=5, inject_col=7, inject_bit=30)
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    got = C.cpu().double().numpy()
    bn = skgemm.launch_shape(256, 256, 256, opts)[0]
    tm, tnn = divmod(1, 256 // bn)
    bad = (tm * 128 + 5, tnn * bn + 7)
    diff = np.abs(got - ref)
    assert not (diff[bad] < 1e-3)       # the flipped value reached C
    diff[bad] = 0
    assert diff.max() < 1e-2            # and nothing else changed


@pytest.mark.parametrize("band", [1, 3, 5, 1000])
def test_raster_bands(band):
    # Every banded tile order covers each output tile exactly once, ragged
    # last band included (band >= tiles_n is the row-major order).
    p = inputs.make_problem(1000, 1900, 320, seed=band, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=0.5, beta=2.0)
    ref = reference(p)
    for mode in ("dp", "sk2_dp"):
        C, ws, st = run(p, skgemm.opts_default(sched=mode, tile_n=128, grid=min(23, sms()),
                                               raster_band=band))
        assert st == skgemm.OK
        check_full(p, C, ref)


@pytest.mark.parametrize("shape", [(300, 300, 200), (1000, 1300, 520), (129, 257, 640),
                                   (2000, 2100, 1000)])
@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_abft_ragged_shapes_clean(shape, tile_n, dtype):
    # Ragged m, n and k with the ABFT check on: no false positives, output
    # within tolerance, every tile checked (encode slices of 128 k-columns
    # with a short last one, B tiles of tile_n columns with a short last tile).
    m, n, k = shape
    p = inputs.make_problem(m, n, k, seed=m + n, in_dtype=dtype, out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=0.5, beta=1.5)
    opts = skgemm.opts_default(abft=1, tile_n=tile_n)
    ws = None
    for _ in range(2):   # the encode scratch must be left clean for the next call
        C, ws, st = run(p, opts, ws=ws)
        assert st == skgemm.OK
        check_full(p, C)
        rep = ws.report(reset=True)
        assert rep.detected == 0 and rep.status_bits == 0
        assert rep.tiles_checked == ((m + 127) // 128) * ((n + tile_n - 1) // tile_n)
        assert rep.max_ratio_row < 0.1 and rep.max_ratio_col < 0.1


@pytest.mark.parametrize("tile_n", [128, 256])
def test_abft_f16_large_encodings(tile_n):
    # fp16 operands whose tile column sums exceed the fp16 range (|sum| up to
    # 128 * 3000): the encode pass must scale each tile's encodings by a power
    # of two before splitting them into fp16 terms. Clean run, then a flipped
    # exponent bit that must be found and corrected.
    m, n, k = 640, 768, 1000
    p = inputs.make_problem(m, n, k, seed=31, in_dtype="f16", out_dtype="f32",
                            law_a="uniform", law_b="uniform", scale_a=3000.0, scale_b=1e-3)
    ref = reference(p)
    C, ws, st = run(p, skgemm.opts_default(abft=1, tile_n=tile_n))
    assert st == skgemm.OK
    check_full(p, C, ref)
    rep = ws.report()
    assert rep.detected == 0 and rep.status_bits == 0
    assert rep.max_ratio_row < 0.1 and rep.max_ratio_col < 0.1
    tiles_n = (n + tile_n - 1) // tile_n
    tm, tn = divmod(3, tiles_n)
    v = ref[tm * 128 + 9, tn * tile_n + 17] / p.alpha
    ma, mb = ab.tile_maxima(p.A.double().numpy(), p.B.double().numpy(), tm, tn, 128, tile_n)
    tau = ab.default_tau(k, tile_n, ma, mb)
    kind, _ = ab.classify_flip(v, 30, tau, 1e-3 * tau)
    assert kind == ab.MUST_DETECT, (v, tau)
    C, ws, st = run(p, skgemm.opts_default(abft=1, tile_n=tile_n, inject_tile=3, inject_row=9,
                                           inject_col=17, inject_bit=30))
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.detected == 1 and rep.corrected == 1
    assert (rep.records[0].tile, rep.records[0].row, rep.records[0].col) == (3, 9, 17)
    check_full(p, C, ref)


# --------------------------------------------------------------------------- CTA pairs
@pytest.mark.parametrize("shape", [(256, 256, 64), (384, 512, 320), (1000, 1300, 520),
                                   (2048, 1536, 1024), (129, 3000, 256)])
@pytest.mark.parametrize("mode", ["dp", "sk", "sk2_dp"])
def test_cta_pairs_parity(shape, mode):
    # Clusters of two CTAs (256 x 256 tiles, one M = 256 MMA): element-wise
    # parity, ragged m (an odd number of 128-row tiles leaves the last pair's
    # second half empty), ragged n and k, alpha / beta.
    m, n, k = shape
    p = inputs.make_problem(m, n, k, seed=m * 7 + n, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=0.75, beta=0.5)
    opts = skgemm.opts_default(sched=mode, cta_pair=2)
    tile_n, grid, _ = skgemm.launch_shape(m, n, k, opts)
    assert tile_n == 256 and grid % 2 == 0
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    check_full(p, C)
    assert ws.report().status_bits == 0


@pytest.mark.parametrize("out", ["f16", "bf16"])
def test_cta_pairs_fp16_outputs(out):
    p = inputs.make_problem(640, 768, 512, seed=5, in_dtype="f16", out_dtype=out,
                            law_a="uniform", law_b="uniform")
    C, ws, st = run(p, skgemm.opts_default(cta_pair=2, grid=min(96, sms() // 2 * 2)))
    assert st == skgemm.OK
    check_full(p, C)


@pytest.mark.parametrize("shape", [(300, 300, 200), (1000, 1300, 520), (2000, 2100, 1000)])
def test_cta_pairs_abft_clean(shape):
    # Fused checksum side tiles in pairs (two 128-row checksum tiles per side
    # tile, encoding rows split between the CTAs): no false positives and
    # every 128-row tile with rows checked.
    m, n, k = shape
    p = inputs.make_problem(m, n, k, seed=m + n + 1, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=0.5, beta=1.5)
    opts = skgemm.opts_default(abft=1, cta_pair=2)
    ws = None
    for _ in range(2):
        C, ws, st = run(p, opts, ws=ws)
        assert st == skgemm.OK
        check_full(p, C)
        rep = ws.report(reset=True)
        assert rep.detected == 0 and rep.status_bits == 0
        assert rep.tiles_checked == ((m + 127) // 128) * ((n + 255) // 256)
        assert rep.max_ratio_row < 0.1 and rep.max_ratio_col < 0.1


@pytest.mark.parametrize("bit", [30, 26])
def test_cta_pairs_abft_injection(bit):
    # A flipped exponent bit in the second CTA of a pair (tile row 1 of a
    # 256-row pair tile) is located and corrected.
    m, n, k = 512, 768, 1024
    p = inputs.make_problem(m, n, k, seed=91, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", scale_b=0.02)
    ref = reference(p)
    tiles_n = (n + 255) // 256
    # tiles in odd 128-row tile rows: the second CTA of a pair
    odd = [tm * tiles_n + tn for tm in (1, 3) for tn in range(tiles_n)]
    tile, row, col = draw_must_detect(ref, p.A.double().numpy(), p.B.double().numpy(), p.alpha,
                                      k, m, n, 256, bit, seed=200 + bit, tiles=odd)
    opts = skgemm.opts_default(abft=1, cta_pair=2, inject_tile=tile, inject_row=row,
                               inject_col=col, inject_bit=bit)
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.detected == 1 and rep.corrected == 1
    rec = rep.records[0]
    assert (rec.tile, rec.row, rec.col, rec.injected) == (tile, row, col, 1)
    check_full(p, C, ref)


# --------------------------------------------------------------------------- MN-major operands
def _ld16(x):
    """Row stride of the stored matrix, rounded up to 16 bytes (TMA rule)."""
    return (x.shape[1] + 7) // 8 * 8


@pytest.mark.parametrize("layouts", [(1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("shape", [(200, 136, 72), (1000, 1304, 520), (129, 3000, 4104),
                                   (77, 50, 77)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_mn_major_layouts(layouts, shape, dtype):
    # Column-major A (stored k x m) and / or N-major B (stored k x n), ragged
    # in every dimension, padded leading dimensions, alpha and beta: element
    # by element against the oracle, which indexes the stored operands as
    # given; and bit for bit against the same logical product from K-major
    # operands (the copy is exact and the plan depends only on m, n, k).
    a_layout, b_layout = layouts
    m, n, k = shape
    p = inputs.make_problem(m, n, k, seed=m + 3 * n + k, in_dtype=dtype, out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=0.5, beta=1.5,
                            a_layout=a_layout, b_layout=b_layout)
    C, ws, st = run(p, skgemm.opts_default(), lda=_ld16(p.A) + 8, ldb=_ld16(p.B))
    assert st == skgemm.OK
    check_full(p, C)
    A_k = p.A.t().contiguous() if a_layout else p.A
    B_k = p.B.t().contiguous() if b_layout else p.B
    pk = inputs.Problem(m, n, k, A_k, B_k, p.C0, p.alpha, p.beta, p.in_dtype, p.out_dtype, 0, 0)
    if k % 8 == 0:  # K-major storage needs 16-byte rows
        Ck, _, stk = run(pk, skgemm.opts_default())
        assert stk == skgemm.OK
        assert torch.equal(C, Ck)


@pytest.mark.parametrize("layouts", [(1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("cfg", [dict(tile_n=128, sched="sk", grid=37), dict(tile_n=256),
                                 dict(tile_n=256, cta_pair=2), dict(tile_n=256, cta_pair=2,
                                                                    sched="sk2_dp")])
def test_mn_major_tile_configs(layouts, cfg):
    # MN-major operands read by the MMAs in every mainloop form: 128- and
    # 256-column tiles, single CTAs and CTA pairs, Stream-K fixup; ragged m
    # and n, a padded leading dimension.
    a_layout, b_layout = layouts
    m, n, k = 1000, 1304, 1032
    p = inputs.make_problem(m, n, k, seed=7, in_dtype="bf16", out_dtype="bf16",
                            law_a="normal", law_b="normal", alpha=1.25, beta=0.5,
                            a_layout=a_layout, b_layout=b_layout)
    o = skgemm.opts_default(**cfg)
    C, ws, st = run(p, o, lda=_ld16(p.A) + 16, ldb=_ld16(p.B))
    assert st == skgemm.OK
    check_full(p, C)


@pytest.mark.parametrize("layouts", [(1, 1), (1, 0), (0, 1)])
@pytest.mark.parametrize("case", [(2048, 2048, 2048, "bf16", {}),
                                  (1000, 1304, 1032, "f16", {}),
                                  (640, 768, 1536, "bf16", dict(cta_pair=2, tile_n=256)),
                                  (16768, 256, 512, "bf16", {}),
                                  (1024, 1024, 1024, "bf16", {}),
                                  (1024, 1024, 1024, "bf16", dict(abft_local=2))])
def test_mn_major_layouts_abft(layouts, case):
    # ABFT with MN-major operands: the encode pass sums stored rows, the
    # checksum tiles read A / B as MN-major MMA operands (fused into the
    # launch, or as separate GEMMs when there are too many tiles to fuse:
    # 16768 rows), CTA pairs, fp16 (scaled encodings); the in-CTA references
    # and small bf16 shapes whose plan encodes in the side CTAs (1024^3) run
    # on K-major copies. Clean run, every tile checked, and the same output
    # bits as the K-major call.
    a_layout, b_layout = layouts
    m, n, k, dt, extra = case
    p = inputs.make_problem(m, n, k, seed=11 + m, in_dtype=dt, out_dtype=dt,
                            law_a="normal", law_b="normal", scale_a=k ** -0.5, scale_b=k ** -0.5,
                            a_layout=a_layout, b_layout=b_layout)
    o = skgemm.opts_default(abft=1, **extra)
    if "abft_local" in extra:
        assert skgemm.launch_plan(m, n, k, o).local_checksums == 1
    C, ws, st = run(p, o)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.detected == 0 and rep.status_bits == 0 and rep.tiles_checked > 0
    assert rep.max_ratio_row < 0.1 and rep.max_ratio_col < 0.1
    check_sampled(p, C, seed=5)
    A_k = p.A.t().contiguous() if a_layout else p.A
    B_k = p.B.t().contiguous() if b_layout else p.B
    pk = inputs.Problem(m, n, k, A_k, B_k, p.C0, p.alpha, p.beta, p.in_dtype, p.out_dtype, 0, 0)
    Ck, wsk, stk = run(pk, o)
    assert stk == skgemm.OK and wsk.report().tiles_checked == rep.tiles_checked
    assert torch.equal(C, Ck)


@pytest.mark.parametrize("layouts", [(1, 1), (1, 0), (0, 1)])
def test_mn_major_preencoded(layouts):
    # skg_abft_encode_layout, then the pre-encoded call on the same MN-major
    # operands: the same output bits and report as the one-call ABFT.
    a_layout, b_layout = layouts
    m, n, k = 1024, 768, 1536
    p = inputs.make_problem(m, n, k, seed=44, in_dtype="bf16", out_dtype="bf16",
                            law_a="normal", law_b="normal", scale_a=k ** -0.5, scale_b=k ** -0.5,
                            a_layout=a_layout, b_layout=b_layout)
    o = skgemm.opts_default(abft=1)
    C1, ws1, st1 = run(p, o)
    assert st1 == skgemm.OK
    A, B = p.A.cuda(), p.B.cuda()
    op = skgemm.opts_default(abft=1, abft_preencoded=1)
    ws = skgemm.Workspace(skgemm.workspace_size_layout(m, n, k, a_layout, b_layout, op), "cuda")
    sh = torch.cuda.current_stream().cuda_stream
    assert skgemm.abft_encode(m, n, k, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                              skgemm.IN_BF16, op, ws.ptr, ws.nbytes, sh, a_layout,
                              b_layout) == skgemm.OK
    C2 = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    assert skgemm.gemm(m, n, k, 1.0, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), 0.0,
                       C2.data_ptr(), n, skgemm.IN_BF16, skgemm.OUT_BF16, a_layout, b_layout, op,
                       ws.ptr, ws.nbytes, sh) == skgemm.OK
    torch.cuda.synchronize()
    r1, r2 = ws1.report(), ws.report()
    assert r2.detected == 0 and r2.status_bits == 0 and r2.tiles_checked == r1.tiles_checked
    assert torch.equal(C1, C2)
    check_sampled(p, C2, seed=2)


@pytest.mark.parametrize("bit", [30, 28])
def test_mn_major_abft_injection(bit):
    # A flipped accumulator bit with both operands MN-major is detected,
    # located and corrected against the in-place references.
    p = inputs.make_problem(512, 640, 1024, seed=78, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", scale_b=0.02, a_layout=1, b_layout=1)
    ref = reference(p)
    A_k = p.A.t().double().numpy()
    B_k = p.B.t().double().numpy()
    tile, row, col = draw_must_detect(ref, A_k, B_k, p.alpha, p.k, 512, 640, 128, bit,
                                      seed=300 + bit)
    C, ws, st = _inject(p, dict(tile_n=128), tile, row, col, bit)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.detected == 1 and rep.corrected == 1 and rep.uncorrectable == 0
    rec = rep.records[0]
    assert (rec.tile, rec.row, rec.col, rec.injected) == (tile, row, col, 1)
    check_full(p, C, ref)


def test_mn_major_noalloc_and_matmul():
    # The allocation-free entry point and the torch helper take the layouts
    # too; an MN-major leading dimension below m is an argument error.
    m, n, k = 256, 384, 192
    p = inputs.make_problem(m, n, k, seed=21, in_dtype="bf16", out_dtype="bf16",
                            law_a="normal", law_b="normal", a_layout=1, b_layout=1)
    A, B = p.A.cuda(), p.B.cuda()
    C = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    skgemm.matmul(A, B, C, a_layout=skgemm.A_COL, b_layout=skgemm.B_NMAJOR)
    check_full(p, C)
    C2 = torch.empty_like(C)
    st = skgemm.gemm_noalloc(m, n, k, 1.0, A.data_ptr(), m, B.data_ptr(), n, 0.0, C2.data_ptr(), n,
                             skgemm.IN_BF16, skgemm.OUT_BF16, 1, 1, None,
                             torch.cuda.current_stream().cuda_stream)
    assert st == skgemm.OK
    assert torch.equal(C, C2)
    st = skgemm.gemm_noalloc(m, n, k, 1.0, A.data_ptr(), m - 8, B.data_ptr(), n, 0.0,
                             C2.data_ptr(), n, skgemm.IN_BF16, skgemm.OUT_BF16, 1, 1, None,
                             torch.cuda.current_stream().cuda_stream)
    assert st == skgemm.ERR_ARG


# --------------------------------------------------------------------------- fp64 Stream-K
F64_SHAPES = [(64, 64, 16), (100, 70, 33), (300, 500, 257), (1000, 1000, 1000),
              (128, 128, 4096)]


def _f64_problem(m, n, k, seed):
    gen = torch.Generator().manual_seed(seed)
    A = torch.rand((m, k), generator=gen, dtype=torch.float64) * 2 - 1
    B = torch.rand((n, k), generator=gen, dtype=torch.float64) * 2 - 1
    C0 = torch.rand((m, n), generator=gen, dtype=torch.float64) * 2 - 1
    return A, B, C0


def _run_f64(A, B, C0, alpha, beta, o, ws=None):
    m, k = A.shape
    n = B.shape[0]
    if ws is None:
        ws = skgemm.Workspace(skgemm.workspace_size_f64(m, n, k, o), "cuda")
    Ad, Bd, C = A.cuda(), B.cuda(), C0.clone().cuda()
    st = skgemm.gemm_f64(m, n, k, alpha, Ad.data_ptr(), max(k, 1), Bd.data_ptr(), max(k, 1),
                         beta, C.data_ptr(), n, o, ws.ptr, ws.nbytes,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return C.cpu(), ws, st


@pytest.mark.parametrize("shape", F64_SHAPES)
@pytest.mark.parametrize("mode", MODES)
def test_f64_stream_k(shape, mode):
    # fp64 Stream-K (Stream-K page, §6: FP64 as well as FP16) against the
    # fp64 oracle on every schedule, a small grid (many peers per tile) and
    # a full one; the same workspace twice (launch epochs keep old flags
    # from counting). Only the summation order differs from the oracle:
    # |C - C_ref| <= 1e-12 sqrt(k) max|A| max|B| (inputs in [-1, 1]).
    m, n, k = shape
    A, B, C0 = _f64_problem(m, n, k, seed=m + 3 * n + k)
    alpha, beta = 1.25, -0.5
    ref = oracle.gemm(A.numpy(), B.numpy(), alpha, beta, C0.numpy())
    tol = 1e-12 * math.sqrt(k) + 1e-15
    for g in (7, sms()):
        o = skgemm.opts_default(sched=mode, grid=g)
        ws = None
        for _ in range(2):
            C, ws, st = _run_f64(A, B, C0, alpha, beta, o, ws)
            assert st == skgemm.OK
            assert float(np.abs(C.numpy() - ref).max()) <= tol, (g, mode)
        assert ws.report().timeouts == 0


def test_f64_k_zero_and_beta_zero():
    A, B, C0 = _f64_problem(50, 40, 0, seed=5)
    C, _, st = _run_f64(A, B, C0, 1.0, 3.0, skgemm.opts_default())
    assert st == skgemm.OK and torch.equal(C, 3.0 * C0)
    A, B, C0 = _f64_problem(200, 300, 96, seed=6)
    C0[0, 0] = float("nan")  # beta = 0 does not read C
    C, _, st = _run_f64(A, B, C0, 2.0, 0.0, skgemm.opts_default(sched="sk", grid=16))
    assert st == skgemm.OK
    ref = oracle.gemm(A.numpy(), B.numpy(), 2.0, 0.0, None)
    assert float(np.abs(C.numpy() - ref).max()) <= 1e-12 * math.sqrt(96)


# --------------------------------------------------------------------------- host buffers
@pytest.mark.parametrize("layouts", [(0, 0), (1, 1)])
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("abft", [0, 1])
def test_gemm_host_buffers(layouts, pinned, abft):
    # skg_gemm_host: operands and C in host memory (page-locked or not),
    # copied through the caller's device staging; the same bits as the
    # device-pointer call, and with ABFT a clean report.
    a_layout, b_layout = layouts
    m, n, k = 1000, 1304, 520
    p = inputs.make_problem(m, n, k, seed=31, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=0.5, beta=1.5,
                            a_layout=a_layout, b_layout=b_layout)
    hA, hB, hC = p.A.contiguous(), p.B.contiguous(), p.C0.clone()
    if pinned:
        hA, hB, hC = hA.pin_memory(), hB.pin_memory(), hC.pin_memory()
    o = skgemm.opts_default(abft=abft)
    staging = torch.empty(skgemm.host_staging_size(m, n, k, skgemm.IN_BF16, skgemm.OUT_F32,
                                                   a_layout, b_layout),
                          dtype=torch.uint8, device="cuda")
    ws = skgemm.Workspace(skgemm.workspace_size_layout(m, n, k, a_layout, b_layout, o), "cuda")
    st = skgemm.gemm_host(m, n, k, p.alpha, hA.data_ptr(), hA.stride(0), hB.data_ptr(),
                          hB.stride(0), p.beta, hC.data_ptr(), hC.stride(0), skgemm.IN_BF16,
                          skgemm.OUT_F32, a_layout, b_layout, o, staging.data_ptr(),
                          staging.numel(), ws.ptr, ws.nbytes,
                          torch.cuda.current_stream().cuda_stream)
    assert st == skgemm.OK
    torch.cuda.synchronize()
    check_full(p, hC)
    if abft:
        rep = ws.report()
        assert rep.detected == 0 and rep.status_bits == 0 and rep.tiles_checked > 0
    Cd, _, std = run(p, o)
    assert std == skgemm.OK
    assert torch.equal(hC, Cd.cpu())


# --------------------------------------------------------------------------- single-launch ABFT
@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
def test_abft_store_first_then_correct(out):
    # The first output tile of a launch whose side CTAs run the encode pass
    # is stored before its references are in (beta = 0); a located fault is
    # then corrected in C by one more store, in the output type.
    m, n, k = 384, 640, 320
    p = inputs.make_problem(m, n, k, seed=97, in_dtype="bf16", out_dtype=out,
                            law_a="normal", law_b="normal", alpha=1.25)
    opts = skgemm.opts_default(abft=1)
    plan = skgemm.launch_plan(m, n, k, opts)
    assert plan.encode_in_kernel == 1 and plan.side_ctas > 0
    ref = reference(p)
    tiles_n = -(-n // plan.tile_n)
    hits = 0
    for (tm, tn, row, col) in [(0, 0, 5, 7), (2, tiles_n - 1, 127, 3), (1, 2, 64, 100)]:
        gi, gj = tm * 128 + row, tn * plan.tile_n + col
        ma, mb = ab.tile_maxima(p.A.double().numpy(), p.B.double().numpy(), tm, tn, 128,
                                plan.tile_n)
        kind, _ = ab.classify_flip(ref[gi, gj] / p.alpha, 30,
                                   ab.default_tau(k, plan.tile_n, ma, mb), 1e-3)
        if kind != ab.MUST_DETECT:
            continue
        hits += 1
        o = skgemm.opts_default(abft=1, inject_tile=tm * tiles_n + tn, inject_row=row,
                                inject_col=col, inject_bit=30)
        C, ws, st = run(p, o)
        assert st == skgemm.OK
        rep = ws.report()
        assert rep.detected == 1 and rep.corrected == 1 and rep.uncorrectable == 0
        assert (rep.records[0].tile, rep.records[0].row, rep.records[0].col) == \
            (tm * tiles_n + tn, row, col)
        check_full(p, C, ref)
    assert hits >= 2
    C, ws, st = run(p, opts)
    assert st == skgemm.OK
    check_full(p, C, ref)
    assert ws.report().detected == 0


@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (384, 640, 320), (300, 1000, 520)])
def test_abft_encode_in_kernel(shape):
    # Small bf16 shapes whose output tiles leave SMs idle: the checksum tiles
    # run on extra CTAs that first run the encode pass, so the whole ABFT
    # call is one launch. Clean run, a reused workspace, then a fault.
    m, n, k = shape
    p = inputs.make_problem(m, n, k, seed=m + 3 * n, in_dtype="bf16", out_dtype="bf16",
                            law_a="normal", law_b="normal", scale_a=k ** -0.5,
                            scale_b=k ** -0.5)
    opts = skgemm.opts_default(abft=1)
    plan = skgemm.launch_plan(m, n, k, opts)
    assert plan.fused_checksums == 1 and plan.encode_in_kernel == 1 and plan.side_ctas > 0
    ref = reference(p)
    ws = None
    for _ in range(2):
        C, ws, st = run(p, opts, ws=ws)
        assert st == skgemm.OK
        check_full(p, C, ref)
        rep = ws.report(reset=True)
        assert rep.detected == 0 and rep.status_bits == 0
        assert rep.tiles_checked == ((m + 127) // 128) * ((n + plan.tile_n - 1) // plan.tile_n)
        assert rep.max_ratio_row < 0.1 and rep.max_ratio_col < 0.1
    tiles_n = (n + plan.tile_n - 1) // plan.tile_n
    tm, tn, row, col = (m - 1) // 128, tiles_n - 1, 3, 5
    gi, gj = tm * 128 + row, tn * plan.tile_n + col
    if gi >= m or gj >= n:
        tm, tn = 0, 0
        gi, gj = row, col
    v = ref[gi, gj] / p.alpha
    ma, mb = ab.tile_maxima(p.A.double().numpy(), p.B.double().numpy(), tm, tn, 128,
                            plan.tile_n)
    kind, _ = ab.classify_flip(v, 30, ab.default_tau(k, plan.tile_n, ma, mb), 1e-3)
    assert kind == ab.MUST_DETECT
    oi = skgemm.opts_default(abft=1, inject_tile=tm * tiles_n + tn, inject_row=row,
                             inject_col=col, inject_bit=30)
    C, ws, st = run(p, oi, ws=ws)
    assert st == skgemm.OK
    rep = ws.report()
    assert rep.detected == 1 and rep.corrected == 1
    assert (rep.records[0].tile, rep.records[0].row, rep.records[0].col) == \
        (tm * tiles_n + tn, row, col)
    check_full(p, C, ref)
