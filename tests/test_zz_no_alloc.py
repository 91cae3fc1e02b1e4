"""skg_gemm_noalloc: the allocation-free entry point, for callers that cannot
allocate device memory (a plugin whose host framework owns all device memory
through its own allocator, or a latency-critical path that cannot afford
cudaMalloc's implicit synchronisation).

Two calls in a row through the C ABI must each match skg_gemm (which takes
a caller workspace) within the parity tolerance of the other GPU tests. The
second call reuses the shared scratch array as the first call left it.
A longer sequence mixes shapes, input types, grids, CTA pairs and ABFT on
the one array, and the array's report (skg_noalloc_report_read) shows what
the device decided. This file is collected last on purpose; it passes alone
or after the rest.
"""
import numpy as np
import pytest
import torch

from oracle import schedule_sim as ss

from stream_decomposition_abft_gb300 import _build, inputs, skgemm

from gpu_util import IN_CODE, OUT_CODE, out_init, tolerance, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    skgemm.lib()


def _call(fn_name, p, A, B, C, opts, ws=None):
    stream = torch.cuda.current_stream().cuda_stream
    args = (p.m, p.n, p.k, p.alpha, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), p.beta,
            C.data_ptr(), C.stride(0), IN_CODE[p.in_dtype], OUT_CODE[p.out_dtype], 0, 0, opts)
    if fn_name == "noalloc":
        return skgemm.gemm_noalloc(*args, stream)
    return skgemm.gemm(*args, ws.ptr, ws.nbytes, stream)


def test_noalloc_matches_gemm_on_two_calls():
    problems = [
        inputs.make_problem(1000, 1200, 520, seed=31, in_dtype="bf16", out_dtype="bf16",
                            law_a="normal", law_b="normal", alpha=1.25, beta=0.5),
        inputs.make_problem(384, 2304, 4096, seed=32, in_dtype="f16", out_dtype="f32",
                            law_a="uniform", law_b="uniform"),
    ]
    opts = skgemm.opts_default(sched="sk2_dp", tile_n=128)
    for p in problems:
        A, B = to_device(p, "cuda")
        ws = skgemm.Workspace(skgemm.workspace_size(p.m, p.n, p.k, opts), "cuda")
        C_ref = out_init(p, "cuda")
        assert _call("gemm", p, A, B, C_ref, opts, ws) == skgemm.OK
        C_new = out_init(p, "cuda")
        assert _call("noalloc", p, A, B, C_new, opts) == skgemm.OK
        torch.cuda.synchronize()
        ref = C_ref.float().cpu().double().numpy()
        got = C_new.float().cpu().double().numpy()
        assert np.all(np.abs(got - ref) <= tolerance(p, ref))


def test_noalloc_rejects_oversized_workspace():
    # BLK_N = 256 with ABFT on needs more than the fixed array on this GPU.
    p = inputs.make_problem(4096, 4096, 4096, seed=33, in_dtype="bf16", out_dtype="bf16")
    opts = skgemm.opts_default(abft=1, tile_n=256)
    need = skgemm.workspace_size(p.m, p.n, p.k, opts)
    if need <= (16 << 20):
        pytest.skip("this GPU's workspace fits the array")
    A, B = to_device(p, "cuda")
    C = out_init(p, "cuda")
    assert _call("noalloc", p, A, B, C, opts) == skgemm.ERR_WORKSPACE


def test_noalloc_sequence_of_shapes_and_options():
    # Calls whose workspace layouts differ, one after the other on the shared
    # array: every result equals skg_gemm's with the same options on a
    # workspace of its own (same plan, same summation order), and the
    # array's report shows the ABFT checks of exactly these calls.
    seq = [
        (inputs.make_problem(2048, 2048, 1024, seed=61, in_dtype="bf16", out_dtype="bf16",
                             law_a="normal", law_b="normal"), dict(tile_n=128)),
        (inputs.make_problem(700, 900, 520, seed=62, in_dtype="f16", out_dtype="f16",
                             alpha=1.5, beta=0.5), dict(abft=1, grid=16, tile_n=128)),
        (inputs.make_problem(1000, 1300, 520, seed=63, in_dtype="bf16", out_dtype="f32",
                             law_a="normal", law_b="normal"),
         dict(abft=1, cta_pair=2, tile_n=256, grid=16)),
        (inputs.make_problem(384, 4096, 704, seed=64, in_dtype="bf16", out_dtype="bf16",
                             law_a="normal", law_b="normal"), dict(sched="sk", tile_n=128)),
        # 64-wide tiles; skg_gemm splits the tiles two CTAs end in, the
        # allocation-free entry keeps the owner fixup (same sums: two parts)
        (inputs.make_problem(640, 512, 8192, seed=65, in_dtype="bf16", out_dtype="f32",
                             law_a="normal", law_b="normal"), dict(sched="sk", tile_n=64, grid=70)),
        (inputs.make_problem(2048, 2048, 1024, seed=61, in_dtype="bf16", out_dtype="bf16",
                             law_a="normal", law_b="normal"), dict(tile_n=128)),
    ]
    stream = torch.cuda.current_stream().cuda_stream
    skgemm.noalloc_report_read(reset=True, stream=stream)
    for i, (p, kw) in enumerate(seq):
        opts = skgemm.opts_default(**kw)
        A, B = to_device(p, "cuda")
        ws = skgemm.Workspace(skgemm.workspace_size(p.m, p.n, p.k, opts), "cuda")
        C_ref = out_init(p, "cuda")
        assert _call("gemm", p, A, B, C_ref, opts, ws) == skgemm.OK, i
        C_new = out_init(p, "cuda")
        assert _call("noalloc", p, A, B, C_new, opts) == skgemm.OK, i
        rep = skgemm.noalloc_report_read(reset=True, stream=stream)
        ref_rep = ws.report()
        assert torch.equal(C_new, C_ref), i
        assert rep.status_bits == 0 and rep.detected == 0, i
        assert rep.tiles_checked == ref_rep.tiles_checked, i
        assert (rep.tiles_checked > 0) == bool(kw.get("abft")), i


def test_noalloc_report_shows_a_timeout():
    # A device-side failure on this path is not silent: a CTA that skips its
    # Stream-K signal makes its owner's bounded wait run out, and the array's
    # report says so; the next call on the array is correct again.
    stream = torch.cuda.current_stream().cuda_stream
    p = inputs.make_problem(256, 256, 4096, seed=65, in_dtype="bf16", out_dtype="f32")
    rows = ss.flatten(ss.schedule(256, 256, 4096, 128, 128, 64, 8, mode="sk"))
    peer = next(r[0] for r in rows if r[4] == ss.PEER)
    opts = skgemm.opts_default(sched="sk", grid=8, tile_n=128, timeout_ns=50_000_000,
                               test_drop_signal=peer + 1)
    A, B = to_device(p, "cuda")
    C = out_init(p, "cuda")
    skgemm.noalloc_report_read(reset=True, stream=stream)
    assert _call("noalloc", p, A, B, C, opts) == skgemm.OK
    rep = skgemm.noalloc_report_read(reset=True, stream=stream)
    assert rep.status_bits & (1 << skgemm.ERR_FIXUP_TIMEOUT) and rep.timeouts >= 1
    good = skgemm.opts_default(sched="sk", grid=8, tile_n=128)
    C2 = out_init(p, "cuda")
    assert _call("noalloc", p, A, B, C2, good) == skgemm.OK
    ws = skgemm.Workspace(skgemm.workspace_size(p.m, p.n, p.k, good), "cuda")
    C3 = out_init(p, "cuda")
    assert _call("gemm", p, A, B, C3, good, ws) == skgemm.OK
    assert torch.equal(C2, C3)
    assert skgemm.noalloc_report_read(reset=True, stream=stream).status_bits == 0
