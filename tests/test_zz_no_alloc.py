"""skg_gemm_noalloc: the allocation-free entry point, for callers that cannot
allocate device memory (a plugin whose host framework owns all device memory
through its own allocator, or a latency-critical path that cannot afford
cudaMalloc's implicit synchronisation).

Two calls in a row through the C ABI must each match skg_gemm (which takes
a caller workspace) within the parity tolerance of the other GPU tests. The
second call reuses the shared scratch array as the first call left it.
This file is collected last on purpose; it passes alone or after the rest.
"""
import numpy as np
import pytest
import torch

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
