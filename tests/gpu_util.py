"""Helpers shared by the GPU tests: run a Problem through the C ABI and
compare with the fp64 oracle under the parity tolerance.

Parity tolerance (fp32 accumulation of fp16 / bf16 products), per element:
    |C - C_ref| <= |alpha| * 1e-3 * sqrt(k) * max|A| * max|B| + u_out * |C_ref|
with u_out the unit roundoff of the output type (2^-24 fp32, 2^-11 fp16,
2^-8 bf16): the final rounding to a 16-bit output is allowed on top of the
accumulation bound.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from stream_decomposition_abft_gb300 import inputs, skgemm

U_OUT = {"f32": 2.0 ** -24, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}
IN_CODE = {"f16": skgemm.IN_F16, "bf16": skgemm.IN_BF16}
OUT_CODE = {"f32": skgemm.OUT_F32, "f16": skgemm.OUT_F16, "bf16": skgemm.OUT_BF16}


def tolerance(p: inputs.Problem, ref: np.ndarray) -> np.ndarray:
    base = abs(p.alpha) * 1e-3 * math.sqrt(max(p.k, 1)) * float(p.A.abs().max()) * \
        float(p.B.abs().max())
    return base + U_OUT[p.out_dtype] * np.abs(ref) + 1e-30


def to_device(p: inputs.Problem, dev, lda=None, ldb=None):
    """A, B on the device, optionally inside wider row strides (padded ld)."""
    def place(x, ld):
        if ld is None or ld == x.shape[1]:
            return x.to(dev).contiguous()
        buf = torch.zeros((x.shape[0], ld), dtype=x.dtype, device=dev)
        buf[:, :x.shape[1]] = x.to(dev)
        return buf[:, :x.shape[1]]
    return place(p.A, lda), place(p.B, ldb)


def out_init(p: inputs.Problem, dev):
    """C on the device with its row stride padded to 16 bytes (TMA rule)."""
    dt = inputs.DTYPES[p.out_dtype]
    per = 16 // torch.empty((), dtype=dt).element_size()
    ldc = (p.n + per - 1) // per * per
    buf = torch.full((p.m, ldc), float("nan"), dtype=dt, device=dev)
    C = buf[:, :p.n]
    if p.C0 is not None:
        C.copy_(p.C0.to(dev))
    return C


def run(p: inputs.Problem, opts=None, ws=None, dev="cuda", verify=False, lda=None, ldb=None):
    """Launch through the C ABI; returns (C on device, workspace, status)."""
    A, B = to_device(p, dev, lda, ldb)
    C = out_init(p, dev)
    if ws is None:
        ws = skgemm.Workspace(skgemm.workspace_size_layout(p.m, p.n, p.k, p.a_layout, p.b_layout,
                                                           opts), dev)
    stream = torch.cuda.current_stream().cuda_stream
    fn = skgemm.gemm_verify if verify else skgemm.gemm
    st = fn(p.m, p.n, p.k, p.alpha, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), p.beta,
            C.data_ptr(), C.stride(0), IN_CODE[p.in_dtype], OUT_CODE[p.out_dtype], p.a_layout,
            p.b_layout, opts, ws.ptr, ws.nbytes, stream)
    return C, ws, st


def reference(p: inputs.Problem) -> np.ndarray:
    C0 = p.C0.float() if p.C0 is not None else None
    return oracle.gemm(p.A, p.B, alpha=p.alpha, beta=p.beta, C0=C0, a_layout=p.a_layout,
                       b_layout=p.b_layout)


def check_full(p: inputs.Problem, C: torch.Tensor, ref: np.ndarray = None):
    if ref is None:
        ref = reference(p)
    got = C.float().cpu().double().numpy()
    tol = tolerance(p, ref)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} entries out of tolerance; worst "
                           f"err {float(np.nanmax(err)):.3e} at "
                           f"{np.unravel_index(int(np.nanargmax(err)), err.shape)}")
    return float(np.max(err / tol))


def sample_plan(m: int, n: int, seed: int, count: int = 256, rows: int = 8, cols: int = 8):
    """Seeded sample: `count` random entries plus `rows` full rows and `cols`
    full columns (first, last and random ones)."""
    rng = np.random.default_rng(seed)
    r = list(rng.integers(0, m, count))
    c = list(rng.integers(0, n, count))
    full_rows = sorted(set([0, m - 1] + list(rng.integers(0, m, max(0, rows - 2)))))
    full_cols = sorted(set([0, n - 1] + list(rng.integers(0, n, max(0, cols - 2)))))
    for i in full_rows:
        r += [i] * n
        c += list(range(n))
    for j in full_cols:
        r += list(range(m))
        c += [j] * m
    return np.array(r, dtype=np.int64), np.array(c, dtype=np.int64)


def check_sampled(p: inputs.Problem, C: torch.Tensor, seed: int = 0, count: int = 256,
                  rows: int = 8, cols: int = 8):
    r, c = sample_plan(p.m, p.n, seed, count, rows, cols)
    C0 = p.C0.float() if p.C0 is not None else None
    ref = oracle.gemm_entries(p.A, p.B, r, c, alpha=p.alpha, beta=p.beta, C0=C0,
                              a_layout=p.a_layout, b_layout=p.b_layout)
    got = C[torch.as_tensor(r, device=C.device), torch.as_tensor(c, device=C.device)]
    got = got.float().cpu().double().numpy()
    tol = tolerance(p, ref)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{int(bad.sum())} sampled entries out of tolerance; worst "
                           f"{float(np.nanmax(err)):.3e}")
    return float(np.max(err / tol))


def check_checksum_probe(p: inputs.Problem, C: torch.Tensor):
    """Whole-matrix probes e^T C vs (e^T A) B and C e vs A (B e), in fp64,
    bounded by the sum of the per-element tolerances along the line."""
    A = p.A.double()
    B = p.B.double()                   # stored n x k
    eA = A.sum(dim=0)                  # k
    Be = B.sum(dim=0)                  # k  (sum over the n rows of the stored B)
    cc = (B @ eA) * p.alpha            # n: (e^T A) B
    cr = (A @ Be) * p.alpha            # m: A (B e)
    if p.C0 is not None:
        C0 = p.C0.double()
        cc = cc + p.beta * C0.sum(dim=0)
        cr = cr + p.beta * C0.sum(dim=1)
    Cd = C.double()
    col = Cd.sum(dim=0).cpu()
    row = Cd.sum(dim=1).cpu()
    base = abs(p.alpha) * 1e-3 * math.sqrt(p.k) * float(p.A.abs().max()) * float(p.B.abs().max())
    u = U_OUT[p.out_dtype]
    tol_c = p.m * base + u * Cd.abs().sum(dim=0).cpu()
    tol_r = p.n * base + u * Cd.abs().sum(dim=1).cpu()
    assert bool(((col - cc).abs() <= tol_c).all()), "column checksum probe failed"
    assert bool(((row - cr).abs() <= tol_r).all()), "row checksum probe failed"


def draw_must_detect(ref, A_km, B_km, alpha, k, m, n, bn, bit, seed, tiles=None, bm=128):
    """A seeded (tile, row, col) of a 128 x bn ABFT tile whose accumulator
    flips by more than ten thresholds when `bit` flips (the fault model's
    must-detect class), so an injection test never has to skip. `ref` is the
    oracle's C (alpha applied), A_km / B_km the K-major stored operands
    (m x k and n x k) for the tile maxima; `tiles` restricts the draw to some
    tile numbers (row-major over 128 x bn tiles)."""
    from oracle import abft_ref as ab
    rng = np.random.default_rng(seed)
    tiles_n = (n + bn - 1) // bn
    tiles_m = (m + bm - 1) // bm
    pool = list(tiles) if tiles is not None else list(range(tiles_m * tiles_n))
    for _ in range(20000):
        tile = int(pool[int(rng.integers(0, len(pool)))])
        tm, tn = divmod(tile, tiles_n)
        row, col = int(rng.integers(0, bm)), int(rng.integers(0, bn))
        gi, gj = tm * bm + row, tn * bn + col
        if gi >= m or gj >= n:
            continue
        v = ref[gi, gj] / alpha
        ma, mb = ab.tile_maxima(A_km, B_km, tm, tn, bm, bn)
        tau = max(ab.default_tau(k, bn, ma, mb), ab.default_tau(k, bm, ma, mb))
        kind, _ = ab.classify_flip(v, bit, tau, 1e-3 * tau)
        if kind == ab.MUST_DETECT:
            return tile, row, col
    raise AssertionError(f"no must-detect position for bit {bit}")
