"""Pins of the fp64 GEMM oracle and the ABFT checksum / fault oracle.

Nothing here compares the oracle with itself: the GEMM is checked against
hand-computed products, closed forms and numpy's matmul (an independent
second definition); the checksum identities are checked exactly on integer
data; the fault model against the IEEE-754 closed form of a bit flip.
"""
import math
import struct

import numpy as np
import pytest
import torch

import oracle
from oracle import abft_ref as ab
from stream_decomposition_abft_gb300 import inputs


def test_hand_computed_2x3x2():
    # A (2x3) and B (3x2) written out; C = alpha*A@B + beta*C0 by hand.
    A = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])
    B_logical = np.array([[7.0, 8.0], [9.0, 10.0], [11.0, 12.0]])
    C0 = np.array([[1.0, -1.0], [0.5, 2.0]])
    # A@B = [[58, 64], [139, 154]]
    want = 2.0 * np.array([[58.0, 64.0], [139.0, 154.0]]) + 0.5 * C0
    got = oracle.gemm(A, B_logical.T.copy(), alpha=2.0, beta=0.5, C0=C0)   # B stored n x k
    assert np.array_equal(got, want)
    # the other storage orders give the same product
    got = oracle.gemm(A.T.copy(), B_logical, alpha=2.0, beta=0.5, C0=C0, a_layout=1, b_layout=1)
    assert np.array_equal(got, want)


def test_ones_and_identity():
    m, n, k = 5, 7, 13
    C = oracle.gemm(np.ones((m, k)), np.ones((n, k)))
    assert np.array_equal(C, np.full((m, n), float(k)))
    X = np.arange(35, dtype=np.float64).reshape(5, 7)
    C = oracle.gemm(np.eye(5), X.T.copy())      # I (5x5) @ X (5x7); B stored (7, 5)
    assert np.array_equal(C, X)


def test_beta_zero_does_not_read_c0():
    A = np.ones((3, 4))
    B = np.ones((2, 4))
    C0 = np.full((3, 2), np.nan)
    C = oracle.gemm(A, B, beta=0.0, C0=C0)
    assert np.all(np.isfinite(C))
    C = oracle.gemm(A, B, beta=1.0, C0=C0)
    assert np.all(np.isnan(C))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_integer_inputs_match_numpy_exactly(dtype):
    p = inputs.make_problem(37, 53, 71, seed=5, in_dtype=dtype, out_dtype="f32",
                            law_a="integer", law_b="integer", alpha=1.0, beta=0.0)
    A = p.A.double().numpy()
    B = p.B.double().numpy()
    got = oracle.gemm(p.A, p.B)
    assert np.array_equal(got, A @ B.T)


def test_random_inputs_match_numpy():
    p = inputs.make_problem(97, 61, 257, seed=6, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=-0.75, beta=1.25,
                            law_c="uniform")
    p.C0 = p.C0.float()
    want = -0.75 * (p.A.double().numpy() @ p.B.double().numpy().T) + 1.25 * p.C0.double().numpy()
    got = oracle.gemm(p.A, p.B, alpha=-0.75, beta=1.25, C0=p.C0)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("a_layout,b_layout", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_entries_match_full(a_layout, b_layout):
    p = inputs.make_problem(40, 33, 29, seed=8, in_dtype="f16", out_dtype="f32",
                            law_a="normal", law_b="normal", alpha=1.5, beta=0.5,
                            a_layout=a_layout, b_layout=b_layout)
    full = oracle.gemm(p.A, p.B, 1.5, 0.5, p.C0, a_layout, b_layout)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, 40, 50)
    cols = rng.integers(0, 33, 50)
    ent = oracle.gemm_entries(p.A, p.B, rows, cols, 1.5, 0.5, p.C0, a_layout, b_layout)
    assert np.array_equal(ent, full[rows, cols])
    # and numpy agrees on the logical product
    A = p.A.double().numpy() if a_layout == 0 else p.A.double().numpy().T
    B = p.B.double().numpy().T if b_layout == 0 else p.B.double().numpy()
    assert np.allclose(full, 1.5 * A @ B + 0.5 * p.C0.double().numpy(), rtol=1e-13, atol=1e-13)


def test_empty_shapes():
    assert oracle.gemm(np.zeros((0, 4)), np.zeros((3, 4))).shape == (0, 3)
    C = oracle.gemm(np.zeros((2, 0)), np.zeros((3, 0)), beta=2.0, C0=np.ones((2, 3)))
    assert np.array_equal(C, np.full((2, 3), 2.0))


# ----------------------------------------------------------------------------
# Checksum identities (fault-tolerance page, Fig. 3 / Fig. 5)
# ----------------------------------------------------------------------------
def test_checksum_identities_exact_on_integers():
    p = inputs.make_problem(128, 96, 200, seed=9, in_dtype="bf16", out_dtype="f32",
                            law_a="integer", law_b="integer")
    A = p.A.double().numpy()
    B = p.B.double().numpy().T          # logical k x n
    C = oracle.gemm(p.A, p.B)
    cc, cr = ab.reference_checksums(A, B)
    colsum, rowsum = ab.product_checksums(C)
    assert np.array_equal(colsum, cc)   # e^T C == (e^T A) B
    assert np.array_equal(rowsum, cr)   # C e   == A (B e)
    # the encodings are the sums they claim to be
    assert np.array_equal(ab.encode_cols(A), A.sum(axis=0))
    assert ab.encode_rows(B).shape == (200,)


def test_checksum_identities_random_close():
    p = inputs.make_problem(64, 80, 300, seed=10, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal")
    A = p.A.double().numpy()
    B = p.B.double().numpy().T
    C = oracle.gemm(p.A, p.B)
    cc, cr = ab.reference_checksums(A, B)
    colsum, rowsum = ab.product_checksums(C)
    scale = np.abs(A).sum() * np.abs(B).max()
    assert np.max(np.abs(colsum - cc)) <= 1e-12 * scale
    assert np.max(np.abs(rowsum - cr)) <= 1e-12 * scale


def test_tile_reference_covers_ragged_tile():
    p = inputs.make_problem(200, 300, 64, seed=11, in_dtype="f16", out_dtype="f32",
                            law_a="integer", law_b="integer")
    A = p.A.double().numpy()
    B = p.B.double().numpy().T
    C = oracle.gemm(p.A, p.B)
    cc, cr = ab.tile_reference(A, B, 1, 2, 128, 128)   # rows 128..199, cols 256..299
    assert cc.shape == (44,) and cr.shape == (72,)
    assert np.array_equal(cc, C[128:200, 256:300].sum(axis=0))
    assert np.array_equal(cr, C[128:200, 256:300].sum(axis=1))


# ----------------------------------------------------------------------------
# Fault model and verify / locate / correct
# ----------------------------------------------------------------------------
def test_exponent_flip_closed_form():
    for v in (1.5, -3.25, 0.0078125, 1234.5):
        for bit in range(23, 31):
            w = ab.flip_f32(v, bit)
            if math.isfinite(w) and w != 0.0 and abs(w) >= 2.0 ** -126:
                assert w == v * ab.exponent_flip_factor(v, bit)


def test_sign_and_mantissa_flips():
    assert ab.flip_f32(2.5, 31) == -2.5
    assert ab.flip_f32(1.0, 22) == 1.5          # top mantissa bit
    assert ab.flip_f32(1.0, 0) == 1.0 + 2.0 ** -23
    (u,) = struct.unpack("<I", struct.pack("<f", 1.0))
    assert u == 0x3F800000
    assert math.isinf(ab.flip_f32(1.5, 30)) or math.isnan(ab.flip_f32(1.5, 30))


def test_classification_bands():
    tau = 1e-3
    assert ab.classify_flip(1.0, 30, tau, 1e-5)[0] == ab.MUST_DETECT   # -> Inf/NaN
    assert ab.classify_flip(1.0, 31, tau, 1e-5)[0] == ab.MUST_DETECT   # sign, |delta| = 2
    assert ab.classify_flip(1.0, 0, tau, 1e-5)[0] == ab.HARMLESS       # 2^-23
    assert ab.classify_flip(1.0, 12, tau, 1e-5)[0] == ab.GREY          # 2^-11 ~ 4.9e-4


@pytest.mark.parametrize("bit", [31, 30, 27, 24, 22, 20])
def test_verify_locates_and_corrects_planted_fault(bit):
    p = inputs.make_problem(128, 128, 256, seed=12, in_dtype="bf16", out_dtype="f32",
                            law_a="normal", law_b="normal")
    A = p.A.double().numpy()
    B = p.B.double().numpy().T
    C = oracle.gemm(p.A, p.B)
    cc, cr = ab.reference_checksums(A, B)
    tau_r = ab.default_tau(256, 128, np.abs(A).max(), np.abs(B).max())
    tau_c = tau_r
    clean = ab.verify_tile(C, cr, cc, tau_r, tau_c)
    assert clean["status"] == ab.CLEAN and clean["max_ratio_r"] < 1e-6
    i, j = 37, 101
    faulty = C.copy()
    kind, delta = ab.classify_flip(C[i, j], bit, tau_r, 1e-6)
    faulty[i, j] = ab.flip_f32(C[i, j], bit)
    res = ab.verify_tile(faulty, cr, cc, tau_r, tau_c)
    if kind == ab.MUST_DETECT:
        assert res["status"] == ab.CORRECTED
        assert (res["row"], res["col"]) == (i, j)
        assert abs(res["value"] - C[i, j]) <= 1e-9 * max(1.0, abs(C[i, j]))


def test_two_faults_are_uncorrectable():
    rng = np.random.default_rng(3)
    C = rng.standard_normal((16, 16))
    cc, cr = C.sum(axis=0), C.sum(axis=1)
    bad = C.copy()
    bad[2, 3] += 10.0
    bad[5, 9] -= 10.0
    assert ab.verify_tile(bad, cr, cc, 1e-6, 1e-6)["status"] == ab.UNCORRECTABLE
    one = C.copy()
    one[4, 4] = np.nan
    res = ab.verify_tile(one, cr, cc, 1e-6, 1e-6)
    assert res["status"] == ab.CORRECTED and (res["row"], res["col"]) == (4, 4)
    assert abs(res["value"] - C[4, 4]) < 1e-12


def test_inputs_are_seeded_and_rounded():
    a = inputs.example_384()
    b = inputs.example_384()
    assert torch.equal(a.A, b.A) and torch.equal(a.B, b.B)
    assert a.A.dtype == torch.float16 and a.A.shape == (384, 128) and a.B.shape == (384, 128)
    assert float(a.A.abs().max()) <= 1.0
    shapes = inputs.random_shapes(1000)
    assert len(shapes) == 1000
    assert all(128 <= d <= 8192 and d % 128 == 0 for s in shapes for d in s)


# ----------------------------------------------------------------------------
# Detection threshold and tile maxima (written out by hand)
# ----------------------------------------------------------------------------
def test_default_tau_hand_computed():
    # tau = 2^-12 * sqrt(k) * sqrt(side) * max|A| * max|B|, values picked so
    # every factor is a power of two: 2^-12 * 4 * 8 * 2 * 0.5 = 2^-7.
    assert ab.default_tau(16, 64, 2.0, 0.5) == 2.0 ** -7
    # side enters under a square root (a row check over 256 columns is twice
    # the threshold of one over 64), and so does k.
    assert ab.default_tau(16, 256, 2.0, 0.5) == 2.0 ** -6
    assert ab.default_tau(64, 64, 2.0, 0.5) == 2.0 ** -6
    # linear in each maximum
    assert ab.default_tau(16, 64, 6.0, 0.5) == 3.0 * 2.0 ** -7
    # k = 1536, side 256 / 128, max 2 and 2: the values the grey-band tests use
    assert abs(ab.default_tau(1536, 256, 2.0, 2.0) - 2.0 ** -10 * math.sqrt(1536) * 16) < 1e-15
    assert ab.default_tau(0, 128, 1.0, 1.0) == 0.0


def test_tile_maxima_hand_placed():
    # A stored m x k = 4 x 3, B stored n x k = 6 x 3, tiles of 2 rows of A
    # and 3 stored rows of B (= 3 output columns).
    A = np.array([[0.5, -1.0, 0.25],
                  [0.0, 0.75, -0.5],      # tile tm = 0: max |.| = 1.0
                  [-4.0, 0.5, 1.0],
                  [2.0, -3.0, 0.0]])      # tile tm = 1: max |.| = 4.0
    B = np.array([[1.0, 0.0, -2.0],
                  [0.5, 0.5, 0.5],
                  [-1.5, 0.0, 0.0],       # tile tn = 0 (stored rows 0..2): max 2.0
                  [0.0, -8.0, 0.0],
                  [0.25, 0.0, 3.0],
                  [0.0, 0.0, -0.125]])    # tile tn = 1 (stored rows 3..5): max 8.0
    assert ab.tile_maxima(A, B, 0, 0, 2, 3) == (1.0, 2.0)
    assert ab.tile_maxima(A, B, 1, 0, 2, 3) == (4.0, 2.0)
    assert ab.tile_maxima(A, B, 0, 1, 2, 3) == (1.0, 8.0)
    assert ab.tile_maxima(A, B, 1, 1, 2, 3) == (4.0, 8.0)
    # A ragged last tile (rows past m are absent, not zero-padded maxima).
    assert ab.tile_maxima(A, B, 1, 1, 3, 4) == (3.0, 3.0)


def test_verify_tile_grey_band_and_patterns():
    # Integer tile with exact checksums; faults planted by hand.
    rng = np.random.default_rng(5)
    C = rng.integers(-20, 21, size=(8, 8)).astype(np.float64)
    cc, cr = C.sum(axis=0), C.sum(axis=1)
    clean = ab.verify_tile(C, cr, cc, 0.6, 0.4)
    assert clean["status"] == ab.CLEAN and clean["bad_rows"] == [] and clean["bad_cols"] == []
    # |delta| = 0.5 between tau_col = 0.4 and tau_row = 0.6: the column sees
    # it, the row does not -> one bad column, no bad row, uncorrectable.
    g = C.copy()
    g[3, 5] += 0.5
    res = ab.verify_tile(g, cr, cc, 0.6, 0.4)
    assert (res["bad_rows"], res["bad_cols"], res["status"]) == ([], [5], ab.UNCORRECTABLE)
    # Two faults in one row: one bad row, two bad columns.
    g = C.copy()
    g[2, 1] += 4.0
    g[2, 6] -= 8.0
    res = ab.verify_tile(g, cr, cc, 0.6, 0.4)
    assert (res["bad_rows"], res["bad_cols"], res["status"]) == ([2], [1, 6], ab.UNCORRECTABLE)
    # Two faults in one column: two bad rows, one bad column.
    g = C.copy()
    g[0, 4] += 4.0
    g[7, 4] += 4.0
    res = ab.verify_tile(g, cr, cc, 0.6, 0.4)
    assert (res["bad_rows"], res["bad_cols"], res["status"]) == ([0, 7], [4], ab.UNCORRECTABLE)
    # Two faults that cancel in their shared row: the row checksum is clean.
    g = C.copy()
    g[6, 0] += 3.0
    g[6, 2] -= 3.0
    res = ab.verify_tile(g, cr, cc, 0.6, 0.4)
    assert (res["bad_rows"], res["bad_cols"], res["status"]) == ([], [0, 2], ab.UNCORRECTABLE)
    # One fault: corrected back to the clean value from the row checksum.
    g = C.copy()
    g[4, 3] = 1e30
    res = ab.verify_tile(g, cr, cc, 0.6, 0.4)
    assert (res["status"], res["row"], res["col"], res["value"]) == (ab.CORRECTED, 4, 3, C[4, 3])


def test_tile_bounds_ragged_edges():
    # A 300 x 200 output in 128 x 128 tiles: the last tile row holds rows
    # 256 .. 299 and the last tile column columns 128 .. 199; a 256-wide
    # tile column covers all 200 columns.
    assert ab.tile_bounds(0, 0, 128, 128, 300, 200) == (0, 128, 0, 128)
    assert ab.tile_bounds(2, 1, 128, 128, 300, 200) == (256, 300, 128, 200)
    assert ab.tile_bounds(1, 0, 128, 256, 300, 200) == (128, 256, 0, 200)
