"""ABFT checksum oracle and fault model (test infrastructure, CPU only, fp64).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU legs may import this module; it shares nothing with the
CUDA path.

Follows "Anatomy of High-Performance GEMM with Online Fault Tolerance on
GPUs":

* thread-level FT-GEMM (Fig. 3): the checksums of a product tile are
  ``C^c = e^T A B`` (one value per column) and ``C^r = A B e`` (one value per
  row), with ``e`` the all-ones vector; a fault is located by the positions
  of the mismatching row and column checksums and corrected from the
  checksum offset;
* threadblock-level FT-GEMM (Figs. 5-7): one check per output tile, with the
  encodings ``e^T A`` and ``B e`` taken over the tile and the checksum
  products accumulated over every k step.

Readings (the page is silent on these):

* A mismatch is ``not (|delta| <= tau)``, so a NaN or Inf delta counts.
* Exactly one mismatching row i* and one mismatching column j* make a
  correctable fault at (i*, j*). The corrected value is recomputed from the
  row checksum and the rest of the row, ``C^r[i*] - sum_{j != j*} acc[i*, j]``,
  which survives an Inf/NaN fault. Any other mismatch pattern is reported as
  uncorrectable.
* The check protects the fp32 product ``A B`` of each tile, before alpha,
  beta and the output cast.
"""
from __future__ import annotations

import math
import struct
from typing import Dict, Tuple

import numpy as np

CLEAN = 0
CORRECTED = 1
UNCORRECTABLE = 2


# --------------------------------------------------------------------------
# Encodings and reference checksums (Fig. 3 / Fig. 5 identities)
# --------------------------------------------------------------------------
def encode_cols(A_tile: np.ndarray) -> np.ndarray:
    """e^T A: sum over the tile's rows, one value per k."""
    return A_tile.sum(axis=0)


def encode_rows(B_tile: np.ndarray) -> np.ndarray:
    """B e: sum over the tile's columns, one value per k."""
    return B_tile.sum(axis=1)


def reference_checksums(A: np.ndarray, B: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """(C^c, C^r) = ((e^T A) B, A (B e)) for logical A (rows x k), B (k x cols).

    These are what the checksums of the product must equal; a library matmul
    of a vector serves as a step."""
    cc = encode_cols(A) @ B
    cr = A @ encode_rows(B)
    return cc, cr


def product_checksums(C: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """(e^T C, C e): the column and row sums of a computed product tile."""
    return C.sum(axis=0), C.sum(axis=1)


def tile_bounds(tm: int, tn: int, bm: int, bn: int, m: int, n: int):
    return tm * bm, min(m, (tm + 1) * bm), tn * bn, min(n, (tn + 1) * bn)


def tile_reference(A: np.ndarray, B: np.ndarray, tm: int, tn: int, bm: int, bn: int):
    """Reference checksums of output tile (tm, tn): A is logical m x k, B k x n."""
    m, n = A.shape[0], B.shape[1]
    r0, r1, c0, c1 = tile_bounds(tm, tn, bm, bn, m, n)
    return reference_checksums(A[r0:r1], B[:, c0:c1])


# --------------------------------------------------------------------------
# Detection threshold
# --------------------------------------------------------------------------
def default_tau(k: int, side: int, max_a: float, max_b: float) -> float:
    """Default mismatch threshold for a checksum that sums `side` products of
    length-k dot products, for one output tile whose rows of A are bounded
    by max_a and whose columns of B are bounded by max_b.

    tau = 2^-12 * sqrt(k) * sqrt(side) * max_a * max_b, with side = BLK_N
    for the row checksums and BLK_M for the column checksums. The fault
    tolerance page gives no threshold; this value sits well above the
    rounding of fp32 accumulation and of the split encodings on every
    workload measured, and far below the change an exponent-bit flip makes."""
    return math.ldexp(1.0, -12) * math.sqrt(k) * math.sqrt(side) * max_a * max_b


def tile_maxima(A: np.ndarray, B_stored: np.ndarray, tm: int, tn: int, bm: int, bn: int):
    """(max |A| over the tile's rows, max |B| over the tile's columns); A is
    stored m x k and B stored n x k."""
    return (float(np.abs(A[tm * bm:(tm + 1) * bm]).max()),
            float(np.abs(B_stored[tn * bn:(tn + 1) * bn]).max()))


# --------------------------------------------------------------------------
# Verify / locate / correct (Fig. 3(d)-(f))
# --------------------------------------------------------------------------
def _mismatch(delta: np.ndarray, tau: float) -> np.ndarray:
    return ~(np.abs(delta) <= tau)


def verify_tile(acc: np.ndarray, cr: np.ndarray, cc: np.ndarray, tau_r: float,
                tau_c: float) -> Dict:
    """Check one product tile against its reference checksums.

    Returns status (CLEAN / CORRECTED / UNCORRECTABLE), the mismatching rows
    and columns and, for CORRECTED, the location and the recomputed value."""
    colsum, rowsum = product_checksums(acc)
    d_r = rowsum - cr
    d_c = colsum - cc
    bad_r = np.nonzero(_mismatch(d_r, tau_r))[0]
    bad_c = np.nonzero(_mismatch(d_c, tau_c))[0]
    out = {"bad_rows": bad_r.tolist(), "bad_cols": bad_c.tolist(),
           "max_ratio_r": float(np.max(np.abs(d_r)) / tau_r) if len(d_r) else 0.0,
           "max_ratio_c": float(np.max(np.abs(d_c)) / tau_c) if len(d_c) else 0.0}
    if len(bad_r) == 0 and len(bad_c) == 0:
        out["status"] = CLEAN
    elif len(bad_r) == 1 and len(bad_c) == 1:
        i, j = int(bad_r[0]), int(bad_c[0])
        rest = np.concatenate([acc[i, :j], acc[i, j + 1:]]).sum()
        out.update(status=CORRECTED, row=i, col=j, value=float(cr[i] - rest))
    else:
        out["status"] = UNCORRECTABLE
    return out


# --------------------------------------------------------------------------
# Fault model: a single bit flip of one fp32 accumulator value
# --------------------------------------------------------------------------
def flip_f32(v: float, bit: int) -> float:
    """Round v to fp32 and flip bit `bit` (0 = lowest mantissa bit, 31 = sign)."""
    if not 0 <= bit < 32:
        raise ValueError("bit must be in [0, 32)")
    (u,) = struct.unpack("<I", struct.pack("<f", v))
    (w,) = struct.unpack("<f", struct.pack("<I", u ^ (1 << bit)))
    return w


def f32(v: float) -> float:
    (w,) = struct.unpack("<f", struct.pack("<f", v))
    return w


def exponent_flip_factor(v: float, bit: int) -> float:
    """Closed form for an exponent-bit flip of a normal fp32 value: flipping
    exponent bit e = bit - 23 multiplies v by 2^(+2^e) if that bit was clear
    and by 2^(-2^e) if it was set (while the result stays normal and finite)."""
    if not 23 <= bit <= 30:
        raise ValueError("not an exponent bit")
    (u,) = struct.unpack("<I", struct.pack("<f", v))
    e = bit - 23
    was_set = (u >> bit) & 1
    return 2.0 ** (-(2 ** e)) if was_set else 2.0 ** (2 ** e)


MUST_DETECT = "must"
HARMLESS = "harmless"
GREY = "grey"


def classify_flip(v: float, bit: int, tau: float, elem_tol: float) -> Tuple[str, float]:
    """Class of flipping `bit` of the fp32 accumulator value v, and its delta.

    must-detect: |delta| > 10 tau (or not finite); harmless: |delta| <=
    elem_tol (within the per-element parity tolerance, so neither detection
    nor a miss is wrong); grey: anything between, which the harness re-draws."""
    v32 = f32(v)
    w = flip_f32(v32, bit)
    delta = w - v32 if (math.isfinite(w)) else math.inf
    if not math.isfinite(delta) or abs(delta) > 10.0 * tau:
        return MUST_DETECT, delta
    if abs(delta) <= elem_tol:
        return HARMLESS, delta
    return GREY, delta
