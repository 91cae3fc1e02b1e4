"""CPU oracle for the Stream-K + ABFT GEMM (test infrastructure).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. It shares no code, header, table or helper with the CUDA path and
never imports it.

* ``gemm`` / ``gemm_entries``: the fp64 triple-loop definition of
  ``C = alpha*A*B + beta*C`` (plain C, OpenMP over output rows), from
  "Stream-K: Work-centric Parallel Decomposition for Dense Matrix-Matrix
  Multiplication on the GPU", §A3.
* ``schedule_sim``: the Stream-K schedule simulator (Algorithms 2, 4, 5; §5.2).
* ``abft_ref``: checksum encodings, verify / locate / correct and the
  bit-flip fault model, from "Anatomy of High-Performance GEMM with Online
  Fault Tolerance on GPUs" (thread- and threadblock-level ABFT, Figs. 3, 5).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_ref.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile gemm_ref.c into liboracle.so with gcc + OpenMP (no -ffast-math:
    the sums run in the order the definition states)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        d, L, i = ctypes.c_double, ctypes.c_long, ctypes.c_int
        p = ctypes.c_void_p
        lib.oracle_gemm.argtypes = [L, L, L, d, p, L, i, p, L, i, d, p, L, p, L]
        lib.oracle_gemm.restype = None
        lib.oracle_gemm_entries.argtypes = [L, d, p, L, i, p, L, i, d, p, L, L, p, p, p]
        lib.oracle_gemm_entries.restype = None
        lib.oracle_threads.argtypes = []
        lib.oracle_threads.restype = i
        _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    """Exact widening of a stored matrix (torch or numpy, any float dtype)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dims(A, B, a_layout, b_layout):
    m, k = (A.shape[0], A.shape[1]) if a_layout == 0 else (A.shape[1], A.shape[0])
    kb, n = (B.shape[1], B.shape[0]) if b_layout == 0 else (B.shape[0], B.shape[1])
    if k != kb:
        raise ValueError(f"inner dimensions differ: {k} vs {kb}")
    return m, n, k


def gemm(A, B, alpha: float = 1.0, beta: float = 0.0, C0=None, a_layout: int = 0,
         b_layout: int = 0) -> np.ndarray:
    """C = alpha * A B + beta * C0 in fp64 (the definition, every entry).

    A is stored (m, k) for a_layout 0 or (k, m) for a_layout 1; B is stored
    (n, k) for b_layout 0 ("K-major") or (k, n) for b_layout 1."""
    A64, B64 = _f64(A), _f64(B)
    m, n, k = _dims(A64, B64, a_layout, b_layout)
    C = np.zeros((m, n), dtype=np.float64)
    C064 = _f64(C0) if (beta != 0.0) else np.zeros((1, 1))
    if m and n:
        _load().oracle_gemm(m, n, k, alpha, _ptr(A64), A64.shape[1], a_layout, _ptr(B64),
                            B64.shape[1], b_layout, beta, _ptr(C064), C064.shape[1], _ptr(C), n)
    return C


def gemm_entries(A, B, rows, cols, alpha: float = 1.0, beta: float = 0.0, C0=None,
                 a_layout: int = 0, b_layout: int = 0) -> np.ndarray:
    """The same definition at the entries (rows[s], cols[s]) only.

    Only the rows of A and columns of B the samples touch are widened, so
    this scales to matrices far larger than a full fp64 copy would allow."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    ur, rinv = np.unique(rows, return_inverse=True)
    uc, cinv = np.unique(cols, return_inverse=True)
    if a_layout == 0:
        A_sub = _f64(A[ur.tolist()] if hasattr(A, "detach") else np.asarray(A)[ur])
        k = A_sub.shape[1]
    else:
        A_sub = _f64(A[:, ur.tolist()] if hasattr(A, "detach") else np.asarray(A)[:, ur])
        A_sub = np.ascontiguousarray(A_sub.T)
        k = A_sub.shape[1]
    if b_layout == 0:
        B_sub = _f64(B[uc.tolist()] if hasattr(B, "detach") else np.asarray(B)[uc])
    else:
        B_sub = _f64(B[:, uc.tolist()] if hasattr(B, "detach") else np.asarray(B)[:, uc])
        B_sub = np.ascontiguousarray(B_sub.T)
    if beta != 0.0:
        C0_full = C0
        C0_sub = np.empty((len(ur), len(uc)))
        C0_rows = _f64(C0_full[ur.tolist()] if hasattr(C0_full, "detach") else np.asarray(C0_full)[ur])
        C0_sub[:, :] = C0_rows[:, uc]
    else:
        C0_sub = np.zeros((1, 1))
    out = np.zeros(len(rows), dtype=np.float64)
    ri = np.ascontiguousarray(rinv.astype(np.int64))
    ci = np.ascontiguousarray(cinv.astype(np.int64))
    if len(rows):
        _load().oracle_gemm_entries(k, alpha, _ptr(A_sub), A_sub.shape[1], 0, _ptr(B_sub),
                                    B_sub.shape[1], 0, beta, _ptr(C0_sub), C0_sub.shape[1],
                                    len(rows), _ptr(ri), _ptr(ci), _ptr(out))
    return out


def threads() -> int:
    """OpenMP threads the oracle GEMM runs on."""
    return int(_load().oracle_threads())
