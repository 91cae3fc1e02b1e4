"""ctypes binding of libskgemm.so (include/skgemm.h): argument marshalling only.

Every function here forwards to the C ABI of the same name (without the
``skg_`` prefix). The torch helpers at the bottom only turn tensors into
pointers, leading dimensions and the current stream handle; all arithmetic
runs in the library's CUDA kernels. There is no fallback: if the library is
missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libskgemm.so")

# Enums of skgemm.h
IN_F16, IN_BF16 = 0, 1
OUT_F32, OUT_F16, OUT_BF16 = 0, 1, 2
A_ROW = 0
A_COL = 1
B_KMAJOR = 0
B_NMAJOR = 1
SCHED_DP, SCHED_SK, SCHED_DP_SK1, SCHED_SK2_DP, SCHED_AUTO = 0, 1, 2, 3, 4
ROLE_FULL, ROLE_OWNER, ROLE_PEER = 0, 1, 2
OK = 0
ERR_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE = 1, 2, 3, 4
ERR_FIXUP_TIMEOUT, ERR_PIPELINE_TIMEOUT = 5, 6
ABFT_CORRECTED, ABFT_UNCORRECTABLE = 16, 17
BLK_M, BLK_K = 128, 64
TRACE_CAP, TRACE_STRIDE, MAX_RECORDS = 255, 1024, 64

SCHED_NAMES = {"dp": SCHED_DP, "sk": SCHED_SK, "dp_sk1": SCHED_DP_SK1, "sk2_dp": SCHED_SK2_DP,
               "auto": SCHED_AUTO}


class Opts(ctypes.Structure):
    _fields_ = [("sched", ctypes.c_int32), ("grid", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("abft", ctypes.c_int32), ("tau_row", ctypes.c_float),
                ("tau_col", ctypes.c_float), ("inject_tile", ctypes.c_int32),
                ("inject_row", ctypes.c_int32), ("inject_col", ctypes.c_int32),
                ("inject_bit", ctypes.c_int32), ("timeout_ns", ctypes.c_uint64),
                ("trace", ctypes.c_void_p), ("cta_clock", ctypes.c_void_p),
                ("test_drop_signal", ctypes.c_int32), ("abft_preencoded", ctypes.c_int32),
                ("raster_band", ctypes.c_int32), ("cta_pair", ctypes.c_int32),
                ("abft_local", ctypes.c_int32), ("inject2_tile", ctypes.c_int32),
                ("inject2_row", ctypes.c_int32), ("inject2_col", ctypes.c_int32),
                ("inject2_bit", ctypes.c_int32), ("inject_kstep", ctypes.c_int32),
                ("stagger", ctypes.c_int32), ("abft_inloop", ctypes.c_int32)]


class Segment(ctypes.Structure):
    _fields_ = [("cta", ctypes.c_int32), ("tile", ctypes.c_int32),
                ("k_iter_begin", ctypes.c_int32), ("k_iter_end", ctypes.c_int32),
                ("role", ctypes.c_int32)]


class FaultRecord(ctypes.Structure):
    _fields_ = [("launch", ctypes.c_uint32), ("tile", ctypes.c_int32), ("row", ctypes.c_int32),
                ("col", ctypes.c_int32), ("status", ctypes.c_int32),
                ("n_bad_rows", ctypes.c_int32), ("n_bad_cols", ctypes.c_int32),
                ("injected", ctypes.c_uint32), ("before", ctypes.c_float),
                ("after", ctypes.c_float), ("delta_row", ctypes.c_float),
                ("delta_col", ctypes.c_float), ("clean_value", ctypes.c_float),
                ("pad", ctypes.c_uint32 * 3)]


class Plan(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("ctas", ctypes.c_int32),
                ("cta_pair", ctypes.c_int32), ("sched", ctypes.c_int32),
                ("side_ctas", ctypes.c_int32), ("fused_checksums", ctypes.c_int32),
                ("encode_in_kernel", ctypes.c_int32), ("local_checksums", ctypes.c_int32),
                ("inloop_checksums", ctypes.c_int32), ("side_checksum_ctas", ctypes.c_int32)]


class Report(ctypes.Structure):
    _fields_ = [("status_bits", ctypes.c_uint32), ("launches", ctypes.c_uint32),
                ("tiles_checked", ctypes.c_uint32), ("detected", ctypes.c_uint32),
                ("corrected", ctypes.c_uint32), ("uncorrectable", ctypes.c_uint32),
                ("timeouts", ctypes.c_uint32), ("n_records", ctypes.c_uint32),
                ("max_ratio_row", ctypes.c_float), ("max_ratio_col", ctypes.c_float),
                ("tau_row", ctypes.c_float), ("tau_col", ctypes.c_float),
                ("mid_injected", ctypes.c_uint32), ("mid_before", ctypes.c_float),
                ("mid_after", ctypes.c_float), ("reserved", ctypes.c_uint32),
                ("records", FaultRecord * MAX_RECORDS)]


SYMBOLS = ("skg_opts_default", "skg_workspace_size", "skg_workspace_init", "skg_gemm",
           "skg_gemm_verify", "skg_abft_encode", "skg_schedule_query", "skg_launch_shape", "skg_report_read",
           "skg_device_sm_count", "skg_status_string", "skg_gemm_noalloc", "skg_schedule_cost",
           "skg_launch_plan", "skg_workspace_size_layout", "skg_host_staging_size",
           "skg_gemm_host", "skg_abft_encode_layout", "skg_workspace_size_f64", "skg_gemm_f64",
           "skg_noalloc_report_read")

_lib = None


class SkgError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


def lib() -> ctypes.CDLL:
    """Load libskgemm.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build(); "
                           "there is no CPU fallback")
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, sz, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
    f32 = ctypes.c_float
    L.skg_opts_default.argtypes = [ctypes.POINTER(Opts)]
    L.skg_opts_default.restype = None
    L.skg_workspace_size.argtypes = [i64, i64, i64, ctypes.POINTER(Opts)]
    L.skg_workspace_size.restype = sz
    L.skg_workspace_size_layout.argtypes = [i64, i64, i64, i32, i32, ctypes.POINTER(Opts)]
    L.skg_workspace_size_layout.restype = sz
    L.skg_workspace_init.argtypes = [vp, sz, vp]
    L.skg_workspace_init.restype = i32
    gemm_args = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, i32, i32, i32, i32,
                 ctypes.POINTER(Opts), vp, sz, vp]
    L.skg_gemm.argtypes = gemm_args
    L.skg_gemm.restype = i32
    f64 = ctypes.c_double
    L.skg_workspace_size_f64.argtypes = [i64, i64, i64, ctypes.POINTER(Opts)]
    L.skg_workspace_size_f64.restype = sz
    L.skg_gemm_f64.argtypes = [i64, i64, i64, f64, vp, i64, vp, i64, f64, vp, i64,
                               ctypes.POINTER(Opts), vp, sz, vp]
    L.skg_gemm_f64.restype = i32
    L.skg_host_staging_size.argtypes = [i64, i64, i64, i32, i32, i32, i32]
    L.skg_host_staging_size.restype = sz
    L.skg_gemm_host.argtypes = gemm_args[:-3] + [vp, sz, vp, sz, vp]
    L.skg_gemm_host.restype = i32
    L.skg_gemm_verify.argtypes = gemm_args
    L.skg_gemm_verify.restype = i32
    L.skg_abft_encode.argtypes = [i64, i64, i64, vp, i64, vp, i64, i32, ctypes.POINTER(Opts),
                                  vp, sz, vp]
    L.skg_abft_encode.restype = i32
    L.skg_abft_encode_layout.argtypes = [i64, i64, i64, vp, i64, vp, i64, i32, i32, i32,
                                         ctypes.POINTER(Opts), vp, sz, vp]
    L.skg_abft_encode_layout.restype = i32
    L.skg_schedule_query.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32,
                                     ctypes.POINTER(Segment), i64, ctypes.POINTER(i64)]
    L.skg_schedule_query.restype = i32
    L.skg_schedule_cost.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32,
                                    ctypes.POINTER(ctypes.c_double)]
    L.skg_schedule_cost.restype = i32
    L.skg_launch_shape.argtypes = [i64, i64, i64, ctypes.POINTER(Opts), ctypes.POINTER(i32),
                                   ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.skg_launch_shape.restype = i32
    L.skg_launch_plan.argtypes = [i64, i64, i64, ctypes.POINTER(Opts), ctypes.POINTER(Plan)]
    L.skg_launch_plan.restype = i32
    L.skg_report_read.argtypes = [vp, ctypes.POINTER(Report), i32, vp]
    L.skg_report_read.restype = i32
    L.skg_gemm_noalloc.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, i32,
                                   i32, i32, i32, ctypes.POINTER(Opts), vp]
    L.skg_gemm_noalloc.restype = i32
    L.skg_noalloc_report_read.argtypes = [ctypes.POINTER(Report), i32, vp]
    L.skg_noalloc_report_read.restype = i32
    L.skg_device_sm_count.argtypes = []
    L.skg_device_sm_count.restype = i32
    L.skg_status_string.argtypes = [i32]
    L.skg_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


# ---------------------------------------------------------------- C ABI 1:1
def opts_default(**kw) -> Opts:
    o = Opts()
    lib().skg_opts_default(ctypes.byref(o))
    for key, val in kw.items():
        if key == "sched" and isinstance(val, str):
            val = SCHED_NAMES[val]
        setattr(o, key, val)
    return o


def workspace_size(m: int, n: int, k: int, opts: Optional[Opts] = None) -> int:
    return int(lib().skg_workspace_size(m, n, k, ctypes.byref(opts) if opts else None))


def workspace_size_layout(m: int, n: int, k: int, a_layout: int, b_layout: int,
                          opts: Optional[Opts] = None) -> int:
    return int(lib().skg_workspace_size_layout(m, n, k, a_layout, b_layout,
                                               ctypes.byref(opts) if opts else None))


def workspace_init(ws_ptr: int, nbytes: int, stream: int = 0) -> int:
    return int(lib().skg_workspace_init(ws_ptr, nbytes, stream))


def gemm(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, in_dtype, out_dtype,
         a_layout, b_layout, opts, ws_ptr, ws_bytes, stream) -> int:
    return int(lib().skg_gemm(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc,
                              in_dtype, out_dtype, a_layout, b_layout,
                              ctypes.byref(opts) if opts else None, ws_ptr, ws_bytes, stream))


def workspace_size_f64(m: int, n: int, k: int, opts: Optional[Opts] = None) -> int:
    return int(lib().skg_workspace_size_f64(m, n, k, ctypes.byref(opts) if opts else None))


def gemm_f64(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, opts, ws_ptr, ws_bytes,
             stream) -> int:
    """skg_gemm_f64: fp64 Stream-K GEMM on device pointers."""
    return int(lib().skg_gemm_f64(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc,
                                  ctypes.byref(opts) if opts else None, ws_ptr, ws_bytes,
                                  stream))


def host_staging_size(m, n, k, in_dtype, out_dtype, a_layout=A_ROW, b_layout=B_KMAJOR) -> int:
    return int(lib().skg_host_staging_size(m, n, k, in_dtype, out_dtype, a_layout, b_layout))


def gemm_host(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, in_dtype, out_dtype,
              a_layout, b_layout, opts, staging_ptr, staging_bytes, ws_ptr, ws_bytes,
              stream) -> int:
    """skg_gemm_host: A, B, C are host addresses; staging and workspace are
    device memory."""
    return int(lib().skg_gemm_host(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc,
                                   in_dtype, out_dtype, a_layout, b_layout,
                                   ctypes.byref(opts) if opts else None, staging_ptr,
                                   staging_bytes, ws_ptr, ws_bytes, stream))


def gemm_verify(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, in_dtype, out_dtype,
                a_layout, b_layout, opts, ws_ptr, ws_bytes, stream) -> int:
    return int(lib().skg_gemm_verify(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc,
                                     in_dtype, out_dtype, a_layout, b_layout,
                                     ctypes.byref(opts) if opts else None, ws_ptr, ws_bytes,
                                     stream))


def abft_encode(m, n, k, A_ptr, lda, B_ptr, ldb, in_dtype, opts, ws_ptr, ws_bytes,
                stream, a_layout: int = A_ROW, b_layout: int = B_KMAJOR) -> int:
    """skg_abft_encode (K-major operands) or skg_abft_encode_layout."""
    o = ctypes.byref(opts) if opts else None
    if a_layout == A_ROW and b_layout == B_KMAJOR:
        return int(lib().skg_abft_encode(m, n, k, A_ptr, lda, B_ptr, ldb, in_dtype, o, ws_ptr,
                                         ws_bytes, stream))
    return int(lib().skg_abft_encode_layout(m, n, k, A_ptr, lda, B_ptr, ldb, in_dtype, a_layout,
                                            b_layout, o, ws_ptr, ws_bytes, stream))


def schedule_query(m: int, n: int, k: int, bm: int, bn: int, bk: int, g: int,
                   sched) -> List[Tuple[int, int, int, int, int]]:
    """(cta, tile, k_iter_begin, k_iter_end, role) rows, CTA by CTA."""
    if isinstance(sched, str):
        sched = SCHED_NAMES[sched]
    count = ctypes.c_int64(0)
    st = lib().skg_schedule_query(m, n, k, bm, bn, bk, g, sched, None, 0, ctypes.byref(count))
    if st != OK:
        raise SkgError(st, "skg_schedule_query")
    buf = (Segment * max(1, count.value))()
    st = lib().skg_schedule_query(m, n, k, bm, bn, bk, g, sched, buf, count.value,
                                  ctypes.byref(count))
    if st != OK:
        raise SkgError(st, "skg_schedule_query")
    return [(s.cta, s.tile, s.k_iter_begin, s.k_iter_end, s.role) for s in buf[:count.value]]


def schedule_cost(m: int, n: int, k: int, bm: int, bn: int, bk: int, g: int, sched) -> float:
    """Grid-size model's predicted time (us) of one launch."""
    if isinstance(sched, str):
        sched = SCHED_NAMES[sched]
    us = ctypes.c_double(0.0)
    st = lib().skg_schedule_cost(m, n, k, bm, bn, bk, g, sched, ctypes.byref(us))
    if st != OK:
        raise SkgError(st, "skg_schedule_cost")
    return us.value


def launch_plan(m: int, n: int, k: int, opts: Optional[Opts] = None) -> Plan:
    """The launch plan skg_gemm would use (tile shape, CTAs, pairs, schedule,
    checksum-tile placement)."""
    out = Plan()
    st = lib().skg_launch_plan(m, n, k, ctypes.byref(opts) if opts else None, ctypes.byref(out))
    if st != OK:
        raise SkgError(st, "skg_launch_plan")
    return out


def launch_shape(m: int, n: int, k: int, opts: Optional[Opts] = None) -> Tuple[int, int, int]:
    """(BLK_N, g, schedule) skg_gemm would use."""
    tn, g, sc = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    st = lib().skg_launch_shape(m, n, k, ctypes.byref(opts) if opts else None, ctypes.byref(tn),
                                ctypes.byref(g), ctypes.byref(sc))
    if st != OK:
        raise SkgError(st, "skg_launch_shape")
    return tn.value, g.value, sc.value


def report_read(ws_ptr: int, reset: bool = False, stream: int = 0) -> Report:
    rep = Report()
    st = lib().skg_report_read(ws_ptr, ctypes.byref(rep), 1 if reset else 0, stream)
    if st != OK:
        raise SkgError(st, "skg_report_read")
    return rep


def gemm_noalloc(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc, in_dtype, out_dtype,
                 a_layout, b_layout, opts, stream) -> int:
    """skg_gemm_noalloc: skg_gemm with the workspace taken from the library's
    fixed device scratch array, for callers that cannot allocate."""
    return int(lib().skg_gemm_noalloc(m, n, k, alpha, A_ptr, lda, B_ptr, ldb, beta, C_ptr, ldc,
                                      in_dtype, out_dtype, a_layout, b_layout,
                                      ctypes.byref(opts) if opts else None, stream))


def noalloc_report_read(reset: bool = False, stream: int = 0) -> Report:
    """skg_noalloc_report_read: the report of skg_gemm_noalloc's array."""
    rep = Report()
    st = lib().skg_noalloc_report_read(ctypes.byref(rep), 1 if reset else 0, stream)
    if st != OK:
        raise SkgError(st, "skg_noalloc_report_read")
    return rep


def device_sm_count() -> int:
    return int(lib().skg_device_sm_count())


def status_string(code: int) -> str:
    return lib().skg_status_string(code).decode()


# ---------------------------------------------------------------- torch marshalling
_IN = {"f16": IN_F16, "bf16": IN_BF16}
_OUT = {"f32": OUT_F32, "f16": OUT_F16, "bf16": OUT_BF16}


def _dt_name(t) -> str:
    import torch
    return {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}[t.dtype]


class Workspace:
    """Caller-owned device workspace (a torch byte buffer), zeroed once."""

    def __init__(self, nbytes: int, device="cuda"):
        import torch
        self.nbytes = int(nbytes)
        self.buf = torch.empty(max(self.nbytes, 1), dtype=torch.uint8, device=device)
        st = workspace_init(self.buf.data_ptr(), self.nbytes,
                            torch.cuda.current_stream(self.buf.device).cuda_stream)
        if st != OK:
            raise SkgError(st, "skg_workspace_init")

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def report(self, reset: bool = False) -> Report:
        import torch
        return report_read(self.ptr, reset, torch.cuda.current_stream(self.buf.device).cuda_stream)


def matmul(A, B, C, alpha: float = 1.0, beta: float = 0.0, opts: Optional[Opts] = None,
           workspace: Optional[Workspace] = None, verify: bool = False, stream=None,
           a_layout: int = A_ROW, b_layout: int = B_KMAJOR):
    """C = alpha * op(A) op(B) + beta * C through skg_gemm (or skg_gemm_verify).

    A: (m, k) row-major (a_layout A_ROW) or (k, m) (A_COL); B: (n, k)
    ("K-major", B_KMAJOR) or (k, n) (B_NMAJOR); C: (m, n). All on the same
    CUDA device, unit stride in the last dimension. Returns C."""
    import torch
    m, k = A.shape if a_layout == A_ROW else A.shape[::-1]
    n, kb = B.shape if b_layout == B_KMAJOR else B.shape[::-1]
    if kb != k or tuple(C.shape) != (m, n):
        raise ValueError("shape mismatch")
    for t in (A, B, C):
        if t.stride(-1) != 1:
            raise ValueError("last dimension must be contiguous")
    if A.dtype != B.dtype:
        raise ValueError("A and B must have the same dtype")
    if workspace is None:
        workspace = Workspace(workspace_size_layout(m, n, k, a_layout, b_layout, opts), A.device)
    st_handle = (stream or torch.cuda.current_stream(A.device)).cuda_stream
    fn = gemm_verify if verify else gemm
    st = fn(m, n, k, alpha, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), beta,
            C.data_ptr(), C.stride(0), _IN[_dt_name(A)], _OUT[_dt_name(C)], a_layout, b_layout,
            opts, workspace.ptr, workspace.nbytes, st_handle)
    if st != OK:
        raise SkgError(st, "skg_gemm_verify" if verify else "skg_gemm")
    return C
