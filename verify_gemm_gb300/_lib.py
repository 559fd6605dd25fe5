"""ctypes binding of libvgemm.so: one Python callable per C entry point,
same names, argument marshalling only (no computation happens here).

The library must exist: if ``_build/libvgemm.so`` is missing the binding
raises instead of falling back to anything else.  Build it with
``python -m verify_gemm_gb300.build`` (``__graft_entry__.build()`` does).
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libvgemm.so")

VG_OK = 0
VG_ERR_INVALID_ARG = 1
VG_ERR_ALIGNMENT = 2
VG_ERR_UNSUPPORTED = 3
VG_ERR_CUDA = 4
VG_ERR_TIMEOUT = 5
VG_ERR_WORKSPACE = 6
VG_FMT_NVFP4 = 0
VG_FMT_FP8_ROWSCALE = 1
VG_FMT_MXFP8 = 2
VG_FMT_INT4G = 3
VG_OP_GEMV = 0
VG_OP_SWIGLU = 1
VG_OP_RMSNORM = 2

P = ctypes.c_void_p
i64 = ctypes.c_int64
i32 = ctypes.c_int
sz = ctypes.c_size_t
f32 = ctypes.c_float
st = ctypes.c_int   # vg_status


class vg_matrix_desc(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("group", ctypes.c_int32), ("M", i64), ("K", i64),
                ("w", P), ("scales", P), ("rowscale", P), ("gscale", f32), ("x", P), ("y", P),
                ("op", ctypes.c_int32), ("x_after_group", ctypes.c_int32), ("gscale_up", f32),
                ("eps", f32), ("rowscale_up", P), ("gamma", P)]


class vg_plan_options(ctypes.Structure):
    _fields_ = [("ordered", ctypes.c_int32), ("max_ctas", ctypes.c_int32),
                ("wait_timeout_ns", i64), ("hold_group", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


SIGNATURES = {
    "vg_status_string": (ctypes.c_char_p, [st]),
    "vg_version": (i32, []),
    "vg_last_cuda_error": (ctypes.c_char_p, []),
    "vg_nvfp4_sizes": (st, [i64, i64, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
    "vg_fp8_sizes": (st, [i64, i64, ctypes.POINTER(sz)]),
    "vg_nvfp4_pack": (st, [P, i64, i64, P, P, ctypes.POINTER(f32), P]),
    "vg_fp8_pack": (st, [P, i64, i64, P, P, P]),
    "vg_nvfp4_unpack": (st, [P, P, i64, i64, P, P, P]),
    "vg_fp8_unpack": (st, [P, i64, i64, P, P]),
    "vg_fp8_rowscale_pack": (st, [P, i64, i64, P, P, P]),
    "vg_fp8_rowscale_unpack": (st, [P, i64, i64, P, P]),
    "vg_nvfp4_from_canonical": (st, [P, P, i64, i64, P, P, P]),
    "vg_nvfp4_pack_gated": (st, [P, P, i64, i64, P, P, ctypes.POINTER(f32), P]),
    "vg_fp8_pack_gated": (st, [P, P, i64, i64, P, P, P, P]),
    "vg_fp8_from_canonical": (st, [P, i64, i64, P, P]),
    "vg_weight_sizes": (st, [i32, i64, i64, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
    "vg_mxfp8_pack": (st, [P, i64, i64, P, P, P]),
    "vg_int4g_pack": (st, [P, i64, i64, P, P, P]),
    "vg_mxfp8_unpack": (st, [P, P, i64, i64, P, P, P]),
    "vg_int4g_unpack": (st, [P, P, i64, i64, P, P, P]),
    "vg_mxfp8_from_canonical": (st, [P, P, i64, i64, P, P, P]),
    "vg_int4g_from_canonical": (st, [P, P, i64, i64, P, P, P]),
    "vg_gemv_mxfp8": (st, [P, P, P, i32, i64, i64, P, P, sz, P]),
    "vg_gemv_int4g": (st, [P, P, P, i32, i64, i64, P, P, sz, P]),
    "vg_gemv_workspace_size": (st, [i64, i64, i32, ctypes.POINTER(sz)]),
    "vg_gemv_workspace_size_n": (st, [i64, i64, i32, i32, ctypes.POINTER(sz)]),
    "vg_gemv_nvfp4": (st, [P, P, f32, P, i32, i64, i64, P, P, sz, P]),
    "vg_gemv_fp8_rowscale": (st, [P, P, P, i32, i64, i64, P, P, sz, P]),
    "vg_gemv_workspace_check": (st, [P, sz, ctypes.POINTER(i32), P]),
    "vg_gemv_nvfp4_noalloc": (st, [P, P, f32, P, i32, i64, i64, P, P]),
    "vg_gemv_nvfp4_noalloc_check": (st, [ctypes.POINTER(i32), P]),
    "vg_hbm_read_probe": (st, [P, sz, i32, i32, i32, P, i32, P]),
    "vg_verify_plan_create": (st, [ctypes.POINTER(vg_matrix_desc), i32, i32, i32,
                                   ctypes.POINTER(P)]),
    "vg_verify_plan_create_ex": (st, [ctypes.POINTER(vg_matrix_desc), i32, i32,
                                      ctypes.POINTER(vg_plan_options), ctypes.POINTER(P)]),
    "vg_verify_pass": (st, [P, P]),
    "vg_verify_plan_set_width": (st, [P, P]),
    "vg_verify_plan_check": (st, [P, P, ctypes.POINTER(i32)]),
    "vg_verify_plan_bytes": (st, [P, ctypes.POINTER(i64)]),
    "vg_verify_plan_grid": (st, [P, ctypes.POINTER(i32)]),
    "vg_verify_plan_destroy": (st, [P]),
}

_lock = threading.Lock()
_lib = None


class VGError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.vg_status_string(status).decode()
        extra = lib.vg_last_cuda_error().decode() if status == VG_ERR_CUDA else ""
        super().__init__(f"{where}: {msg} ({status}) {extra}".strip())
        self.status = status


def load():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:      # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libvgemm.so not found at {LIB_PATH}; build it with "
                    "`python -m verify_gemm_gb300.build` (there is no fallback path)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def check(status: int, where: str):
    if status != VG_OK:
        raise VGError(status, where)


def __getattr__(name):
    if name in SIGNATURES:
        return getattr(load(), name)
    raise AttributeError(name)
