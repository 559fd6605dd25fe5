"""CPU oracle for the NVFP4 / row-scaled FP8 verify GEMV.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this package.  The product package ``verify_gemm_gb300`` never imports it,
and this package imports nothing from the product.

The arithmetic lives in ``vg_oracle.c`` (plain C, FP64 accumulation); this
module only builds it with gcc and marshals numpy arrays through ctypes.
Layouts are canonical: ``nib[M, K/2]`` (low nibble = even k), ``sc[M, K/16]``
E4M3 bytes, ``gs`` FP32; FP8 ``q[M, K]`` with FP32 ``rs[M]``; ``x[N, K]`` as
BF16 bit patterns (uint16); results ``y[N, rows]`` and ``a[N, rows]``
(``a`` = sum of |w*x|, the scale of the tolerance).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vg_oracle.c")
_HDR = os.path.join(_HERE, "vg_oracle.h")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Pass criterion of the verify GEMV: |y - y_ref| <= REL * sum|w*x| + ABS.
REL_TOL = 4e-3
ABS_TOL = 1e-6


def build(force: bool = False) -> str:
    """Compile vg_oracle.c into oracle/_build/liboracle.so with gcc."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    stale = not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or stale:
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = [
            "gcc", "-O2", "-std=c99", "-D_GNU_SOURCE", "-ffp-contract=off",
            "-fno-fast-math", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC,
            "-lm", "-lpthread",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _declare(lib):
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    sig = {
        "vgo_e2m1_value": (ctypes.c_double, [ctypes.c_int]),
        "vgo_e4m3_value": (ctypes.c_double, [ctypes.c_int]),
        "vgo_bf16_value": (ctypes.c_double, [ctypes.c_uint16]),
        "vgo_e4m3_encode": (ctypes.c_int, [ctypes.c_float]),
        "vgo_e2m1_encode": (ctypes.c_int, [ctypes.c_float]),
        "vgo_nvfp4_quantise": (ctypes.c_int, [P, i64, i64, P, P, P]),
        "vgo_fp8_quantise": (ctypes.c_int, [P, i64, i64, P, P]),
        "vgo_amax": (ctypes.c_float, [P, i64]),
        "vgo_nvfp4_quantise_gs": (None, [P, i64, i64, ctypes.c_float, P, P]),
        "vgo_nvfp4_dequant": (None, [P, P, ctypes.c_float, i64, i64, P]),
        "vgo_fp8_dequant": (None, [P, P, i64, i64, P]),
        "vgo_gemv_nvfp4": (None, [P, P, ctypes.c_float, P, ctypes.c_int, i64, i64,
                                  P, i64, P, P, ctypes.c_int]),
        "vgo_gemv_fp8": (None, [P, P, P, ctypes.c_int, i64, i64, P, i64, P, P,
                                ctypes.c_int]),
        "vgo_e8m0_value": (ctypes.c_double, [ctypes.c_int]),
        "vgo_mxfp8_quantise": (ctypes.c_int, [P, i64, i64, P, P]),
        "vgo_int4g_quantise": (ctypes.c_int, [P, i64, i64, P, P]),
        "vgo_mxfp8_dequant": (None, [P, P, i64, i64, P]),
        "vgo_int4g_dequant": (None, [P, P, i64, i64, P]),
        "vgo_gemv_mxfp8": (None, [P, P, P, ctypes.c_int, i64, i64, P, i64, P, P, ctypes.c_int]),
        "vgo_gemv_int4g": (None, [P, P, P, ctypes.c_int, i64, i64, P, i64, P, P, ctypes.c_int]),
        "vgo_bf16_round": (ctypes.c_uint16, [ctypes.c_double]),
        "vgo_silu": (ctypes.c_double, [ctypes.c_double]),
        "vgo_swiglu": (None, [P, P, P, P, i64, P, P]),
        "vgo_rmsnorm": (None, [P, P, ctypes.c_int, i64, ctypes.c_double, P]),
        "vgo_check": (ctypes.c_int64, [P, P, P, i64, ctypes.c_double, ctypes.c_double,
                                       ctypes.POINTER(ctypes.c_double)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str | None = None):
    """The oracle library (built on first use).  ``path`` loads another build
    of the same source (used by the planted-mistake tests)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            build()
            _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """numpy-facing wrappers around one build of the oracle library."""

    REL_TOL = REL_TOL
    ABS_TOL = ABS_TOL

    def __init__(self, lib):
        self.lib = lib

    # -------------------------------------------------------- scalar codes
    def e2m1_value(self, code):
        return self.lib.vgo_e2m1_value(int(code))

    def e4m3_value(self, byte):
        return self.lib.vgo_e4m3_value(int(byte))

    def bf16_value(self, bits):
        return self.lib.vgo_bf16_value(int(bits))

    def e4m3_encode(self, v):
        return self.lib.vgo_e4m3_encode(float(np.float32(v)))

    def e2m1_encode(self, v):
        return self.lib.vgo_e2m1_encode(float(np.float32(v)))

    # ---------------------------------------------------------- quantisers
    def nvfp4_quantise(self, W):
        """FP32 [M, K] -> (nib uint8 [M, K/2], sc uint8 [M, K/16], gs float)."""
        W = np.ascontiguousarray(W, dtype=np.float32)
        M, K = W.shape
        if K % 16:
            raise ValueError("K must be a multiple of 16")
        nib = np.zeros((M, K // 2), np.uint8)
        sc = np.zeros((M, K // 16), np.uint8)
        gs = np.zeros(1, np.float32)
        if self.lib.vgo_nvfp4_quantise(_ptr(W), M, K, _ptr(nib), _ptr(sc), _ptr(gs)):
            raise ValueError("non-finite weight")
        return nib, sc, float(gs[0])

    def amax(self, W):
        W = np.ascontiguousarray(W, dtype=np.float32)
        return float(self.lib.vgo_amax(_ptr(W), W.size))

    def nvfp4_quantise_gs(self, W, gs):
        """Per-block NVFP4 quantisation of rows W [R, K] with a given gs."""
        W = np.ascontiguousarray(W, dtype=np.float32)
        M, K = W.shape
        nib = np.zeros((M, K // 2), np.uint8)
        sc = np.zeros((M, K // 16), np.uint8)
        self.lib.vgo_nvfp4_quantise_gs(_ptr(W), M, K, float(gs), _ptr(nib), _ptr(sc))
        return nib, sc

    def fp8_quantise(self, W):
        """FP32 [M, K] -> (q uint8 [M, K], rs float32 [M])."""
        W = np.ascontiguousarray(W, dtype=np.float32)
        M, K = W.shape
        q = np.zeros((M, K), np.uint8)
        rs = np.zeros(M, np.float32)
        if self.lib.vgo_fp8_quantise(_ptr(W), M, K, _ptr(q), _ptr(rs)):
            raise ValueError("non-finite weight")
        return q, rs

    def nvfp4_dequant(self, nib, sc, gs, M, K):
        out = np.zeros((M, K), np.float64)
        self.lib.vgo_nvfp4_dequant(_ptr(np.ascontiguousarray(nib)),
                                   _ptr(np.ascontiguousarray(sc)), float(gs), M, K, _ptr(out))
        return out

    def fp8_dequant(self, q, rs, M, K):
        out = np.zeros((M, K), np.float64)
        self.lib.vgo_fp8_dequant(_ptr(np.ascontiguousarray(q)),
                                 _ptr(np.ascontiguousarray(rs, dtype=np.float32)), M, K,
                                 _ptr(out))
        return out

    # ---------------------------------------------------------------- gemv
    @staticmethod
    def _rows(rows, M):
        if rows is None:
            return None, M
        r = np.ascontiguousarray(rows, dtype=np.int64)
        if r.size and (r.min() < 0 or r.max() >= M):
            raise ValueError("row index out of range")
        return r, r.size

    def gemv_nvfp4(self, nib, sc, gs, x_bits, rows=None, threads=1):
        """FP64 y[N, rows], a[N, rows] for canonical NVFP4 weights."""
        nib = np.ascontiguousarray(nib, dtype=np.uint8)
        sc = np.ascontiguousarray(sc, dtype=np.uint8)
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        M, K = nib.shape[0], nib.shape[1] * 2
        N = x_bits.shape[0]
        assert x_bits.shape[1] == K and sc.shape == (M, K // 16)
        r, nr = self._rows(rows, M)
        y = np.zeros((N, nr), np.float64)
        a = np.zeros((N, nr), np.float64)
        self.lib.vgo_gemv_nvfp4(_ptr(nib), _ptr(sc), float(gs), _ptr(x_bits), N, M, K,
                                None if r is None else _ptr(r), nr, _ptr(y), _ptr(a),
                                int(threads))
        return y, a

    def gemv_fp8(self, q, rs, x_bits, rows=None, threads=1):
        """FP64 y[N, rows], a[N, rows] for canonical row-scaled FP8 weights."""
        q = np.ascontiguousarray(q, dtype=np.uint8)
        rs = np.ascontiguousarray(rs, dtype=np.float32)
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        M, K = q.shape
        N = x_bits.shape[0]
        assert x_bits.shape[1] == K and rs.shape == (M,)
        r, nr = self._rows(rows, M)
        y = np.zeros((N, nr), np.float64)
        a = np.zeros((N, nr), np.float64)
        self.lib.vgo_gemv_fp8(_ptr(q), _ptr(rs), _ptr(x_bits), N, M, K,
                              None if r is None else _ptr(r), nr, _ptr(y), _ptr(a),
                              int(threads))
        return y, a

    # --------------------------------------------------------- other formats
    def e8m0_value(self, byte):
        return self.lib.vgo_e8m0_value(int(byte))

    def mxfp8_quantise(self, W):
        """MXFP8: q [M, K] E4M3 bytes, sc [M, K/32] E8M0 bytes."""
        W = np.ascontiguousarray(W, dtype=np.float32)
        M, K = W.shape
        assert K % 32 == 0
        q = np.zeros((M, K), np.uint8)
        sc = np.zeros((M, K // 32), np.uint8)
        if self.lib.vgo_mxfp8_quantise(_ptr(W), M, K, _ptr(q), _ptr(sc)) != 0:
            raise ValueError("non-finite weight")
        return q, sc

    def int4g_quantise(self, W):
        """Groupwise INT4: nib [M, K/2] codes, sc [M, K/128] BF16 bits."""
        W = np.ascontiguousarray(W, dtype=np.float32)
        M, K = W.shape
        assert K % 128 == 0
        nib = np.zeros((M, K // 2), np.uint8)
        sc = np.zeros((M, K // 128), np.uint16)
        if self.lib.vgo_int4g_quantise(_ptr(W), M, K, _ptr(nib), _ptr(sc)) != 0:
            raise ValueError("non-finite weight")
        return nib, sc

    def mxfp8_dequant(self, q, sc, M, K):
        out = np.zeros((M, K), np.float64)
        self.lib.vgo_mxfp8_dequant(_ptr(np.ascontiguousarray(q, dtype=np.uint8)),
                                   _ptr(np.ascontiguousarray(sc, dtype=np.uint8)), M, K,
                                   _ptr(out))
        return out

    def int4g_dequant(self, nib, sc, M, K):
        out = np.zeros((M, K), np.float64)
        self.lib.vgo_int4g_dequant(_ptr(np.ascontiguousarray(nib, dtype=np.uint8)),
                                   _ptr(np.ascontiguousarray(sc, dtype=np.uint16)), M, K,
                                   _ptr(out))
        return out

    def gemv_mxfp8(self, q, sc, x_bits, rows=None, threads=1):
        q = np.ascontiguousarray(q, dtype=np.uint8)
        sc = np.ascontiguousarray(sc, dtype=np.uint8)
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        M, K = q.shape
        N = x_bits.shape[0]
        assert x_bits.shape[1] == K and sc.shape == (M, K // 32)
        r, nr = self._rows(rows, M)
        y = np.zeros((N, nr), np.float64)
        a = np.zeros((N, nr), np.float64)
        self.lib.vgo_gemv_mxfp8(_ptr(q), _ptr(sc), _ptr(x_bits), N, M, K,
                                None if r is None else _ptr(r), nr, _ptr(y), _ptr(a),
                                int(threads))
        return y, a

    def gemv_int4g(self, nib, sc, x_bits, rows=None, threads=1):
        nib = np.ascontiguousarray(nib, dtype=np.uint8)
        sc = np.ascontiguousarray(sc, dtype=np.uint16)
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        M, K = nib.shape[0], nib.shape[1] * 2
        N = x_bits.shape[0]
        assert x_bits.shape[1] == K and sc.shape == (M, K // 128)
        r, nr = self._rows(rows, M)
        y = np.zeros((N, nr), np.float64)
        a = np.zeros((N, nr), np.float64)
        self.lib.vgo_gemv_int4g(_ptr(nib), _ptr(sc), _ptr(x_bits), N, M, K,
                                None if r is None else _ptr(r), nr, _ptr(y), _ptr(a),
                                int(threads))
        return y, a

    # ----------------------------------------------------- fused neighbours
    def bf16_round(self, v):
        return self.lib.vgo_bf16_round(float(v))

    def silu(self, g):
        return self.lib.vgo_silu(float(g))

    def swiglu(self, g, u, ag, au):
        """h = SiLU(g) * u and its acceptance bound (FP64, same shapes)."""
        g, u, ag, au = (np.ascontiguousarray(v, dtype=np.float64) for v in (g, u, ag, au))
        h = np.empty_like(g)
        b = np.empty_like(g)
        self.lib.vgo_swiglu(_ptr(g), _ptr(u), _ptr(ag), _ptr(au), g.size, _ptr(h), _ptr(b))
        return h, b

    def rmsnorm(self, x_bits, gamma_bits, eps=1e-6):
        """BF16 bits of RMSNorm(x) * gamma, x [N, K], gamma [K] as BF16 bits."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        gamma_bits = np.ascontiguousarray(gamma_bits, dtype=np.uint16)
        N, K = x_bits.shape
        assert gamma_bits.shape == (K,)
        out = np.empty_like(x_bits)
        self.lib.vgo_rmsnorm(_ptr(x_bits), _ptr(gamma_bits), N, K, float(eps), _ptr(out))
        return out

    def check(self, y_bits, yref, a, rel=REL_TOL, abs_tol=ABS_TOL):
        """(number of elements out of tolerance, worst error / tolerance)."""
        y_bits = np.ascontiguousarray(y_bits, dtype=np.uint16).reshape(-1)
        yref = np.ascontiguousarray(yref, dtype=np.float64).reshape(-1)
        a = np.ascontiguousarray(a, dtype=np.float64).reshape(-1)
        assert y_bits.size == yref.size == a.size
        worst = ctypes.c_double(0.0)
        bad = self.lib.vgo_check(_ptr(y_bits), _ptr(yref), _ptr(a), y_bits.size, rel,
                                 abs_tol, ctypes.byref(worst))
        return int(bad), float(worst.value)


_default = None


def get() -> Oracle:
    """The default oracle (oracle/_build/liboracle.so)."""
    global _default
    if _default is None:
        _default = Oracle(load())
    return _default


def __getattr__(name):
    # module-level shortcuts: oracle.nvfp4_quantise(...) etc.
    if hasattr(Oracle, name) and not name.startswith("_"):
        return getattr(get(), name)
    raise AttributeError(name)
