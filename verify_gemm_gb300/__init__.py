"""GB300 (sm_103a) NVFP4 / row-scaled FP8 verify GEMV.

y[N, M] = x[N, K] . dequant(W)[M, K]^T for N = 1..8 BF16 columns (up to 32
for several requests' drafts in one pass), the weight-streaming product of
decode and speculative verification (the "GEMVs" row of the
mtp7-device-confidence engine card's Design table); MXFP8 and groupwise
INT4 weights as well, and a fused verify pass over a layer stack with RMS
norms and the gated activation.

Every step runs in the CUDA kernels of ``libvgemm.so`` (C ABI declared in
``include/vgemm.h``); this module only marshals torch tensors (device
memory and streams) into that ABI.  There is no CPU or PyTorch fallback:
if the library is missing, calls raise.
"""
from __future__ import annotations

from dataclasses import dataclass

import ctypes

import torch

from . import _lib
from ._lib import (VG_FMT_FP8_ROWSCALE, VG_FMT_INT4G, VG_FMT_MXFP8, VG_FMT_NVFP4,  # noqa: F401
                   VG_OP_GEMV, VG_OP_RMSNORM, VG_OP_SWIGLU, VGError)

__all__ = [
    "NVFP4Weight", "FP8Weight", "nvfp4_pack", "fp8_pack", "nvfp4_unpack", "fp8_unpack",
    "nvfp4_from_canonical", "fp8_from_canonical", "gemv", "workspace_for", "VerifyPlan",
    "VGError", "VG_FMT_NVFP4", "VG_FMT_FP8_ROWSCALE", "NVFP4GatedWeight", "FP8GatedWeight",
    "nvfp4_pack_gated", "fp8_pack_gated", "RMSNorm", "BlockScaledWeight", "mxfp8_pack",
    "int4g_pack", "mxfp8_unpack", "int4g_unpack", "mxfp8_from_canonical",
    "int4g_from_canonical", "VG_FMT_MXFP8", "VG_FMT_INT4G",
]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev_tensor(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor")
    return t


@dataclass
class NVFP4Weight:
    """Packed NVFP4 weight (codes + block scales in the device layout)."""

    w: torch.Tensor          # uint8, opaque packed codes
    scales: torch.Tensor     # uint8, opaque packed block scales
    gscale: float            # FP32 tensor scale (dequantisation multiplier)
    M: int
    K: int
    fmt: int = VG_FMT_NVFP4

    @property
    def nbytes(self) -> int:
        """Algorithmic weight+scale bytes: M*K/2 codes + M*K/16 scales + 4."""
        return self.M * self.K // 2 + self.M * self.K // 16 + 4


@dataclass
class FP8Weight:
    """Packed row-scaled FP8-E4M3 weight."""

    w: torch.Tensor          # uint8, opaque packed codes
    rowscale: torch.Tensor   # float32 [M]
    M: int
    K: int
    fmt: int = VG_FMT_FP8_ROWSCALE

    @property
    def nbytes(self) -> int:
        """Algorithmic weight+scale bytes: M*K codes + 4*M row scales."""
        return self.M * self.K + 4 * self.M


@dataclass
class NVFP4GatedWeight:
    """A gate/up pair packed for the fused gated activation: M = 2*I rows,
    each 16-row tile holding 8 gate rows and the same 8 up rows."""

    w: torch.Tensor
    scales: torch.Tensor
    gscale: float            # tensor scale of the gate half
    gscale_up: float         # tensor scale of the up half
    I: int
    K: int
    fmt: int = VG_FMT_NVFP4
    op: int = VG_OP_SWIGLU

    @property
    def M(self) -> int:
        return 2 * self.I

    @property
    def nbytes(self) -> int:
        """Both halves' codes and block scales, and their two tensor scales."""
        return self.M * self.K // 2 + self.M * self.K // 16 + 8


@dataclass
class FP8GatedWeight:
    """A gate/up pair of row-scaled FP8 weights packed like NVFP4GatedWeight."""

    w: torch.Tensor
    rowscale: torch.Tensor     # float32 [I], gate rows
    rowscale_up: torch.Tensor  # float32 [I], up rows
    I: int
    K: int
    fmt: int = VG_FMT_FP8_ROWSCALE
    op: int = VG_OP_SWIGLU

    @property
    def M(self) -> int:
        return 2 * self.I

    @property
    def nbytes(self) -> int:
        return self.M * self.K + 4 * self.M


@dataclass
class RMSNorm:
    """An RMS normalisation entry of a verify pass: y = x * gamma / rms(x)."""

    gamma: torch.Tensor      # bfloat16 [K]
    eps: float = 1e-6
    op: int = VG_OP_RMSNORM
    nbytes: int = 0          # no weights


@dataclass
class BlockScaledWeight:
    """Packed MXFP8 (fmt VG_FMT_MXFP8) or groupwise INT4 (VG_FMT_INT4G) weight."""

    w: torch.Tensor          # uint8, opaque packed codes
    scales: torch.Tensor     # uint8, opaque packed block scales
    M: int
    K: int
    fmt: int

    @property
    def nbytes(self) -> int:
        """Algorithmic bytes: MXFP8 M*K codes + M*K/32 scales; INT4 M*K/2 codes +
        2*M*K/128 scales."""
        E = self.M * self.K
        return E + E // 32 if self.fmt == VG_FMT_MXFP8 else E // 2 + 2 * (E // 128)


def weight_sizes(fmt: int, M: int, K: int):
    wb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _lib.check(_lib.vg_weight_sizes(fmt, M, K, ctypes.byref(wb), ctypes.byref(sb)),
               "vg_weight_sizes")
    return wb.value, sb.value


def _block_pack(fmt, fn, W, stream):
    _dev_tensor(W, torch.float32, "W")
    M, K = W.shape
    wb, sb = weight_sizes(fmt, M, K)
    w = torch.empty(wb, dtype=torch.uint8, device=W.device)
    sc = torch.empty(sb, dtype=torch.uint8, device=W.device)
    _lib.check(fn(_ptr(W), M, K, _ptr(w), _ptr(sc), _stream(stream)), fn.__name__)
    return BlockScaledWeight(w, sc, M, K, fmt)


def mxfp8_pack(W: torch.Tensor, stream=None) -> BlockScaledWeight:
    """MXFP8 quantisation (E4M3 codes, E8M0 scale per 32 along K; K % 256 == 0)."""
    return _block_pack(VG_FMT_MXFP8, _lib.vg_mxfp8_pack, W, stream)


def int4g_pack(W: torch.Tensor, stream=None) -> BlockScaledWeight:
    """Groupwise INT4 quantisation (BF16 scale per 128 along K; K % 512 == 0)."""
    return _block_pack(VG_FMT_INT4G, _lib.vg_int4g_pack, W, stream)


def mxfp8_unpack(wt: BlockScaledWeight, stream=None):
    """Packed -> canonical (q uint8 [M, K], sc uint8 [M, K/32]) on the device."""
    q = torch.empty((wt.M, wt.K), dtype=torch.uint8, device=wt.w.device)
    sc = torch.empty((wt.M, wt.K // 32), dtype=torch.uint8, device=wt.w.device)
    _lib.check(_lib.vg_mxfp8_unpack(_ptr(wt.w), _ptr(wt.scales), wt.M, wt.K, _ptr(q), _ptr(sc),
                                    _stream(stream)), "vg_mxfp8_unpack")
    return q, sc


def int4g_unpack(wt: BlockScaledWeight, stream=None):
    """Packed -> canonical (nib uint8 [M, K/2], sc BF16 bits as int16 [M, K/128])."""
    nib = torch.empty((wt.M, wt.K // 2), dtype=torch.uint8, device=wt.w.device)
    sc = torch.empty((wt.M, wt.K // 128), dtype=torch.int16, device=wt.w.device)
    _lib.check(_lib.vg_int4g_unpack(_ptr(wt.w), _ptr(wt.scales), wt.M, wt.K, _ptr(nib), _ptr(sc),
                                    _stream(stream)), "vg_int4g_unpack")
    return nib, sc


def mxfp8_from_canonical(q: torch.Tensor, sc: torch.Tensor, stream=None) -> BlockScaledWeight:
    _dev_tensor(q, torch.uint8, "q")
    _dev_tensor(sc, torch.uint8, "sc")
    M, K = q.shape
    wb, sb = weight_sizes(VG_FMT_MXFP8, M, K)
    w = torch.empty(wb, dtype=torch.uint8, device=q.device)
    s = torch.empty(sb, dtype=torch.uint8, device=q.device)
    _lib.check(_lib.vg_mxfp8_from_canonical(_ptr(q), _ptr(sc), M, K, _ptr(w), _ptr(s),
                                            _stream(stream)), "vg_mxfp8_from_canonical")
    return BlockScaledWeight(w, s, M, K, VG_FMT_MXFP8)


def int4g_from_canonical(nib: torch.Tensor, sc: torch.Tensor, stream=None) -> BlockScaledWeight:
    """sc: BF16 scale bits [M, K/128] as an int16 (or bfloat16) tensor."""
    _dev_tensor(nib, torch.uint8, "nib")
    if sc.dtype == torch.bfloat16:
        sc = sc.view(torch.int16)
    _dev_tensor(sc, torch.int16, "sc")
    M, K = nib.shape[0], nib.shape[1] * 2
    wb, sb = weight_sizes(VG_FMT_INT4G, M, K)
    w = torch.empty(wb, dtype=torch.uint8, device=nib.device)
    s = torch.empty(sb, dtype=torch.uint8, device=nib.device)
    _lib.check(_lib.vg_int4g_from_canonical(_ptr(nib), _ptr(sc), M, K, _ptr(w), _ptr(s),
                                            _stream(stream)), "vg_int4g_from_canonical")
    return BlockScaledWeight(w, s, M, K, VG_FMT_INT4G)


def nvfp4_sizes(M: int, K: int):
    wb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _lib.check(_lib.vg_nvfp4_sizes(M, K, ctypes.byref(wb), ctypes.byref(sb)), "vg_nvfp4_sizes")
    return wb.value, sb.value


def fp8_sizes(M: int, K: int) -> int:
    wb = ctypes.c_size_t()
    _lib.check(_lib.vg_fp8_sizes(M, K, ctypes.byref(wb)), "vg_fp8_sizes")
    return wb.value


def nvfp4_pack(W: torch.Tensor, stream=None) -> NVFP4Weight:
    """Round-to-nearest NVFP4 quantisation of a CUDA FP32 [M, K] matrix."""
    _dev_tensor(W, torch.float32, "W")
    M, K = W.shape
    wb, sb = nvfp4_sizes(M, K)
    w = torch.empty(wb, dtype=torch.uint8, device=W.device)
    sc = torch.empty(sb, dtype=torch.uint8, device=W.device)
    gs = ctypes.c_float()
    _lib.check(_lib.vg_nvfp4_pack(_ptr(W), M, K, _ptr(w), _ptr(sc), ctypes.byref(gs),
                                  _stream(stream)), "vg_nvfp4_pack")
    return NVFP4Weight(w, sc, gs.value, M, K)


def fp8_pack(W: torch.Tensor, stream=None) -> FP8Weight:
    """Row-scaled FP8-E4M3 quantisation of a CUDA FP32 [M, K] matrix."""
    _dev_tensor(W, torch.float32, "W")
    M, K = W.shape
    w = torch.empty(fp8_sizes(M, K), dtype=torch.uint8, device=W.device)
    rs = torch.empty(M, dtype=torch.float32, device=W.device)
    _lib.check(_lib.vg_fp8_pack(_ptr(W), M, K, _ptr(w), _ptr(rs), _stream(stream)), "vg_fp8_pack")
    return FP8Weight(w, rs, M, K)


def nvfp4_pack_gated(Wgate: torch.Tensor, Wup: torch.Tensor, stream=None) -> NVFP4GatedWeight:
    """NVFP4 gate/up pair for the fused gated activation (each half with its
    own tensor scale, quantised exactly as nvfp4_pack would)."""
    _dev_tensor(Wgate, torch.float32, "Wgate")
    _dev_tensor(Wup, torch.float32, "Wup")
    if Wgate.shape != Wup.shape:
        raise ValueError("gate and up must have the same shape")
    I, K = Wgate.shape
    wb, sb = nvfp4_sizes(2 * I, K)
    w = torch.empty(wb, dtype=torch.uint8, device=Wgate.device)
    sc = torch.empty(sb, dtype=torch.uint8, device=Wgate.device)
    gs = (ctypes.c_float * 2)()
    _lib.check(_lib.vg_nvfp4_pack_gated(_ptr(Wgate), _ptr(Wup), I, K, _ptr(w), _ptr(sc), gs,
                                        _stream(stream)), "vg_nvfp4_pack_gated")
    return NVFP4GatedWeight(w, sc, gs[0], gs[1], I, K)


def fp8_pack_gated(Wgate: torch.Tensor, Wup: torch.Tensor, stream=None) -> FP8GatedWeight:
    """Row-scaled FP8 gate/up pair for the fused gated activation."""
    _dev_tensor(Wgate, torch.float32, "Wgate")
    _dev_tensor(Wup, torch.float32, "Wup")
    if Wgate.shape != Wup.shape:
        raise ValueError("gate and up must have the same shape")
    I, K = Wgate.shape
    w = torch.empty(fp8_sizes(2 * I, K), dtype=torch.uint8, device=Wgate.device)
    rg = torch.empty(I, dtype=torch.float32, device=Wgate.device)
    ru = torch.empty(I, dtype=torch.float32, device=Wgate.device)
    _lib.check(_lib.vg_fp8_pack_gated(_ptr(Wgate), _ptr(Wup), I, K, _ptr(w), _ptr(rg), _ptr(ru),
                                      _stream(stream)), "vg_fp8_pack_gated")
    return FP8GatedWeight(w, rg, ru, I, K)


def nvfp4_unpack(wt: NVFP4Weight, stream=None):
    """Packed -> canonical (nib uint8 [M, K/2], sc uint8 [M, K/16]) on the device."""
    nib = torch.empty((wt.M, wt.K // 2), dtype=torch.uint8, device=wt.w.device)
    sc = torch.empty((wt.M, wt.K // 16), dtype=torch.uint8, device=wt.w.device)
    _lib.check(_lib.vg_nvfp4_unpack(_ptr(wt.w), _ptr(wt.scales), wt.M, wt.K, _ptr(nib), _ptr(sc),
                                    _stream(stream)), "vg_nvfp4_unpack")
    return nib, sc


def fp8_unpack(wt: FP8Weight, stream=None):
    q = torch.empty((wt.M, wt.K), dtype=torch.uint8, device=wt.w.device)
    _lib.check(_lib.vg_fp8_unpack(_ptr(wt.w), wt.M, wt.K, _ptr(q), _stream(stream)),
               "vg_fp8_unpack")
    return q


def nvfp4_from_canonical(nib: torch.Tensor, sc: torch.Tensor, gscale: float,
                         stream=None) -> NVFP4Weight:
    _dev_tensor(nib, torch.uint8, "nib")
    _dev_tensor(sc, torch.uint8, "sc")
    M, K = nib.shape[0], nib.shape[1] * 2
    wb, sb = nvfp4_sizes(M, K)
    w = torch.empty(wb, dtype=torch.uint8, device=nib.device)
    s = torch.empty(sb, dtype=torch.uint8, device=nib.device)
    _lib.check(_lib.vg_nvfp4_from_canonical(_ptr(nib), _ptr(sc), M, K, _ptr(w), _ptr(s),
                                            _stream(stream)), "vg_nvfp4_from_canonical")
    return NVFP4Weight(w, s, float(gscale), M, K)


def fp8_from_canonical(q: torch.Tensor, rowscale: torch.Tensor, stream=None) -> FP8Weight:
    _dev_tensor(q, torch.uint8, "q")
    _dev_tensor(rowscale, torch.float32, "rowscale")
    M, K = q.shape
    w = torch.empty(fp8_sizes(M, K), dtype=torch.uint8, device=q.device)
    _lib.check(_lib.vg_fp8_from_canonical(_ptr(q), M, K, _ptr(w), _stream(stream)),
               "vg_fp8_from_canonical")
    return FP8Weight(w, rowscale, M, K)


def workspace_for(wt, device=None, N: int = 8) -> torch.Tensor:
    """A zero-filled workspace large enough for GEMVs of up to N columns
    (N <= 8 by default) with this weight."""
    n = ctypes.c_size_t()
    _lib.check(_lib.vg_gemv_workspace_size_n(wt.M, wt.K, wt.fmt, max(N, 1), ctypes.byref(n)),
               "vg_gemv_workspace_size_n")
    return torch.zeros(n.value, dtype=torch.uint8, device=device or wt.w.device)


def gemv(wt, x: torch.Tensor, y: torch.Tensor | None = None, workspace=None, stream=None):
    """y[N, M] = x[N, K] . dequant(W)^T (BF16 in, BF16 out, FP32 accumulate)."""
    _dev_tensor(x, torch.bfloat16, "x")
    N, K = x.shape
    if K != wt.K:
        raise ValueError("x has the wrong K")
    if y is None:
        y = torch.empty((N, wt.M), dtype=torch.bfloat16, device=x.device)
    _dev_tensor(y, torch.bfloat16, "y")
    if workspace is None:
        workspace = workspace_for(wt, x.device, N)
    if wt.fmt == VG_FMT_NVFP4:
        s = _lib.vg_gemv_nvfp4(_ptr(wt.w), _ptr(wt.scales), wt.gscale, _ptr(x), N, wt.M, wt.K,
                               _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream))
        _lib.check(s, "vg_gemv_nvfp4")
    elif wt.fmt in (VG_FMT_MXFP8, VG_FMT_INT4G):
        fn = _lib.vg_gemv_mxfp8 if wt.fmt == VG_FMT_MXFP8 else _lib.vg_gemv_int4g
        s = fn(_ptr(wt.w), _ptr(wt.scales), _ptr(x), N, wt.M, wt.K, _ptr(y), _ptr(workspace),
               workspace.numel(), _stream(stream))
        _lib.check(s, fn.__name__)
    else:
        s = _lib.vg_gemv_fp8_rowscale(_ptr(wt.w), _ptr(wt.rowscale), _ptr(x), N, wt.M, wt.K,
                                      _ptr(y), _ptr(workspace), workspace.numel(),
                                      _stream(stream))
        _lib.check(s, "vg_gemv_fp8_rowscale")
    return y


def workspace_error(workspace: torch.Tensor, stream=None) -> int:
    """Device error word of a GEMV workspace (0 = none); clears it."""
    err = ctypes.c_int()
    s = _lib.vg_gemv_workspace_check(_ptr(workspace), workspace.numel(), ctypes.byref(err),
                                     _stream(stream))
    if s not in (_lib.VG_OK, _lib.VG_ERR_TIMEOUT):
        _lib.check(s, "vg_gemv_workspace_check")
    return err.value


class VerifyPlan:
    """A fused verify pass over a list of entries (op, x, y, group) or
    (op, x, y, group, x_after_group): op is a packed weight (a GEMV, or a
    gated pair's fused activation) or an RMSNorm; x_after_group marks an x
    that the previous group of the same pass writes."""

    def __init__(self, entries, N: int, ordered: bool = True, max_ctas: int = 0,
                 wait_timeout_ns: int = 0, hold_group: int = -1):
        self.entries = list(entries)    # keep tensors alive
        arr = (_lib.vg_matrix_desc * len(self.entries))()
        for i, e in enumerate(self.entries):
            wt, x, y, group = e[:4]
            after = bool(e[4]) if len(e) > 4 else False
            _dev_tensor(x, torch.bfloat16, "x")
            _dev_tensor(y, torch.bfloat16, "y")
            d = arr[i]
            d.group = group
            d.x_after_group = int(after)
            d.x = x.data_ptr()
            d.y = y.data_ptr()
            op = getattr(wt, "op", VG_OP_GEMV)
            d.op = op
            if op == VG_OP_RMSNORM:
                _dev_tensor(wt.gamma, torch.bfloat16, "gamma")
                d.M, d.K = 1, x.shape[1]
                d.gamma = wt.gamma.data_ptr()
                d.eps = wt.eps
                continue
            d.format = wt.fmt
            d.M, d.K = wt.M, wt.K
            d.w = wt.w.data_ptr()
            if wt.fmt == VG_FMT_NVFP4:
                d.scales = wt.scales.data_ptr()
                d.gscale = wt.gscale
                if op == VG_OP_SWIGLU:
                    d.gscale_up = wt.gscale_up
            elif wt.fmt in (VG_FMT_MXFP8, VG_FMT_INT4G):
                d.scales = wt.scales.data_ptr()
            else:
                d.rowscale = wt.rowscale.data_ptr()
                if op == VG_OP_SWIGLU:
                    d.rowscale_up = wt.rowscale_up.data_ptr()
        opt = _lib.vg_plan_options(int(bool(ordered)), int(max_ctas), int(wait_timeout_ns),
                                   int(hold_group), 0)
        h = ctypes.c_void_p()
        _lib.check(_lib.vg_verify_plan_create_ex(arr, len(self.entries), N, ctypes.byref(opt),
                                                 ctypes.byref(h)), "vg_verify_plan_create_ex")
        self._h = h
        self.N = N

    def run(self, stream=None):
        _lib.check(_lib.vg_verify_pass(self._h, _stream(stream)), "vg_verify_pass")

    def set_width(self, width: torch.Tensor | None):
        """Read each pass's width from a device int32 tensor (one element)
        instead of the fixed N; None returns to the fixed N."""
        if width is not None:
            if not (width.is_cuda and width.dtype == torch.int32 and width.numel() == 1):
                raise ValueError("width: expected a one-element CUDA int32 tensor")
            self._width = width                      # keep it alive
        else:
            self._width = None
        _lib.check(_lib.vg_verify_plan_set_width(self._h, _ptr(width) if width is not None
                                                 else None), "vg_verify_plan_set_width")

    def check(self, stream=None) -> int:
        err = ctypes.c_int()
        s = _lib.vg_verify_plan_check(self._h, _stream(stream), ctypes.byref(err))
        if s not in (_lib.VG_OK, _lib.VG_ERR_TIMEOUT):
            _lib.check(s, "vg_verify_plan_check")
        return err.value

    @property
    def bytes(self) -> int:
        b = ctypes.c_int64()
        _lib.check(_lib.vg_verify_plan_bytes(self._h, ctypes.byref(b)), "vg_verify_plan_bytes")
        return b.value

    @property
    def grid(self) -> int:
        g = ctypes.c_int()
        _lib.check(_lib.vg_verify_plan_grid(self._h, ctypes.byref(g)), "vg_verify_plan_grid")
        return g.value

    def close(self):
        if getattr(self, "_h", None):
            _lib.vg_verify_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
