"""The C-ABI library on the host: it builds, loads, exports every entry point
that include/vgemm.h declares, answers size queries, and rejects bad
arguments before touching a GPU.  No compute call runs here."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "vgemm.h")


@pytest.fixture(scope="module")
def lib():
    from verify_gemm_gb300 import _lib, build

    build.build()
    return _lib.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(vg_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_abi():
    """Every call of the boundary's listing is declared under its own name."""
    names = _declared_functions()
    for want in ("vg_status_string", "vg_nvfp4_sizes", "vg_nvfp4_pack", "vg_nvfp4_unpack",
                 "vg_gemv_nvfp4", "vg_fp8_rowscale_pack", "vg_fp8_rowscale_unpack",
                 "vg_gemv_fp8_rowscale", "vg_verify_plan_create", "vg_verify_pass",
                 "vg_verify_plan_destroy", "vg_gemv_nvfp4_noalloc_check"):
        assert want in names, want


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    from verify_gemm_gb300 import _lib

    assert sorted(_lib.SIGNATURES) == _declared_functions()


def test_status_strings(lib):
    for s in range(7):
        assert lib.vg_status_string(s)
    assert lib.vg_status_string(99) == b"unknown status"
    assert lib.vg_version() >= 100


def test_size_queries(lib):
    wb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.vg_nvfp4_sizes(5120, 5120, ctypes.byref(wb), ctypes.byref(sb)) == 0
    # exact algorithmic bytes when M % 16 == 0 and K % 256 == 0
    assert wb.value == 5120 * 5120 // 2 and sb.value == 5120 * 5120 // 16
    assert lib.vg_nvfp4_sizes(151936, 5120, ctypes.byref(wb), ctypes.byref(sb)) == 0
    assert wb.value + sb.value == 437_575_680
    assert lib.vg_fp8_sizes(5120, 17408, ctypes.byref(wb)) == 0
    assert wb.value + 4 * 5120 == 89_149_440
    # ragged shapes round up to 16-row tiles and 64-column units
    assert lib.vg_nvfp4_sizes(17, 80, ctypes.byref(wb), ctypes.byref(sb)) == 0
    assert wb.value == 2 * 2 * 512 and sb.value == 2 * 1 * 512
    assert lib.vg_fp8_sizes(1, 16, ctypes.byref(wb)) == 0 and wb.value == 1024


@pytest.mark.parametrize("M,K", [(0, 64), (16, 8), (16, 24), (-1, 64), (1 << 30, 1 << 20)])
def test_bad_shapes_are_rejected(lib, M, K):
    wb = ctypes.c_size_t()
    assert lib.vg_nvfp4_sizes(M, K, ctypes.byref(wb), None) in (1, 3)
    assert lib.vg_fp8_sizes(M, K, ctypes.byref(wb)) in (1, 3)


def test_gemv_argument_validation_happens_on_the_host(lib):
    p16 = ctypes.c_void_p(0x10000)
    p8 = ctypes.c_void_p(0x10008)
    # N out of range, null pointers, K % 16, misalignment: no CUDA call is made
    assert lib.vg_gemv_nvfp4(p16, p16, 1.0, p16, 0, 64, 64, p16, p16, 1 << 20, None) == 1
    assert lib.vg_gemv_nvfp4(p16, p16, 1.0, p16, 33, 64, 64, p16, p16, 1 << 20, None) == 1
    assert lib.vg_gemv_nvfp4(None, p16, 1.0, p16, 1, 64, 64, p16, p16, 1 << 20, None) == 1
    assert lib.vg_gemv_nvfp4(p16, None, 1.0, p16, 1, 64, 64, p16, p16, 1 << 20, None) == 1
    assert lib.vg_gemv_nvfp4(p16, p16, 1.0, p16, 1, 64, 40, p16, p16, 1 << 20, None) == 1
    assert lib.vg_gemv_nvfp4(p8, p16, 1.0, p16, 1, 64, 64, p16, p16, 1 << 20, None) == 2
    assert lib.vg_gemv_nvfp4(p16, p16, 1.0, p8, 1, 64, 64, p16, p16, 1 << 20, None) == 2
    assert lib.vg_gemv_fp8_rowscale(p16, None, p16, 1, 64, 64, p16, p16, 1 << 20, None) == 1
    assert lib.vg_nvfp4_pack(None, 64, 64, p16, p16, None, None) == 1
    assert lib.vg_nvfp4_unpack(p8, p16, 64, 64, p16, p16, None) == 2
    assert lib.vg_verify_plan_create(None, 1, 1, 1, None) == 1


def test_oracle_and_product_share_nothing():
    """The CUDA path and the oracle are independent: neither imports or
    includes anything from the other."""
    pkg = os.path.join(ROOT, "verify_gemm_gb300")
    imp_oracle = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[<\"].*oracle)", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not imp_oracle.search(text), os.path.join(dirpath, f)
    imp_pkg = re.compile(r"^\s*(import\s+verify_gemm_gb300|from\s+verify_gemm_gb300|"
                         r"#\s*include\s*[<\"].*(csrc|vg_device|vgemm))", re.M)
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c", ".h")):
            assert not imp_pkg.search(open(os.path.join(ROOT, "oracle", f)).read()), f


def test_format_sizes_and_host_checks(lib):
    """Sizes of the block-scaled formats, and the argument checks of the newer
    entry points, answered on the host without a GPU."""
    wb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    # MXFP8: E4M3 codes (FP8 units) + 1 E8M0 byte per 32 elements
    assert lib.vg_weight_sizes(2, 5120, 5120, ctypes.byref(wb), ctypes.byref(sb)) == 0
    assert wb.value == 5120 * 5120 and sb.value == 5120 * 5120 // 32
    # groupwise INT4: 4-bit codes + a BF16 scale per 128 elements
    assert lib.vg_weight_sizes(3, 5120, 5120, ctypes.byref(wb), ctypes.byref(sb)) == 0
    assert wb.value == 5120 * 5120 // 2 and sb.value == 2 * 5120 * 5120 // 128
    # NVFP4 and FP8 agree with their own size calls
    assert lib.vg_weight_sizes(0, 17, 80, ctypes.byref(wb), ctypes.byref(sb)) == 0
    assert (wb.value, sb.value) == (2 * 2 * 512, 2 * 1 * 512)
    assert lib.vg_weight_sizes(9, 64, 64, ctypes.byref(wb), ctypes.byref(sb)) == 1
    p16 = ctypes.c_void_p(0x10000)
    # K not a multiple of a chunk: the block-scaled packers refuse before any CUDA call
    assert lib.vg_int4g_pack(p16, 64, 768, p16, p16, None) == 3
    assert lib.vg_mxfp8_pack(p16, 64, 320, p16, p16, None) == 3
    assert lib.vg_gemv_int4g(p16, p16, p16, 8, 64, 768, p16, p16, 1 << 20, None) == 3
    # widths: 1..32
    n = ctypes.c_size_t()
    assert lib.vg_gemv_workspace_size_n(64, 512, 0, 33, ctypes.byref(n)) == 1
    assert lib.vg_gemv_workspace_size_n(64, 512, 0, 0, ctypes.byref(n)) == 1
    assert lib.vg_gemv_nvfp4(p16, p16, 1.0, p16, 33, 64, 64, p16, p16, 1 << 20, None) == 1
    # gated pairs need I % 8 == 0
    gs = (ctypes.c_float * 2)()
    assert lib.vg_nvfp4_pack_gated(p16, p16, 12, 64, p16, p16, gs, None) == 1
    # the width word must be 4-byte aligned (checked before the plan is touched)
    assert lib.vg_verify_plan_set_width(None, None) == 1
