"""vg_gemv_nvfp4_noalloc: the NVFP4 GEMV for callers that cannot allocate
device memory (a host application that owns all device memory and lends out
only the input and output buffers, code that must not call cudaMalloc
because it can synchronise the device, code under a fixed memory budget).
It runs the same GEMV on a fixed scratch array inside the library, and
vg_gemv_nvfp4_noalloc_check reports, again without allocating, whether a
call's bounded device-side waits ran out.

This file is collected last on purpose.  It calls the entry point through
the C ABI several times in a row, changing the matrix shape (and so the
number of thread blocks) between calls, since the shared array keeps each
call's contents for the next; every result is checked against the
workspace entry point, vg_gemv_nvfp4, and against the CPU oracle, within
the tolerance the other tests use.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def test_noalloc_matches_workspace_entry_point(orc):
    from verify_gemm_gb300 import build

    build.build()
    import verify_gemm_gb300 as vg
    from verify_gemm_gb300 import _lib

    lib = _lib.load()
    g = torch.Generator().manual_seed(123)
    mats = {}
    for M, K in ((1040, 2560), (16, 4032)):   # 10 row blocks x 5 items; 1 x 8 (8 blocks)
        W = torch.randn((M, K), generator=g) * 0.02
        mats[(M, K)] = (vg.nvfp4_pack(W.cuda()), orc.nvfp4_quantise(W.numpy()))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two calls in a row, a call with another shape and grid, then the first
    # shape again
    calls = [((1040, 2560), 8), ((1040, 2560), 3), ((16, 4032), 5), ((1040, 2560), 8)]
    for call, ((M, K), N) in enumerate(calls):
        wt, (nib, sc, gs) = mats[(M, K)]
        x = (torch.randn((N, K), generator=g)).to(torch.bfloat16).cuda()
        y_ref = vg.gemv(wt, x)           # existing entry point, own workspace
        y = torch.full((N, M), 7.0, dtype=torch.bfloat16, device="cuda")
        s = lib.vg_gemv_nvfp4_noalloc(ctypes.c_void_p(wt.w.data_ptr()),
                                      ctypes.c_void_p(wt.scales.data_ptr()), wt.gscale,
                                      ctypes.c_void_p(x.data_ptr()), N, M, K,
                                      ctypes.c_void_p(y.data_ptr()), stream)
        assert s == 0, (call, lib.vg_status_string(s))
        err = ctypes.c_int(-1)
        assert lib.vg_gemv_nvfp4_noalloc_check(ctypes.byref(err), stream) == 0, call
        assert err.value == 0, call
        yr, a = orc.gemv_nvfp4(nib, sc, gs, _bits(x), threads=8)
        bad_new, _ = orc.check(_bits(y), yr, a)
        bad_old, _ = orc.check(_bits(y_ref), yr, a)
        assert bad_new == 0 and bad_old == 0, (call, bad_new, bad_old)
        # both use the same kernel and split, so they agree within tolerance
        # of each other too (in practice bit for bit)
        diff = (y.double() - y_ref.double()).abs().cpu().numpy()
        assert np.all(diff <= 4e-3 * a + 1e-6), call


def test_noalloc_scratch_covers_every_matrix_size():
    """The workspace is a header plus one partial-sum slot per thread block,
    whatever the matrix: every shape, up to the largest the library takes,
    fits the fixed array.  Only sizes are queried; nothing is launched."""
    from verify_gemm_gb300 import _lib

    lib = _lib.load()
    need = set()
    for M, K in ((16, 16), (1040, 2560), (151936, 5120), (1 << 29, 1024)):
        n = ctypes.c_size_t()
        assert lib.vg_gemv_workspace_size(M, K, 0, ctypes.byref(n)) == 0
        need.add(n.value)
    assert max(need) <= 4 << 20          # VG_NOALLOC_SCRATCH_BYTES
    big = ctypes.c_size_t()
    assert lib.vg_gemv_workspace_size(1 << 29, 1024, 0, ctypes.byref(big)) == 0
    assert big.value == max(need)
