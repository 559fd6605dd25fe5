"""Bit-exact checks of the kernels' in-register dequantisation.

The GEMV decodes every weight to BF16 before it reaches the tensor cores
(engine card, Design table, "GEMVs" row: FP8 and NVFP4 bytes fed into BF16
MMA fragments; Checks section: operators checked against FP64 or plain
decoding).  A decoded NVFP4 weight e2m1 * e4m3 has at most 2 + 4 = 6
significant bits and a decoded FP8 weight 4, so with x one-hot (a single
BF16 1.0 per column) and a power-of-two tensor or row scale, every product
and the FP32 sum are exact and y[n, m] must equal the FP64 dequantised
weight W^[m, k_n] exactly: any wrong bit placement, scale re-encoding or
subnormal handling shows as a wrong value, not as an error inside the
tolerance.  The weights span every E2M1 code against every finite,
non-negative E4M3 scale byte 0x00..0x7E (subnormal scales 0x01..0x07
included), and every finite E4M3 code 0x00..0xFE except the two NaNs, in
every register position of the decode and in both rows (g, g + 8) a lane
holds, on the tensor-copied and the row-copied x paths.

Then GEMVs whose blocks sit at the bottom of the scale range (rows scaled
by 1e-5: subnormal E4M3 block scales) and FP8 rows whose codes are mostly
E4M3 subnormals or whose row scale is tiny, checked against the oracle with
the tolerance's relative part alone for those rows (the absolute 1e-6 would
hide any error at their magnitude).
"""
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def vg():
    from verify_gemm_gb300 import build

    build.build()
    import verify_gemm_gb300 as vg

    torch.cuda.init()
    return vg


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def one_hot_columns(vg, wt, K):
    """Decoded weights recovered column by column: x row n is the unit
    vector e_(k0 + n), eight columns per call.  Returns W^ as [M, K] FP64."""
    M = wt.M
    out = np.zeros((M, K), np.float64)
    x = torch.zeros((8, K), dtype=torch.bfloat16, device="cuda")
    ws = vg.workspace_for(wt)
    y = torch.empty((8, M), dtype=torch.bfloat16, device="cuda")
    ar = torch.arange(8, device="cuda")
    for k0 in range(0, K, 8):
        n = min(8, K - k0)
        x.zero_()
        x[ar[:n], k0 + ar[:n]] = 1.0
        vg.gemv(wt, x[:n], y=y[:n], workspace=ws)
        out[:, k0:k0 + n] = y[:n].float().cpu().numpy().astype(np.float64).T
    assert vg.workspace_error(ws) == 0
    return out


# (M, K): 32 x 2048 packs as 4-tile x 4-chunk items (tensor-copied x), 32 x
# 2112 as one-chunk items of 16 tiles with a 1-unit tail chunk (tensor-copied
# x), 48 x 2032 as one-chunk items with x copied row by row (K % 64 != 0)
NV_SHAPES = [(32, 2048), (32, 2112), (48, 2032)]


@pytest.mark.parametrize("M,K", NV_SHAPES)
def test_nvfp4_decode_is_bit_exact(vg, orc, M, K):
    m = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    # every code in every 16-block of every row, shifted from block to block
    # and row to row so each code meets every scale byte and register slot
    codes = ((k % 16) + m + k // 16) % 16
    nib = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    blocks = np.arange(K // 16)[None, :]
    sc = ((blocks + 5 * m) % 127).astype(np.uint8)         # every byte 0x00..0x7E
    assert set(np.unique(sc)) == set(range(127))
    gs = 2.0 ** -4
    wt = vg.nvfp4_from_canonical(torch.from_numpy(nib).cuda(), torch.from_numpy(sc).cuda(), gs)
    want = orc.nvfp4_dequant(nib, sc, gs, M, K)
    # each decoded weight is a BF16 value (<= 6 significant bits, in range)
    assert np.array_equal(torch.from_numpy(want).to(torch.bfloat16).double().numpy(), want)
    got = one_hot_columns(vg, wt, K)
    bad = np.argwhere(got != want)
    assert bad.size == 0, (f"{len(bad)} decoded weights differ, first at {bad[0].tolist()}: "
                           f"{got[tuple(bad[0])]} != {want[tuple(bad[0])]}")


# 32 x 1024 FP8 packs as 4-tile x 4-chunk items; 16 x 1040 as one-chunk
# items with a K tail and row-copied x
F8_SHAPES = [(32, 1024), (16, 1040)]


@pytest.mark.parametrize("M,K", F8_SHAPES)
def test_fp8_decode_is_bit_exact(vg, orc, M, K):
    m = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    q = ((k + 37 * m) % 256).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x00                             # no NaN codes
    finite = set(range(256)) - {0x7F, 0xFF}
    assert set(np.unique(q)) == finite                       # all 254 finite codes
    rs = (2.0 ** -(3 + (np.arange(M) % 5))).astype(np.float32)   # powers of two
    wt = vg.fp8_from_canonical(torch.from_numpy(q).cuda(), torch.from_numpy(rs).cuda())
    want = orc.fp8_dequant(q, rs, M, K)
    assert np.array_equal(torch.from_numpy(want).to(torch.bfloat16).double().numpy(), want)
    got = one_hot_columns(vg, wt, K)
    bad = np.argwhere(got != want)
    assert bad.size == 0, (f"{len(bad)} decoded weights differ, first at {bad[0].tolist()}: "
                           f"{got[tuple(bad[0])]} != {want[tuple(bad[0])]}")


def _check_rows_relative(y, yref, a, rows, what):
    """|y - y_ref| <= 4e-3 * sum|w x| on `rows`, without the absolute term."""
    yg = y.float().cpu().numpy().astype(np.float64)[:, rows]
    err = np.abs(yg - yref[:, rows])
    bound = 4e-3 * a[:, rows]
    assert np.all(a[:, rows] > 0), what
    worst = float((err / bound).max())
    assert worst <= 1.0, f"{what}: worst error / relative bound {worst:.3g}"


@pytest.mark.parametrize("M,K", [(512, 2048), (300, 5120)])
def test_gemv_nvfp4_subnormal_block_scales(vg, orc, M, K):
    """Rows far below the tensor's amax get E4M3 block scales in the
    subnormal range (codes 0x01..0x07) or zero; the GEMV stays within the
    relative tolerance on them."""
    g = torch.Generator().manual_seed(M + K)
    W = torch.randn((M, K), generator=g) * 0.02
    tiny = np.r_[16:32, 40, 41, 299]                  # a whole tile and scattered rows
    W[tiny] *= 1e-5
    W[50] *= 1e-7                                     # scales that round to zero
    W[60, : K // 2] *= 1e-5                           # half a row tiny
    wt = vg.nvfp4_pack(W.cuda())
    nib, sc, gs = orc.nvfp4_quantise(W.numpy())
    sub = sc[tiny]
    assert np.any((sub >= 1) & (sub <= 7)), "the tiny rows carry subnormal scale codes"
    assert not sc[50].any()
    ws = vg.workspace_for(wt)
    for N in (1, 8):
        x = torch.randn((N, K), generator=g).to(torch.bfloat16)
        y = vg.gemv(wt, x.cuda(), workspace=ws)
        yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(x), threads=THREADS)
        bad, worst = orc.check(bits(y), yref, a)
        assert bad == 0, f"N={N}: {bad} out of tolerance (worst {worst:.3g})"
        _check_rows_relative(y, yref, a, np.r_[tiny, 60], f"tiny rows N={N}")
        assert not y[:, 50].float().any()
    assert vg.workspace_error(ws) == 0


@pytest.mark.parametrize("M,K", [(256, 2048), (300, 4096)])
def test_gemv_fp8_subnormal_codes_and_tiny_row_scales(vg, orc, M, K):
    """FP8 rows whose codes are mostly E4M3 subnormals (one element 1e5 times
    the others sets the row scale) and rows with a tiny row scale (1e-30
    times the others); within the relative tolerance."""
    g = torch.Generator().manual_seed(3 * M + K)
    W = torch.randn((M, K), generator=g) * 0.02
    spiky = np.r_[0:16, 100, 255]
    W[spiky, 7] = 2000.0
    tiny = np.r_[16:32, 101]
    W[tiny] *= 1e-30
    wt = vg.fp8_pack(W.cuda())
    q, rs = orc.fp8_quantise(W.numpy())
    mag = q[spiky] & 0x7F
    assert np.mean((mag >= 1) & (mag <= 7)) > 0.5, "most codes of the spiky rows are subnormal"
    ws = vg.workspace_for(wt)
    for N in (1, 8):
        x = torch.randn((N, K), generator=g).to(torch.bfloat16)
        y = vg.gemv(wt, x.cuda(), workspace=ws)
        yref, a = orc.gemv_fp8(q, rs, bits(x), threads=THREADS)
        bad, worst = orc.check(bits(y), yref, a)
        assert bad == 0, f"N={N}: {bad} out of tolerance (worst {worst:.3g})"
        _check_rows_relative(y, yref, a, np.r_[spiky, tiny], f"N={N}")
    assert vg.workspace_error(ws) == 0
