"""Verify passes wider than 8 columns (N = 9..32): several requests' drafts
checked in one pass over the weights (NInfer README: one to eight execution
lanes, each verifying its MTP drafts; concurrent MTP3 decode at C = 1..8).

* every format within the GEMV tolerance of the oracle at widths 9..32;
* column invariance: the first 8 columns of a wide pass equal, bit for bit,
  the same columns of an 8-column pass (each block of 8 columns runs its own
  MMAs over the same K split);
* the limits: 16 columns for every layout, 32 for matrices in row blocks of
  16 tiles; wider requests are refused on the host;
* the wide kernel's decode, bit exact: with x one-hot, 16 or 32 columns per
  call, every code of each format against every scale it supports comes out
  as the oracle's dequantised weight, in row blocks of 16, 8 and 4 tiles;
* the full 64-layer stack at N = 16 in the benchmark's launch configuration
  (sampled rows), and the head at N = 32.
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


def rand_w(seed, M, K, std=0.02):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((M, K), generator=g) * std


def rand_x(seed, N, K):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((N, K), generator=g).to(torch.bfloat16)


def pack_and_ref(vg, orc, fmt, W):
    Wh = W.numpy()
    if fmt == "nvfp4":
        wt = vg.nvfp4_pack(W.cuda())
        nib, sc, gs = orc.nvfp4_quantise(Wh)
        return wt, lambda xb: orc.gemv_nvfp4(nib, sc, gs, xb, threads=THREADS)
    if fmt == "fp8":
        wt = vg.fp8_pack(W.cuda())
        q, rs = orc.fp8_quantise(Wh)
        return wt, lambda xb: orc.gemv_fp8(q, rs, xb, threads=THREADS)
    if fmt == "mxfp8":
        wt = vg.mxfp8_pack(W.cuda())
        q, sc = orc.mxfp8_quantise(Wh)
        return wt, lambda xb: orc.gemv_mxfp8(q, sc, xb, threads=THREADS)
    wt = vg.int4g_pack(W.cuda())
    nib, sc = orc.int4g_quantise(Wh)
    return wt, lambda xb: orc.gemv_int4g(nib, sc, xb, threads=THREADS)


# (M, K, widths, widest accepted): 4096 x 512 and 13056 x 1024 pack in row
# blocks of 16 tiles in every format (items of 8 or 4 units: up to 32
# columns); 5120 x 5120 in row blocks of 8 tiles (4-bit) or 4 tiles (8-bit),
# 16-unit items: up to 16 columns; 520 x 2048 in row blocks of 4 tiles (NVFP4,
# INT4) or 2 tiles (FP8, MXFP8), 32-unit items: 8 columns at most, so its
# wide requests are refused
WIDE = [(4096, 512, (9, 16, 24, 32), 32), (13056, 1024, (12, 32), 32),
        (5120, 5120, (16, 24), 16), (520, 2048, (10, 16), 8)]


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8", "mxfp8", "int4g"])
@pytest.mark.parametrize("M,K,Ns,widest", WIDE)
def test_wide_gemv_parity_and_column_invariance(vg, orc, fmt, M, K, Ns, widest):
    W = rand_w(M + 11 * K, M, K)
    wt, ref = pack_and_ref(vg, orc, fmt, W)
    x32 = rand_x(M + K, 32, K).cuda()
    y8 = vg.gemv(wt, x32[:8].clone())
    for N in Ns:
        if N > widest:
            with pytest.raises(vg.VGError) as e:      # refused on the host
                vg.gemv(wt, x32[:N].clone())
            assert e.value.status == 3, (fmt, M, K, N)
            continue
        y = vg.gemv(wt, x32[:N].clone())
        yref, a = ref(bits(x32[:N]))
        bad, worst = orc.check(bits(y), yref, a)
        assert bad == 0, f"{fmt} {M}x{K} N={N}: {bad} out of tolerance (worst {worst:.3g})"
        assert torch.equal(y[:8].view(torch.int16), y8.view(torch.int16)), (fmt, N)


def test_wide_limits(vg):
    wt = vg.nvfp4_pack(rand_w(1, 256, 640).cuda())        # K % 512 != 0
    with pytest.raises(vg.VGError) as e:
        vg.gemv(wt, rand_x(1, 12, 640).cuda())
    assert e.value.status == 3
    with pytest.raises(vg.VGError) as e:
        vg.gemv(wt, rand_x(1, 33, 640).cuda())
    assert e.value.status == 1


@pytest.mark.parametrize("N", [12, 16])
def test_wide_verify_pass_every_format(vg, orc, N):
    specs = [("nvfp4", 1040, 1024, 0), ("fp8", 520, 512, 0), ("mxfp8", 300, 1024, 1),
             ("int4g", 2048, 512, 1), ("nvfp4", 4096, 512, 2)]
    entries, refs = [], []
    for i, (fmt, M, K, group) in enumerate(specs):
        wt, ref = pack_and_ref(vg, orc, fmt, rand_w(70 + i, M, K))
        x = rand_x(170 + i, N, K).cuda()
        y = torch.zeros((N, M), dtype=torch.bfloat16, device="cuda")
        refs.append(ref(bits(x)))
        entries.append((wt, x, y, group))
    plan = vg.VerifyPlan(entries, N, ordered=True)
    for _ in range(2):
        plan.run()
        assert plan.check() == 0
        for (fmt, M, K, _), (_, _, y, _), (yref, a) in zip(specs, entries, refs):
            bad, worst = orc.check(bits(y), yref, a)
            assert bad == 0, f"{fmt} {M}x{K} N={N}: {bad} out of tolerance (worst {worst:.3g})"
    plan.close()


def test_full_stack_n16_and_head_n32(vg, orc):
    from verify_gemm_gb300.inputs import draw_stack_matrix, draw_workload
    from verify_gemm_gb300.workloads import build_stack

    N = 16
    st = build_stack(N)
    plan = st.plan(ordered=True)
    plan.run()
    assert plan.check() == 0
    plan.close()
    rng = np.random.default_rng(2)
    for i in (0, 4, 5, 6, len(st.mats) - 2, len(st.mats) - 1):
        m, wt, x, y = st.mats[i], st.weights[i], st.xs[i], st.ys[i]
        W, _ = draw_stack_matrix(m, N, 4, "cuda")
        Wh = W.cpu().numpy()
        del W
        rows = np.unique(np.concatenate([[0, m.M - 1], rng.integers(0, m.M, 200)]))
        if m.fmt == "nvfp4":
            gs = np.float32(orc.amax(Wh)) / np.float32(2688.0)
            assert gs == np.float32(wt.gscale)
            nib, sc = orc.nvfp4_quantise_gs(Wh[rows], gs)
            yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(x), threads=THREADS)
        else:
            q, rs = orc.fp8_quantise(Wh[rows])
            yref, a = orc.gemv_fp8(q, rs, bits(x), threads=THREADS)
        bad, worst = orc.check(bits(y[:, rows]), yref, a)
        assert bad == 0, f"{m.name} N=16: {bad} out of tolerance (worst {worst:.3g})"
    del st
    Ws, xs = draw_workload("down_head", 32, device="cuda")
    head = Ws[1]
    wt = vg.nvfp4_pack(head)
    Wh = head.cpu().numpy()
    del Ws, head
    x = xs[5120]
    y = vg.gemv(wt, x)
    rows = np.unique(np.concatenate([[0, 151935], rng.integers(0, 151936, 400)]))
    gs = np.float32(orc.amax(Wh)) / np.float32(2688.0)
    nib, sc = orc.nvfp4_quantise_gs(Wh[rows], gs)
    yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(x), threads=THREADS)
    bad, worst = orc.check(bits(y[:, rows]), yref, a)
    assert bad == 0, f"head N=32: {bad} out of tolerance (worst {worst:.3g})"


# ------------------------------------------- wide decode, bit exact (one-hot)

def one_hot_columns_wide(vg, wt, K, N):
    """Decoded weights recovered N > 8 columns per call (the wide kernel: one
    decode feeds N / 8 MMAs): x row n is the unit vector e_(k0 + n).  Returns
    W^ as [M, K] FP64."""
    M = wt.M
    out = np.zeros((M, K), np.float64)
    x = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    ws = vg.workspace_for(wt, N=N)
    y = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
    ar = torch.arange(N, device="cuda")
    for k0 in range(0, K, N):
        x.zero_()
        x[ar, k0 + ar] = 1.0
        vg.gemv(wt, x, y=y, workspace=ws)
        out[:, k0:k0 + N] = y.float().cpu().numpy().astype(np.float64).T
    assert vg.workspace_error(ws) == 0
    return out


def _codes4(M, K):
    m = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    codes = ((k % 16) + m + k // 16) % 16
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def _codes8(M, K):
    m = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    q = ((k + 37 * m) % 256).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0                               # no NaN codes
    return q


def _one_hot_case(vg, orc, fmt, M, K):
    """(packed weight, exact decoded weights) with every code of the format
    against every scale it supports, in every register slot and both rows a
    lane holds."""
    m = np.arange(M)[:, None]
    if fmt == "nvfp4":
        nib = _codes4(M, K)
        sc = ((np.arange(K // 16)[None, :] + 5 * m) % 127).astype(np.uint8)
        assert set(np.unique(sc)) == set(range(127))      # 0x00..0x7E, subnormals too
        gs = 2.0 ** -4
        wt = vg.nvfp4_from_canonical(torch.from_numpy(nib).cuda(), torch.from_numpy(sc).cuda(),
                                     gs)
        return wt, orc.nvfp4_dequant(nib, sc, gs, M, K)
    if fmt == "fp8":
        q = _codes8(M, K)
        assert len(np.unique(q)) == 254
        rs = (2.0 ** -(3 + (np.arange(M) % 5))).astype(np.float32)
        wt = vg.fp8_from_canonical(torch.from_numpy(q).cuda(), torch.from_numpy(rs).cuda())
        return wt, orc.fp8_dequant(q, rs, M, K)
    if fmt == "mxfp8":
        q = _codes8(M, K)
        sc = (10 + (np.arange(K // 32)[None, :] + 7 * m) % 125).astype(np.uint8)
        assert set(np.unique(sc)) == set(range(10, 135))
        wt = vg.mxfp8_from_canonical(torch.from_numpy(q).cuda(), torch.from_numpy(sc).cuda())
        return wt, orc.mxfp8_dequant(q, sc, M, K)
    rng = np.random.default_rng(M + K)
    nib = _codes4(M, K)
    exps = rng.integers(-20, 21, (M, K // 128))
    mant = rng.integers(0, 128, (M, K // 128))
    sc = (((exps + 127) << 7) | mant).astype(np.uint16)
    sc[0, 0] = 0                                           # a zero scale
    sc[1, 0] |= 0x8000                                     # a negative scale
    wt = vg.int4g_from_canonical(torch.from_numpy(nib).cuda(),
                                 torch.from_numpy(sc.view(np.int16)).cuda())
    exact = orc.int4g_dequant(nib, sc, M, K)
    # y is the single BF16 rounding of (q - 8) * s
    vals, inv = np.unique(exact, return_inverse=True)
    rounded = np.array([orc.bf16_value(orc.bf16_round(v)) for v in vals])
    return wt, rounded[inv].reshape(M, K)


# (fmt, M, K, N): row blocks of 16 tiles (one chunk per item) at 32 and 16
# columns; of 8 tiles (two chunks per item) and of 4 tiles (four chunks per
# item, 8-bit formats), where a warp's x columns start one or more chunks
# into the item's slice
WIDE_ONE_HOT = [("nvfp4", 256, 512, 32), ("nvfp4", 256, 512, 16), ("nvfp4", 256, 1024, 16),
                ("int4g", 256, 512, 32), ("int4g", 256, 1024, 16),
                ("fp8", 256, 256, 32), ("fp8", 256, 512, 32), ("fp8", 256, 1024, 16),
                ("mxfp8", 256, 512, 32), ("mxfp8", 256, 1024, 16)]


@pytest.mark.parametrize("fmt,M,K,N", WIDE_ONE_HOT)
def test_wide_decode_is_bit_exact(vg, orc, fmt, M, K, N):
    wt, want = _one_hot_case(vg, orc, fmt, M, K)
    if fmt != "int4g":
        # each decoded weight is a BF16 value: products and sums are exact
        assert np.array_equal(torch.from_numpy(want).to(torch.bfloat16).double().numpy(), want)
    got = one_hot_columns_wide(vg, wt, K, N)
    bad = np.argwhere(got != want)
    assert bad.size == 0, (f"{fmt} {M}x{K} N={N}: {len(bad)} decoded weights differ, first at "
                           f"{bad[0].tolist()}: {got[tuple(bad[0])]} != {want[tuple(bad[0])]}")
