"""MXFP8 and groupwise INT4 weights through the C ABI, against the oracle.

MXFP8 is the block-scaled FP8 that the crit README's Kernels section lists
for cuBLASLt; groupwise INT4 is the "groupwise-int" artifact format of the
NInfer README's model table (Marlin's GPTQ-style 4-bit groups, crit README
Kernels section).  Checked here:
* the packers: GPU quantise -> unpack equals the oracle's quantisation bit
  for bit, and canonical -> packed -> canonical is the identity;
* the decode, bit for bit: with x one-hot every product and sum is exact, so
  y must equal the oracle's dequantised weight (MXFP8: e4m3 * 2^(e-127),
  always a BF16 value in the supported scale range) or its single BF16
  rounding (INT4: (q - 8) * s has up to 12 significant bits), over every
  finite E4M3 code against every supported scale byte and every INT4 code;
* GEMVs within |y - y_ref| <= 4e-3 * sum|w x| + 1e-6, alone and mixed with
  NVFP4 and FP8 matrices in one verify pass.
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


def rand_x(seed, N, K, outliers=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((N, K), generator=g)
    if outliers:
        x[:, torch.randperm(K, generator=g)[:outliers]] *= 20
    return x.to(torch.bfloat16)


def one_hot_columns(vg, wt, K):
    out = np.zeros((wt.M, K), np.float64)
    x = torch.zeros((8, K), dtype=torch.bfloat16, device="cuda")
    ws = vg.workspace_for(wt)
    y = torch.empty((8, wt.M), dtype=torch.bfloat16, device="cuda")
    ar = torch.arange(8, device="cuda")
    for k0 in range(0, K, 8):
        x.zero_()
        x[ar, k0 + ar] = 1.0
        vg.gemv(wt, x, y=y, workspace=ws)
        out[:, k0:k0 + 8] = y.float().cpu().numpy().astype(np.float64).T
    assert vg.workspace_error(ws) == 0
    return out


# ------------------------------------------------------------------ packers

@pytest.mark.parametrize("M,K", [(64, 512), (17, 1024), (130, 2048), (300, 5120)])
def test_mxfp8_pack_is_bit_exact(vg, orc, M, K):
    W = rand_w(M + K, M, K)
    W[1, 32:64] = 0.0                                   # zero block: scale 127
    W[2, 64:96] *= 1e-36                                # below the scale range: clamped
    W[3, :32] *= 1e7                                    # above it: clamped, codes saturate
    wt = vg.mxfp8_pack(W.cuda())
    q, sc = vg.mxfp8_unpack(wt)
    q_ref, sc_ref = orc.mxfp8_quantise(W.numpy())
    assert np.array_equal(sc.cpu().numpy(), sc_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert sc_ref[1, 1] == 127 and sc_ref[2, 2] == 10 and sc_ref[3, 0] == 134


@pytest.mark.parametrize("M,K", [(64, 512), (17, 1024), (130, 2048), (300, 5120)])
def test_int4g_pack_is_bit_exact(vg, orc, M, K):
    W = rand_w(3 * M + K, M, K)
    W[1, 128:256] = 0.0                                 # zero group: scale 0, codes 8
    W[2, 5] = 3.0                                       # one large weight in a group
    wt = vg.int4g_pack(W.cuda())
    nib, sc = vg.int4g_unpack(wt)
    nib_ref, sc_ref = orc.int4g_quantise(W.numpy())
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), sc_ref)
    assert np.array_equal(nib.cpu().numpy(), nib_ref)


def test_from_canonical_round_trips_and_rejections(vg):
    rng = np.random.default_rng(4)
    M, K = 40, 1024
    q = rng.integers(0, 256, (M, K), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0
    sc = rng.integers(10, 135, (M, K // 32), dtype=np.uint8)
    wt = vg.mxfp8_from_canonical(torch.from_numpy(q).cuda(), torch.from_numpy(sc).cuda())
    q2, s2 = vg.mxfp8_unpack(wt)
    assert np.array_equal(q2.cpu().numpy(), q) and np.array_equal(s2.cpu().numpy(), sc)
    for b, status in ((9, 3), (135, 3), (255, 3)):
        bad = sc.copy()
        bad[3, 3] = b
        with pytest.raises(vg.VGError) as e:
            vg.mxfp8_from_canonical(torch.from_numpy(q).cuda(), torch.from_numpy(bad).cuda())
        assert e.value.status == status
    qb = q.copy()
    qb[0, 0] = 0x7F
    with pytest.raises(vg.VGError) as e:
        vg.mxfp8_from_canonical(torch.from_numpy(qb).cuda(), torch.from_numpy(sc).cuda())
    assert e.value.status == 1
    nib = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    s16 = torch.randn((M, K // 128)).to(torch.bfloat16)
    wt = vg.int4g_from_canonical(torch.from_numpy(nib).cuda(), s16.cuda())
    n2, t2 = vg.int4g_unpack(wt)
    assert np.array_equal(n2.cpu().numpy(), nib)
    assert torch.equal(t2.cpu(), s16.view(torch.int16))
    s16[1, 1] = float("inf")
    with pytest.raises(vg.VGError):
        vg.int4g_from_canonical(torch.from_numpy(nib).cuda(), s16.cuda())
    with pytest.raises(vg.VGError) as e:                # K not a multiple of 512
        vg.int4g_pack(torch.zeros((16, 768), device="cuda"))
    assert e.value.status == 3


# ------------------------------------------------------- decode, bit exact

@pytest.mark.parametrize("M,K", [(32, 1024), (16, 2048)])
def test_mxfp8_decode_is_bit_exact(vg, orc, M, K):
    """Every finite E4M3 code against every supported scale byte 10..134, in
    every byte position and both rows a lane holds."""
    m = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    q = ((k + 37 * m) % 256).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0
    blocks = np.arange(K // 32)[None, :]
    sc = (10 + (blocks + 7 * m) % 125).astype(np.uint8)
    assert set(np.unique(sc)) == set(range(10, 135))
    wt = vg.mxfp8_from_canonical(torch.from_numpy(q).cuda(), torch.from_numpy(sc).cuda())
    want = orc.mxfp8_dequant(q, sc, M, K)
    assert np.array_equal(torch.from_numpy(want).to(torch.bfloat16).double().numpy(), want)
    got = one_hot_columns(vg, wt, K)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} differ, first {bad[0].tolist()}"


@pytest.mark.parametrize("M,K", [(32, 1024), (48, 512)])
def test_int4g_decode_is_bit_exact(vg, orc, M, K):
    """Every INT4 code in every register slot, with BF16 group scales of
    every binade from 2^-20 to 2^20 and random significands: y is the single
    BF16 rounding of (q - 8) * s."""
    rng = np.random.default_rng(M + K)
    m = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    codes = ((k % 16) + m + k // 16) % 16
    nib = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    exps = rng.integers(-20, 21, (M, K // 128))
    mant = rng.integers(0, 128, (M, K // 128))
    sc = (((exps + 127) << 7) | mant).astype(np.uint16)
    sc[0, 0] = 0                                          # a zero scale
    sc[1, 0] |= 0x8000                                    # a negative scale
    wt = vg.int4g_from_canonical(torch.from_numpy(nib).cuda(),
                                 torch.from_numpy(sc.view(np.int16)).cuda())
    exact = orc.int4g_dequant(nib, sc, M, K)
    want = np.vectorize(lambda v: orc.bf16_value(orc.bf16_round(v)))(exact)
    got = one_hot_columns(vg, wt, K)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} differ, first {bad[0].tolist()}"


# --------------------------------------------------------------------- GEMV

SHAPES = [
    (1, 512, (1, 8)),            # a single row: 15 padding rows in its tile
    (16, 512, (4,)),             # exactly one tile
    (256, 512, (1,)),            # INT4: one chunk; MXFP8: two chunks
    (17, 1024, (1, 3, 8)),       # ragged rows
    (520, 2048, (8,)),           # several row blocks, split between blocks
    (100, 4096, (2, 8)),         # few rows: items of several chunks
    (5000, 2048, (8,)),          # many row blocks with a ragged last one
    (5120, 5120, (1, 8)),        # a full projection
]


@pytest.mark.parametrize("fmt", ["mxfp8", "int4g"])
@pytest.mark.parametrize("M,K,Ns", SHAPES)
def test_gemv_parity(vg, orc, fmt, M, K, Ns):
    W = rand_w(7 * M + K, M, K)
    if fmt == "mxfp8":
        wt = vg.mxfp8_pack(W.cuda())
        q, sc = orc.mxfp8_quantise(W.numpy())
    else:
        wt = vg.int4g_pack(W.cuda())
        q, sc = orc.int4g_quantise(W.numpy())
    ws = vg.workspace_for(wt)
    for N in Ns:
        x = rand_x(N + 5 * M, N, K, outliers=8)
        y = vg.gemv(wt, x.cuda(), workspace=ws)
        fn = orc.gemv_mxfp8 if fmt == "mxfp8" else orc.gemv_int4g
        yref, a = fn(q, sc, bits(x), threads=THREADS)
        bad, worst = orc.check(bits(y), yref, a)
        assert bad == 0, f"{fmt} {M}x{K} N={N}: {bad} out of tolerance (worst {worst:.3g})"
    assert vg.workspace_error(ws) == 0


@pytest.mark.parametrize("ordered", [True, False])
def test_verify_pass_with_every_format(vg, orc, ordered):
    """One pass over NVFP4, row-scaled FP8, MXFP8 and INT4 matrices, mixed in
    a group and across groups."""
    N = 5
    specs = [("nvfp4", 512, 1024, 0), ("mxfp8", 520, 1024, 0), ("int4g", 300, 2048, 0),
             ("fp8", 256, 512, 1), ("int4g", 1040, 512, 1), ("mxfp8", 100, 4096, 2)]
    entries, refs = [], []
    for i, (fmt, M, K, group) in enumerate(specs):
        W = rand_w(50 + i, M, K)
        x = rand_x(150 + i, N, K).cuda()
        y = torch.zeros((N, M), dtype=torch.bfloat16, device="cuda")
        if fmt == "nvfp4":
            wt = vg.nvfp4_pack(W.cuda())
            nib, sc, gs = orc.nvfp4_quantise(W.numpy())
            refs.append(orc.gemv_nvfp4(nib, sc, gs, bits(x), threads=THREADS))
        elif fmt == "fp8":
            wt = vg.fp8_pack(W.cuda())
            q, rs = orc.fp8_quantise(W.numpy())
            refs.append(orc.gemv_fp8(q, rs, bits(x), threads=THREADS))
        elif fmt == "mxfp8":
            wt = vg.mxfp8_pack(W.cuda())
            q, sc = orc.mxfp8_quantise(W.numpy())
            refs.append(orc.gemv_mxfp8(q, sc, bits(x), threads=THREADS))
        else:
            wt = vg.int4g_pack(W.cuda())
            nib, sc = orc.int4g_quantise(W.numpy())
            refs.append(orc.gemv_int4g(nib, sc, bits(x), threads=THREADS))
        entries.append((wt, x, y, group))
    plan = vg.VerifyPlan(entries, N, ordered=ordered)
    for _ in range(2):
        plan.run()
        assert plan.check() == 0
        for (fmt, M, K, _), (_, _, y, _), (yref, a) in zip(specs, entries, refs):
            bad, worst = orc.check(bits(y), yref, a)
            assert bad == 0, f"{fmt} {M}x{K}: {bad} out of tolerance (worst {worst:.3g})"
    plan.close()
