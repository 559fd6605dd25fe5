"""Verify passes wider than 8 columns (N = 9..32): several requests' drafts
checked in one pass over the weights (NInfer README: one to eight execution
lanes, each verifying its MTP drafts; concurrent MTP3 decode at C = 1..8).

* every format within the GEMV tolerance of the oracle at widths 9..32;
* column invariance: the first 8 columns of a wide pass equal, bit for bit,
  the same columns of an 8-column pass (each block of 8 columns runs its own
  MMAs over the same K split);
* the limits: 16 columns for every layout, 32 for matrices in row blocks of
  16 tiles; wider requests are refused on the host;
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
