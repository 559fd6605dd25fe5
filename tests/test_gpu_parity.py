"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

* Packers: GPU pack -> unpack equals the oracle's quantisation bit for bit.
* GEMV: every element within |y - y_ref| <= 4e-3 * sum|w x| + 1e-6, at
  sizes that span several tiles, chunks and row blocks plus ragged tails,
  and at the full workload sizes (all rows where the oracle is quick,
  sampled rows for the 151936-row head).
* Properties the pages ask of the operator (engine card, Checks section:
  FP8/NVFP4 GEMVs for 1-8 columns with column invariance; crit README,
  Kernel workbench: the same bits on a repeat).
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


def assert_close(orc, y_gpu, yref, a, what=""):
    bad, worst = orc.check(bits(y_gpu), yref, a)
    assert bad == 0, f"{what}: {bad} elements out of tolerance (worst ratio {worst:.3g})"
    return worst


# ------------------------------------------------------------------ packers

PACK_SHAPES = [(256, 512), (17, 80), (48, 16), (1, 16), (130, 1040), (300, 2064), (64, 5120)]


@pytest.mark.parametrize("M,K", PACK_SHAPES)
def test_nvfp4_pack_is_bit_exact(vg, orc, M, K):
    W = rand_w(M * 7 + K, M, K)
    W[0, :16] = 0.0                                       # zero block
    if M > 2:
        W[2, 16:32 if K > 16 else 16] *= 1e-5             # tiny (subnormal) scale
    wt = vg.nvfp4_pack(W.cuda())
    nib_g, sc_g = vg.nvfp4_unpack(wt)
    nib, sc, gs = orc.nvfp4_quantise(W.numpy())
    assert wt.gscale == gs
    assert np.array_equal(sc_g.cpu().numpy(), sc)
    assert np.array_equal(nib_g.cpu().numpy(), nib)


@pytest.mark.parametrize("M,K", PACK_SHAPES)
def test_fp8_pack_is_bit_exact(vg, orc, M, K):
    W = rand_w(M * 11 + K, M, K)
    W[M // 2] = 0.0                                       # zero row
    wt = vg.fp8_pack(W.cuda())
    q, rs = orc.fp8_quantise(W.numpy())
    assert np.array_equal(wt.rowscale.cpu().numpy(), rs)
    assert np.array_equal(vg.fp8_unpack(wt).cpu().numpy(), q)


def test_nvfp4_all_zero_matrix(vg, orc):
    wt = vg.nvfp4_pack(torch.zeros(32, 64, device="cuda"))
    assert wt.gscale == 0.0
    y = vg.gemv(wt, rand_x(1, 3, 64).cuda())
    assert not y.float().any()


def test_pack_rejects_non_finite(vg):
    for bad in (float("nan"), float("inf")):
        W = torch.zeros(16, 32, device="cuda")
        W[3, 5] = bad
        with pytest.raises(vg.VGError):
            vg.nvfp4_pack(W)
        with pytest.raises(vg.VGError):
            vg.fp8_pack(W)


def test_from_canonical_round_trip(vg):
    rng = np.random.default_rng(3)
    M, K = 40, 320
    nib = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    sc = rng.integers(1, 0x7F, (M, K // 16), dtype=np.uint8)     # no zero, no NaN
    wt = vg.nvfp4_from_canonical(torch.from_numpy(nib).cuda(), torch.from_numpy(sc).cuda(), 0.5)
    n2, s2 = vg.nvfp4_unpack(wt)
    assert np.array_equal(n2.cpu().numpy(), nib) and np.array_equal(s2.cpu().numpy(), sc)
    # a zero scale stores zero codes (the block's value is 0 either way)
    sc[1, 2] = 0
    wt = vg.nvfp4_from_canonical(torch.from_numpy(nib).cuda(), torch.from_numpy(sc).cuda(), 0.5)
    n2, _ = vg.nvfp4_unpack(wt)
    assert not n2.cpu().numpy()[1, 16:24].any()
    # negative or NaN scale bytes are rejected
    for b in (0x80, 0x7F):
        sc[0, 0] = b
        with pytest.raises(vg.VGError):
            vg.nvfp4_from_canonical(torch.from_numpy(nib).cuda(), torch.from_numpy(sc).cuda(), 1.0)
    q = rng.integers(0, 256, (M, K), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0
    f8 = vg.fp8_from_canonical(torch.from_numpy(q).cuda(), torch.ones(M, device="cuda"))
    assert np.array_equal(vg.fp8_unpack(f8).cpu().numpy(), q)
    q[3, 3] = 0xFF
    with pytest.raises(vg.VGError):
        vg.fp8_from_canonical(torch.from_numpy(q).cuda(), torch.ones(M, device="cuda"))


# --------------------------------------------------------------------- GEMV

GEMV_SHAPES = [
    (256, 512, (1,)),             # tiny workload shape
    (17, 80, (1, 3, 8)),          # ragged rows, K tail inside a unit
    (272, 1088, (1, 2, 5, 8)),    # 17 tiles (two row blocks), K tail chunk
    (520, 2560, (8,)),            # several row blocks x chunks: stream-K splits
    (4096, 576, (2,)),            # many row blocks, short K
    (1, 16, (1, 8)),              # one row, the smallest K (one scale block)
    (33, 48, (4,)),               # K below one unit (row-copied x)
    (300, 1600, (3, 8)),          # K a multiple of 64 with a 1-unit tail chunk
    # items of several chunks of fewer tiles (row blocks of rt < 16 tiles)
    (100, 1024, (1, 7, 8)),       # NVFP4 rt 8: one ragged row block; FP8 rt 4: two
    (100, 4096, (2, 8)),          # NVFP4 rt 4, FP8 rt 2 (8 chunks): row blocks split in two
    (5000, 2048, (8,)),           # rt 4, 79 row blocks, the last of 2 tiles and 8 rows
    (333, 3072, (5,)),            # NVFP4 rt 8, FP8 rt 4, three items per row block
]


@pytest.mark.parametrize("M,K,Ns", GEMV_SHAPES)
def test_gemv_nvfp4_parity(vg, orc, M, K, Ns):
    W = rand_w(M + 3 * K, M, K)
    wt = vg.nvfp4_pack(W.cuda())
    nib, sc, gs = orc.nvfp4_quantise(W.numpy())
    ws = vg.workspace_for(wt)
    for N in Ns:
        x = rand_x(N + M, N, K, outliers=min(8, K // 16))
        y = vg.gemv(wt, x.cuda(), workspace=ws)
        yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(x), threads=THREADS)
        assert_close(orc, y, yref, a, f"nvfp4 {M}x{K} N={N}")
    assert vg.workspace_error(ws) == 0
    err, finished, epoch = ws[:12].cpu().numpy().view(np.uint32)
    assert finished == 0, "the finished-block count must be left at zero"
    assert epoch == len(Ns), "each call advances the pass counter once"


def test_gemv_pass_counter_wrap(vg, orc):
    """Split row blocks (32 items on 32 blocks, every row block of 16 tiles
    summed from 8 blocks' tagged partials) stay exact when the pass counter
    that tags them reaches its end: the pass then restarts the counter at 0
    and clears every slot, and the next pass's tags are fresh again."""
    M, K, N = 1024, 4032, 8
    W = rand_w(77, M, K)
    wt = vg.nvfp4_pack(W.cuda())
    nib, sc, gs = orc.nvfp4_quantise(W.numpy())
    x = rand_x(78, N, K).cuda()
    ws = vg.workspace_for(wt)
    y0 = vg.gemv(wt, x, workspace=ws)
    yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(x.cpu()), threads=THREADS)
    assert_close(orc, y0, yref, a, "before the wrap")
    last = np.array([0xFFFFFFFE], dtype=np.uint32).view(np.uint8)
    ws[8:12] = torch.from_numpy(last).cuda()
    y1 = vg.gemv(wt, x, workspace=ws)          # tags 0xFFFFFFFF, then wrap
    torch.cuda.synchronize()
    assert int(ws[8:12].cpu().numpy().view(np.uint32)[0]) == 0
    assert not ws[256:].any(), "the wrap clears every partial-sum slot"
    y2 = vg.gemv(wt, x, workspace=ws)          # tags 1 again
    assert int(ws[8:12].cpu().numpy().view(np.uint32)[0]) == 1
    assert vg.workspace_error(ws) == 0
    assert torch.equal(y0, y1) and torch.equal(y0, y2)


def test_gemv_pass_counter_wrap_after_a_larger_grid(vg, orc):
    """Calls of different grid sizes share one workspace.  A large-grid call
    (256 items on every SM, row blocks split over about five blocks) fills
    the partial-sum slots with its tags; the pass counter is then set to its
    last value and a small-grid call (8 blocks) wraps it.  The wrap must clear
    every slot the workspace holds, not only the small call's: otherwise the
    next large-grid call, whose tags restart at the first call's, would accept
    the first call's stale sums.  That call uses a different x, so stale sums
    would show."""
    K, N = 4032, 8
    big, small = rand_w(91, 8192, K), rand_w(92, 256, K)
    wb, wsm = vg.nvfp4_pack(big.cuda()), vg.nvfp4_pack(small.cuda())
    ws = vg.workspace_for(wb)
    assert ws.numel() >= vg.workspace_for(wsm).numel()
    xa, xb = rand_x(93, N, K).cuda(), rand_x(94, N, K).cuda()
    vg.gemv(wb, xa, workspace=ws)              # epoch 0: every slot tagged 1
    torch.cuda.synchronize()
    last = np.array([0xFFFFFFFE], dtype=np.uint32).view(np.uint8)
    ws[8:12] = torch.from_numpy(last).cuda()
    ys = vg.gemv(wsm, xa, workspace=ws)        # 8 blocks; wraps the counter
    torch.cuda.synchronize()
    assert int(ws[8:12].cpu().numpy().view(np.uint32)[0]) == 0
    assert not ws[256:].any(), "the wrap clears every slot of the workspace"
    yb = vg.gemv(wb, xb, workspace=ws)         # tags 1 again
    assert vg.workspace_error(ws) == 0
    nib, sc, gs = orc.nvfp4_quantise(big.numpy())
    yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(xb.cpu()), threads=THREADS)
    assert_close(orc, yb, yref, a, "large grid after the wrap")
    nib, sc, gs = orc.nvfp4_quantise(small.numpy())
    yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(xa.cpu()), threads=THREADS)
    assert_close(orc, ys, yref, a, "small grid at the wrap")


@pytest.mark.parametrize("M,K,Ns", GEMV_SHAPES)
def test_gemv_fp8_parity(vg, orc, M, K, Ns):
    W = rand_w(M + 5 * K, M, K)
    wt = vg.fp8_pack(W.cuda())
    q, rs = orc.fp8_quantise(W.numpy())
    ws = vg.workspace_for(wt)
    for N in Ns:
        x = rand_x(N + 2 * M, N, K)
        y = vg.gemv(wt, x.cuda(), workspace=ws)
        yref, a = orc.gemv_fp8(q, rs, bits(x), threads=THREADS)
        assert_close(orc, y, yref, a, f"fp8 {M}x{K} N={N}")
    assert vg.workspace_error(ws) == 0


def test_gemv_all_max_codes_closed_form(vg, orc):
    M, K, N = 32, 256, 4
    nib = torch.full((M, K // 2), 0x77, dtype=torch.uint8)
    sc = torch.full((M, K // 16), 0x7E, dtype=torch.uint8)
    wt = vg.nvfp4_from_canonical(nib.cuda(), sc.cuda(), 2.0 ** -9)
    x = rand_x(9, N, K)
    y = vg.gemv(wt, x.cuda())
    yref, a = orc.gemv_nvfp4(nib.numpy(), sc.numpy(), 2.0 ** -9, bits(x))
    assert_close(orc, y, yref, a, "all-max")
    want = 2688.0 * 2.0 ** -9 * x.double().sum(1)[:, None]
    scale = 2688.0 * 2.0 ** -9 * x.double().abs().sum(1)[:, None]
    assert torch.all((y.double().cpu() - want).abs() <= 4e-3 * scale + 1e-6)


def test_column_invariance_and_repeat_bits(vg):
    """Column j's bits do not depend on N (1..8) or the other columns, and a
    repeated call gives the same bits."""
    M, K = 1040, 2048
    for fmt in ("nvfp4", "fp8"):
        W = rand_w(77, M, K).cuda()
        wt = vg.nvfp4_pack(W) if fmt == "nvfp4" else vg.fp8_pack(W)
        x8 = rand_x(78, 8, K).cuda()
        ref = vg.gemv(wt, x8)
        for N in range(1, 9):
            xn = x8[:N].clone()
            y = vg.gemv(wt, xn)
            assert torch.equal(y.view(torch.int16), ref[:N].view(torch.int16)), (fmt, N)
        x_other = x8.clone()
        x_other[1:] = rand_x(79, 7, K).cuda()
        y = vg.gemv(wt, x_other)
        assert torch.equal(y[0].view(torch.int16), ref[0].view(torch.int16))
        assert torch.equal(vg.gemv(wt, x8).view(torch.int16), ref.view(torch.int16))


def test_output_canaries_untouched(vg):
    M, K, N = 17, 96, 3
    wt = vg.nvfp4_pack(rand_w(5, M, K).cuda())
    buf = torch.full((N * M + 64,), 12345.0, dtype=torch.bfloat16, device="cuda")
    y = buf[32:32 + N * M].view(N, M)
    vg.gemv(wt, rand_x(6, N, K).cuda(), y=y)
    assert torch.all(buf[:32] == 12345.0) and torch.all(buf[32 + N * M:] == 12345.0)


def test_workspace_too_small_is_rejected(vg):
    wt = vg.nvfp4_pack(rand_w(1, 64, 64).cuda())
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(vg.VGError) as e:
        vg.gemv(wt, rand_x(1, 1, 64).cuda(), workspace=ws)
    assert e.value.status == 6


# ------------------------------------------------------- full-size workloads

def _full_nvfp4(vg, orc, W, Ns, outliers=0, seed=0, rows=None):
    """Pack on the GPU, quantise on the CPU (whole matrix or sampled rows
    with the whole matrix's tensor scale), compare y."""
    Wd = W.cuda()
    wt = vg.nvfp4_pack(Wd)
    Wh = W.numpy()
    gs = orc.amax(Wh) / np.float32(2688.0)
    assert wt.gscale == np.float32(gs)
    if rows is None:
        nib, sc, gs2 = orc.nvfp4_quantise(Wh)
        assert gs2 == wt.gscale
        sel = slice(None)
    else:
        nib, sc = orc.nvfp4_quantise_gs(Wh[rows], wt.gscale)
        sel = rows
    nib_g, sc_g = vg.nvfp4_unpack(wt)
    assert np.array_equal(nib_g.cpu().numpy()[sel], nib)
    assert np.array_equal(sc_g.cpu().numpy()[sel], sc)
    ws = vg.workspace_for(wt)
    for N in Ns:
        x = rand_x(seed + N, N, W.shape[1], outliers)
        y = vg.gemv(wt, x.cuda(), workspace=ws)
        yref, a = orc.gemv_nvfp4(nib, sc, wt.gscale, bits(x), threads=THREADS)
        assert_close(orc, y[:, sel] if rows is not None else y, yref, a, f"N={N}")


def test_full_projection_5120_outliers(vg, orc):
    from verify_gemm_gb300.inputs import draw_workload

    Ws, xs = draw_workload("proj", 1)
    wt = vg.nvfp4_pack(Ws[0].cuda())
    nib, sc, gs = orc.nvfp4_quantise(Ws[0].numpy())
    assert gs == wt.gscale
    x = xs[5120]
    y = vg.gemv(wt, x.cuda())
    yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(x), threads=THREADS)
    assert_close(orc, y, yref, a, "proj")


def test_full_gate_up_fused(vg, orc):
    """34816x5120 as two 17408x5120 halves with their own tensor scales,
    run as one fused group, N in {1, 2, 4, 8}."""
    from verify_gemm_gb300.inputs import draw_workload

    for N in (1, 2, 4, 8):
        Ws, xs = draw_workload("gateup", N)
        x = xs[5120].cuda()
        wts = [vg.nvfp4_pack(W.cuda()) for W in Ws]
        ys = [torch.empty(N, 17408, dtype=torch.bfloat16, device="cuda") for _ in wts]
        plan = vg.VerifyPlan([(wt, x, y, 0) for wt, y in zip(wts, ys)], N)
        plan.run()
        assert plan.check() == 0
        for W, wt, y in zip(Ws, wts, ys):
            nib, sc, gs = orc.nvfp4_quantise(W.numpy())
            assert gs == wt.gscale
            yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(xs[5120]), threads=THREADS)
            assert_close(orc, y, yref, a, f"gate/up N={N}")
        plan.close()


def test_full_down_fp8_and_head(vg, orc):
    from verify_gemm_gb300.inputs import draw_workload

    Ws, xs = draw_workload("down_head", 8)
    down, head = Ws
    wt = vg.fp8_pack(down.cuda())
    q, rs = orc.fp8_quantise(down.numpy())
    assert np.array_equal(wt.rowscale.cpu().numpy(), rs)
    for N in (1, 8):
        x = xs[17408][:N]
        y = vg.gemv(wt, x.cuda())
        yref, a = orc.gemv_fp8(q, rs, bits(x), threads=THREADS)
        assert_close(orc, y, yref, a, f"down N={N}")
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(151936 - 64, 151936),
                                     rng.integers(0, 151936, 768)]))
    _full_nvfp4(vg, orc, head, (1, 8), seed=3, rows=rows)


# ------------------------------------------------------------- verify pass

def _small_stack(vg, N, ordered, layers=2, down_fmt="fp8"):
    from verify_gemm_gb300.workloads import build_stack

    return build_stack(N, layers=layers, hidden=256, inter=704, vocab=1000, down_fmt=down_fmt,
                       seed=9)


@pytest.mark.parametrize("ordered", [True, False])
@pytest.mark.parametrize("N", [1, 8])
def test_verify_pass_small_stack(vg, orc, N, ordered):
    from verify_gemm_gb300.inputs import draw_stack_matrix

    st = _small_stack(vg, N, ordered)
    plan = st.plan(ordered=ordered)
    for _ in range(2):                      # counters are left clean for a repeat
        st.y_all.zero_()
        plan.run()
        assert plan.check() == 0
        for m, wt, x, y in zip(st.mats, st.weights, st.xs, st.ys):
            W, _ = draw_stack_matrix(m, N, 9, "cuda")
            Wh = W.cpu().numpy()
            if m.fmt == "nvfp4":
                nib, sc, gs = orc.nvfp4_quantise(Wh)
                assert gs == wt.gscale
                yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(x), threads=THREADS)
            else:
                q, rs = orc.fp8_quantise(Wh)
                yref, a = orc.gemv_fp8(q, rs, bits(x), threads=THREADS)
            assert_close(orc, y, yref, a, m.name)
    plan.close()


@pytest.mark.parametrize("ctas", [1, 2, 7])
def test_verify_pass_on_few_blocks(vg, orc, ctas):
    """The ordered pass on 1, 2 and 7 thread blocks: one block holds every row
    block whole (no partial sums at all), a few blocks split long ranges of
    items between them; every product within the tolerance of the oracle."""
    from verify_gemm_gb300.inputs import draw_stack_matrix

    N = 5
    st = _small_stack(vg, N, True)
    plan = st.plan(ordered=True, max_ctas=ctas)
    assert plan.grid == ctas
    for _ in range(2):
        st.y_all.zero_()
        plan.run()
        assert plan.check() == 0
    for m, wt, x, y in zip(st.mats, st.weights, st.xs, st.ys):
        W, _ = draw_stack_matrix(m, N, 9, "cuda")
        Wh = W.cpu().numpy()
        if m.fmt == "nvfp4":
            nib, sc, gs = orc.nvfp4_quantise(Wh)
            yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(x), threads=THREADS)
        else:
            q, rs = orc.fp8_quantise(Wh)
            yref, a = orc.gemv_fp8(q, rs, bits(x), threads=THREADS)
        assert_close(orc, y, yref, a, f"{m.name} on {ctas} blocks")
    plan.close()


@pytest.mark.parametrize("ordered", [True, False])
@pytest.mark.parametrize("N", [3, 8])
def test_verify_pass_multi_chunk_items(vg, orc, N, ordered):
    """A stack whose matrices take items of several chunks: NVFP4 1024-column
    matrices in row blocks of 8 tiles (2 chunks per item) and the FP8 down
    projection (K 2048) in row blocks of 2 tiles (8 chunks per item), so the
    warps sharing a tile add their sums in shared memory before the row
    blocks split between thread blocks are reduced."""
    from verify_gemm_gb300.inputs import draw_stack_matrix
    from verify_gemm_gb300.workloads import build_stack

    st = build_stack(N, layers=2, hidden=1024, inter=2048, vocab=1000, down_fmt="fp8", seed=11)
    plan = st.plan(ordered=ordered)
    plan.run()
    assert plan.check() == 0
    for m, wt, x, y in zip(st.mats, st.weights, st.xs, st.ys):
        W, _ = draw_stack_matrix(m, N, 11, "cuda")
        Wh = W.cpu().numpy()
        if m.fmt == "nvfp4":
            nib, sc, gs = orc.nvfp4_quantise(Wh)
            yref, a = orc.gemv_nvfp4(nib, sc, gs, bits(x), threads=THREADS)
        else:
            q, rs = orc.fp8_quantise(Wh)
            yref, a = orc.gemv_fp8(q, rs, bits(x), threads=THREADS)
        assert_close(orc, y, yref, a, m.name)
    plan.close()


@pytest.mark.parametrize("ordered", [True, False])
def test_verify_pass_mixed_item_shapes_in_one_group(vg, orc, ordered):
    """One group holding matrices whose items have different shapes: 16-tile
    row blocks (256 x 512), 8-tile row blocks of 2-chunk items (NVFP4
    100 x 1024) and 2-tile row blocks of 8-chunk items (FP8 100 x 4096),
    followed by a second group; every product matches the oracle."""
    N = 6
    specs = [("nvfp4", 256, 512, 0), ("nvfp4", 100, 1024, 0), ("fp8", 100, 4096, 0),
             ("nvfp4", 300, 1024, 1)]
    entries, refs = [], []
    for i, (fmt, M, K, group) in enumerate(specs):
        W = rand_w(90 + i, M, K)
        x = rand_x(190 + i, N, K).cuda()
        y = torch.zeros((N, M), dtype=torch.bfloat16, device="cuda")
        if fmt == "nvfp4":
            wt = vg.nvfp4_pack(W.cuda())
            nib, sc, gs = orc.nvfp4_quantise(W.numpy())
            refs.append(orc.gemv_nvfp4(nib, sc, gs, bits(x.cpu()), threads=THREADS))
        else:
            wt = vg.fp8_pack(W.cuda())
            q, rs = orc.fp8_quantise(W.numpy())
            refs.append(orc.gemv_fp8(q, rs, bits(x.cpu()), threads=THREADS))
        entries.append((wt, x, y, group))
    plan = vg.VerifyPlan(entries, N, ordered=ordered)
    for _ in range(2):
        plan.run()
        assert plan.check() == 0
        for (fmt, M, K, _), (_, _, y, _), (yref, a) in zip(specs, entries, refs):
            assert_close(orc, y, yref, a, f"{fmt} {M}x{K}")
    plan.close()


def test_verify_pass_ordered_and_unordered_agree(vg):
    st = _small_stack(vg, 4, True, layers=3)
    outs = []
    for ordered in (True, False):
        st.y_all.zero_()
        plan = st.plan(ordered=ordered, max_ctas=40)
        plan.run()
        assert plan.check() == 0
        outs.append(st.y_all.clone())
        plan.close()
    # the two modes split K between blocks at different points, so their FP32
    # sums may round differently: they agree within the tolerance scale
    assert torch.allclose(outs[0].float(), outs[1].float(), rtol=2e-2, atol=1e-2)


def test_graph_capture_replays_gemv_and_verify_pass(vg):
    """A GEMV and an ordered verify pass captured in one CUDA graph replay to
    the same bits as the eager calls: the launches are cooperative, their x
    tensor maps travel in the kernel parameters, and the workspace and plan
    state advance on the device, so each replay leaves them clean."""
    M, K, N = 520, 2560, 8
    wt = vg.nvfp4_pack(rand_w(5, M, K).cuda())
    x = rand_x(6, N, K).cuda()
    ws = vg.workspace_for(wt)
    y_eager = vg.gemv(wt, x, workspace=ws)
    st = _small_stack(vg, 4, True)
    plan = st.plan(ordered=True)
    st.y_all.zero_()
    plan.run()
    torch.cuda.synchronize()
    stack_eager = st.y_all.clone()
    y = torch.empty_like(y_eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):            # warm-up on a side stream
        vg.gemv(wt, x, y=y, workspace=ws)
        plan.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        vg.gemv(wt, x, y=y, workspace=ws)
        plan.run()
    for _ in range(3):
        y.zero_()
        st.y_all.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_eager)
        assert torch.equal(st.y_all, stack_eager)
    assert vg.workspace_error(ws) == 0
    assert plan.check() == 0
    plan.close()


def test_verify_pass_wait_timeout_reports_error(vg):
    """A group whose completion is never signalled makes the next group's
    bounded wait run out: the pass returns, the plan reports a timeout, and
    after the reset the same plan runs clean."""
    st = _small_stack(vg, 2, True)
    plan = st.plan(ordered=True, wait_timeout_ns=2_000_000, hold_group=0)
    plan.run()
    torch.cuda.synchronize()
    err = plan.check()
    assert err == 3
    plan.close()
    plan = st.plan(ordered=True)
    plan.run()
    assert plan.check() == 0
    plan.close()


@pytest.mark.parametrize("attn_fmt", ["nvfp4", "fp8"])
def test_full_stack_sampled(vg, orc, attn_fmt):
    """The 64-layer stack + head in the launch configuration the benchmark
    times (ordered), at every width it reports (N = 8, 4, 2, 1): sampled
    matrices checked row-sampled.  One packed stack serves all widths; the
    narrower passes take the first N rows of each x (a column's result does
    not depend on the others).  With FP8 q/k/v/o (the 19.28 GB mix) those run
    as items of 4 tiles x 4 chunks."""
    from verify_gemm_gb300.inputs import draw_stack_matrix
    from verify_gemm_gb300.workloads import build_stack

    st = build_stack(8, attn_fmt=attn_fmt)
    rng = np.random.default_rng(1)
    picks = [0, 3, 4, 6, len(st.mats) // 2 + 2, len(st.mats) - 2, len(st.mats) - 1]
    refs = {}
    for i in picks:
        m, wt = st.mats[i], st.weights[i]
        W, _ = draw_stack_matrix(m, 8, 4, "cuda")
        rows = np.unique(np.concatenate([[0, m.M - 1], rng.integers(0, m.M, 256)]))
        Wh = W.cpu().numpy()
        if m.fmt == "nvfp4":
            assert wt.gscale == np.float32(orc.amax(Wh)) / np.float32(2688.0)
            refs[i] = (rows, orc.nvfp4_quantise_gs(Wh[rows], wt.gscale))
        else:
            refs[i] = (rows, orc.fp8_quantise(Wh[rows]))
        del W, Wh
    for N in (8, 4, 2, 1):
        if N == 8:
            xs, ys = st.xs, st.ys
        else:
            xs = [x[:N] for x in st.xs]
            ys = [torch.zeros((N, m.M), dtype=torch.bfloat16, device="cuda") for m in st.mats]
        plan = vg.VerifyPlan([(wt, x, y, m.group) for m, wt, x, y in
                              zip(st.mats, st.weights, xs, ys)], N, ordered=True)
        plan.run()
        assert plan.check() == 0
        for i in picks:
            m, wt, x, y = st.mats[i], st.weights[i], xs[i], ys[i]
            rows, qz = refs[i]
            if m.fmt == "nvfp4":
                yref, a = orc.gemv_nvfp4(qz[0], qz[1], wt.gscale, bits(x), threads=THREADS)
            else:
                yref, a = orc.gemv_fp8(qz[0], qz[1], bits(x), threads=THREADS)
            assert_close(orc, y[:, rows], yref, a, f"{m.name} N={N}")
        plan.close()
        del ys


def test_quickstart_example_runs(vg):
    """examples/quickstart.py, the library's usage example, runs as written."""
    import os

    path = os.path.join(os.path.dirname(os.path.dirname(__file__)), "examples", "quickstart.py")
    scope = {"__file__": path, "__name__": "quickstart"}
    exec(compile(open(path).read(), path, "exec"), scope)
    y = scope["y"]
    assert y.shape == (8, 5120) and y.dtype == torch.bfloat16 and torch.isfinite(y.float()).all()


def test_fused_layer_example_runs(vg):
    """examples/fused_layer.py, the fused-pass usage example, runs as written
    (it checks its gated activation against PyTorch arithmetic itself)."""
    path = os.path.join(os.path.dirname(os.path.dirname(__file__)), "examples", "fused_layer.py")
    scope = {"__file__": path, "__name__": "fused_layer"}
    exec(compile(open(path).read(), path, "exec"), scope)
    h, y = scope["h"], scope["y"]
    assert h.shape == (8, 2816) and y.shape == (8, 1024)
    assert torch.isfinite(h.float()).all() and torch.isfinite(y.float()).all()


def test_graph_width_example_runs(vg):
    """examples/graph_width.py, the captured-graph usage example, runs as
    written (it compares each width's columns with the full-width replay)."""
    path = os.path.join(os.path.dirname(os.path.dirname(__file__)), "examples", "graph_width.py")
    scope = {"__file__": path, "__name__": "graph_width"}
    exec(compile(open(path).read(), path, "exec"), scope)
    y_full = scope["y_full"]
    assert y_full.shape == (8, 2048) and torch.isfinite(y_full.float()).all()
    assert torch.count_nonzero(y_full) > 0


def test_c_example_builds_and_runs(vg, tmp_path):
    """examples/c_gemv.c drives the C ABI from C with no Python: nvcc
    compiles and links it against libvgemm.so, and the program packs,
    runs the GEMV, reads the device error word and checks its own y."""
    import subprocess

    from verify_gemm_gb300 import build as B

    root = os.path.dirname(os.path.dirname(__file__))
    exe = str(tmp_path / "c_gemv")
    cmd = [B.nvcc(), "-x", "c", "-O2", os.path.join(root, "examples", "c_gemv.c"),
           f"-I{os.path.join(root, 'include')}", f"-L{B.OUT_DIR}", "-lvgemm", "-lm",
           "-Xlinker", "-rpath", "-Xlinker", B.OUT_DIR, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "worst error / tolerance" in r.stdout
