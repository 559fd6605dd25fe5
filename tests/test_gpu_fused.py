"""Fused neighbours of the GEMV inside one verify pass, with real data
dependencies: the RMS normalisation before q/k/v and before the MLP (engine
card, Checks section: row reductions are checked next to the GEMVs) and the
SiLU-gated activation fused into the epilogue of the gate/up pair, whose
output is the down projection's x (card, Model section: the MLPs).

The oracle computes every intermediate itself (its own normalised x, its
own gate and up sums and activation, rounded to BF16 where the pass stores
them) and checks each stored result: RMS norms within one BF16 unit in the
last place, gated activations within the bound derived from the GEMV
tolerance (oracle.swiglu), GEMVs within the GEMV tolerance.  Intermediate
buffers start filled with a canary, so an x copied before its producer
finished would show.
"""
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1
CANARY = 1280.0


@pytest.fixture(scope="module")
def vg():
    from verify_gemm_gb300 import build

    build.build()
    import verify_gemm_gb300 as vg

    torch.cuda.init()
    return vg


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_of(orc, v):
    """BF16 bits of FP64 values, one rounding each (oracle)."""
    flat = np.asarray(v, dtype=np.float64).ravel()
    return np.array([orc.bf16_round(x) for x in flat], dtype=np.uint16).reshape(np.shape(v))


def ulp_diff(a_bits, b_bits):
    """Distance in BF16 steps between two arrays of finite BF16 bits."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(key(a_bits) - key(b_bits))


def check_norm(orc, y, x, gamma, eps, what):
    want = orc.rmsnorm(bits(x), bits(gamma), eps)
    d = ulp_diff(bits(y), want)
    assert d.max() <= 1, f"{what}: {int((d > 1).sum())} elements more than 1 BF16 step off"
    assert (d > 0).mean() <= 0.01, f"{what}: {(d > 0).mean():.2%} elements differ"
    return want


def quantise(orc, fmt, W, rows=None, gs_gpu=None):
    """The oracle's quantisation of W (or of its sampled rows, with the whole
    matrix's tensor scale, computed by the oracle and checked against the
    packer's)."""
    Wh = W.cpu().numpy()
    if fmt == "nvfp4":
        if rows is None:
            nib, sc, gs = orc.nvfp4_quantise(Wh)
        else:
            gs = np.float32(orc.amax(Wh)) / np.float32(2688.0)
            nib, sc = orc.nvfp4_quantise_gs(Wh[rows], gs)
        if gs_gpu is not None:
            assert gs == np.float32(gs_gpu)
        return ("nvfp4", nib, sc, gs)
    q, rs = orc.fp8_quantise(Wh if rows is None else Wh[rows])
    return ("fp8", q, rs)


def gemv_ref(orc, qz, x_bits):
    if qz[0] == "nvfp4":
        return orc.gemv_nvfp4(qz[1], qz[2], qz[3], x_bits, threads=THREADS)
    return orc.gemv_fp8(qz[1], qz[2], x_bits, threads=THREADS)


def deinterleave(t, I):
    """Canonical rows of a gated pair (tiles of 8 gate + 8 up rows) -> halves."""
    v = t.reshape(I // 8, 2, 8, *t.shape[1:])
    return v[:, 0].reshape(I, *t.shape[1:]), v[:, 1].reshape(I, *t.shape[1:])


# ------------------------------------------------------------ gated packers

@pytest.mark.parametrize("I,K", [(64, 512), (200, 1040), (1088, 2048)])
def test_gated_pack_is_bit_exact(vg, orc, I, K):
    g = torch.Generator().manual_seed(I + K)
    Wg = torch.randn((I, K), generator=g) * 0.02
    Wu = torch.randn((I, K), generator=g) * 0.05
    pair = vg.nvfp4_pack_gated(Wg.cuda(), Wu.cuda())
    nib, sc = vg.nvfp4_unpack(pair)
    for half, W, gs in ((0, Wg, pair.gscale), (1, Wu, pair.gscale_up)):
        n_ref, s_ref, gs_ref = orc.nvfp4_quantise(W.numpy())
        assert gs == gs_ref
        assert np.array_equal(deinterleave(nib.cpu().numpy(), I)[half], n_ref)
        assert np.array_equal(deinterleave(sc.cpu().numpy(), I)[half], s_ref)
    p8 = vg.fp8_pack_gated(Wg.cuda(), Wu.cuda())
    q = vg.fp8_unpack(p8).cpu().numpy()
    for half, W, rs in ((0, Wg, p8.rowscale), (1, Wu, p8.rowscale_up)):
        q_ref, rs_ref = orc.fp8_quantise(W.numpy())
        assert np.array_equal(rs.cpu().numpy(), rs_ref)
        assert np.array_equal(deinterleave(q, I)[half], q_ref)


# ------------------------------------------------- one fused op in a plan

@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
@pytest.mark.parametrize("I,K,Ns", [(1088, 2048, (1, 8)), (200, 1040, (5,)), (4096, 576, (3,))])
def test_gated_activation(vg, orc, fmt, I, K, Ns):
    g = torch.Generator().manual_seed(3 * I + K)
    Wg = torch.randn((I, K), generator=g) * 0.02
    Wu = torch.randn((I, K), generator=g) * 0.02
    pair = (vg.nvfp4_pack_gated if fmt == "nvfp4" else vg.fp8_pack_gated)(Wg.cuda(), Wu.cuda())
    qg = quantise(orc, fmt, Wg)
    qu = quantise(orc, fmt, Wu)
    for N in Ns:
        x = (torch.randn((N, K), generator=g) * 3).to(torch.bfloat16).cuda()
        h = torch.full((N, I), CANARY, dtype=torch.bfloat16, device="cuda")
        plan = vg.VerifyPlan([(pair, x, h, 0)], N)
        plan.run()
        assert plan.check() == 0
        plan.close()
        gr, ag = gemv_ref(orc, qg, bits(x))
        ur, au = gemv_ref(orc, qu, bits(x))
        href, bound = orc.swiglu(gr, ur, ag, au)
        err = np.abs(h.float().cpu().numpy().astype(np.float64) - href)
        worst = float((err / bound).max())
        assert worst <= 1.0, f"{fmt} {I}x{K} N={N}: worst error / bound {worst:.3g}"


@pytest.mark.parametrize("fmt", ["nvfp4", "fp8"])
def test_gated_activation_saturates(vg, orc, fmt):
    """Gates far past SiLU's bends: gate rows of constant weight +-0.5 (exact
    in both formats) against x rows of constant sign give g near +-512 and
    +-128, where SiLU(g) is g or underflows to zero (exp(-g) overflows FP32
    below -88.7).  Every h is finite and within the bound."""
    I, K, N = 64, 1024, 4
    g = torch.Generator().manual_seed(91)
    Wg = torch.randn((I, K), generator=g) * 0.02
    Wg[:32] = 0.5 * torch.sign(torch.randn((32, 1), generator=g))
    Wu = torch.randn((I, K), generator=g) * 0.02
    xf = torch.empty((N, K))
    xf[0], xf[1], xf[3] = 1.0, -1.0, 0.25
    xf[2] = torch.randn(K, generator=g) * 3
    x = xf.to(torch.bfloat16).cuda()
    pair = (vg.nvfp4_pack_gated if fmt == "nvfp4" else vg.fp8_pack_gated)(Wg.cuda(), Wu.cuda())
    h = torch.full((N, I), CANARY, dtype=torch.bfloat16, device="cuda")
    plan = vg.VerifyPlan([(pair, x, h, 0)], N)
    plan.run()
    assert plan.check() == 0
    plan.close()
    gr, ag = gemv_ref(orc, quantise(orc, fmt, Wg), bits(x))
    ur, au = gemv_ref(orc, quantise(orc, fmt, Wu), bits(x))
    assert np.abs(gr[:2, :32]).min() > 400          # the gates this test is about
    href, bound = orc.swiglu(gr, ur, ag, au)
    hf = h.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(hf).all()
    worst = float((np.abs(hf - href) / bound).max())
    assert worst <= 1.0, f"{fmt}: worst error / bound {worst:.3g}"


# (N, K): K = 1040 and 48 are not multiples of 64 (rows of 130 and 6 vectors
# of 8), K = 16 is the smallest K (two slices of one vector each); the last
# case has an all-zero row (its y is zero: 0 * 1 / sqrt(eps))
@pytest.mark.parametrize("N,K,zero_row", [(1, 5120, False), (8, 5120, False), (3, 512, False),
                                          (8, 17408, False), (5, 1040, False), (2, 16, False),
                                          (8, 48, False), (4, 1024, True)])
def test_rmsnorm_entry(vg, orc, N, K, zero_row):
    g = torch.Generator().manual_seed(N * K)
    x = (torch.randn((N, K), generator=g) * 2).to(torch.bfloat16).cuda()
    if zero_row:
        x[1].zero_()
    gamma = (1 + 0.1 * torch.randn((K,), generator=g)).to(torch.bfloat16).cuda()
    y = torch.full((N, K), CANARY, dtype=torch.bfloat16, device="cuda")
    plan = vg.VerifyPlan([(vg.RMSNorm(gamma, 1e-6), x, y, 0)], N)
    for _ in range(2):
        plan.run()
        assert plan.check() == 0
        check_norm(orc, y, x, gamma, 1e-6, f"N={N} K={K}")
    plan.close()


@pytest.mark.parametrize("N,K", [(8, 5120), (3, 1024), (8, 17408)])
def test_rmsnorm_of_a_produced_x(vg, orc, N, K):
    """GEMV -> RMS norm of its y (dependent x) -> GEMV of the norm's y.  At
    (N + 1) K 2 bytes within an item slot the producer copies the norm's rows
    into the item's slot only after the GEMV's group has completed; the
    widest case reads them from L2 instead.  Intermediates start as canaries."""
    g = torch.Generator().manual_seed(N * 7 + K)
    W1 = torch.randn((K, 512), generator=g) * 0.05
    W2 = torch.randn((640, K), generator=g) * 0.02
    w1, w2 = vg.nvfp4_pack(W1.cuda()), vg.nvfp4_pack(W2.cuda())
    x = torch.randn((N, 512), generator=g).to(torch.bfloat16).cuda()
    gamma = (1 + 0.1 * torch.randn((K,), generator=g)).to(torch.bfloat16).cuda()
    h = torch.full((N, K), CANARY, dtype=torch.bfloat16, device="cuda")
    hn = torch.full((N, K), CANARY, dtype=torch.bfloat16, device="cuda")
    y = torch.full((N, 640), CANARY, dtype=torch.bfloat16, device="cuda")
    plan = vg.VerifyPlan([(w1, x, h, 0), (vg.RMSNorm(gamma, 1e-6), h, hn, 1, True),
                          (w2, hn, y, 2, True)], N)
    for _ in range(2):
        for t in (h, hn, y):
            t.fill_(CANARY)
        plan.run()
        assert plan.check() == 0
        q1 = quantise(orc, "nvfp4", W1)
        h_ref, a1 = gemv_ref(orc, q1, bits(x))
        bad, worst = orc.check(bits(h), h_ref, a1)
        assert bad == 0, f"first GEMV: {bad} out of tolerance (worst {worst:.3g})"
        hn_ref = check_norm(orc, hn, h, gamma, 1e-6, f"norm of a produced x, N={N} K={K}")
        q2 = quantise(orc, "nvfp4", W2)
        y_ref, a2 = gemv_ref(orc, q2, hn_ref)
        bad, worst = orc.check(bits(y), y_ref, a2)
        assert bad == 0, f"second GEMV: {bad} out of tolerance (worst {worst:.3g})"
    plan.close()


def test_fused_ops_need_the_group_order(vg):
    x = torch.zeros((2, 512), dtype=torch.bfloat16, device="cuda")
    gamma = torch.ones(512, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vg.VGError):
        vg.VerifyPlan([(vg.RMSNorm(gamma), x, torch.empty_like(x), 0)], 2, ordered=False)
    wt = vg.nvfp4_pack(torch.randn(64, 512, device="cuda"))
    y = torch.empty((2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vg.VGError):       # the first group has no earlier group
        vg.VerifyPlan([(wt, x, y, 0, True)], 2)


# ------------------------------------------------------- the fused stack

def oracle_chain(orc, fs, seed, rows_for=None):
    """Check every entry of a fused stack against the oracle's own chain.
    rows_for(entry) -> sampled rows to check (None: all)."""
    from verify_gemm_gb300.inputs import draw_stack_matrix

    produced = {}          # data_ptr of a stored y -> the oracle's BF16 bits of it
    for e in fs.entries:
        if e.after:
            x_bits = produced[e.x.data_ptr()]
        else:
            x_bits = bits(e.x)
        if e.kind == "norm":
            want = check_norm(orc, e.y, e.x, e.op.gamma, e.op.eps, e.name)
            produced[e.y.data_ptr()] = want
            continue
        rows = rows_for(e) if rows_for else None
        if e.kind == "gemv":
            (m,) = e.mats
            W, _ = draw_stack_matrix(m, fs.N, seed, "cuda")
            qz = quantise(orc, m.fmt, W, rows, e.op.gscale if m.fmt == "nvfp4" else None)
            del W
            yref, a = gemv_ref(orc, qz, x_bits)
            y = e.y if rows is None else e.y[:, rows]
            bad, worst = orc.check(bits(y), yref, a)
            assert bad == 0, f"{e.name}: {bad} out of tolerance (worst {worst:.3g})"
        else:
            mg, mu = e.mats
            out = []
            nv = e.op.fmt == 0
            for m, gs in ((mg, e.op.gscale if nv else None), (mu, e.op.gscale_up if nv else None)):
                W, _ = draw_stack_matrix(m, fs.N, seed, "cuda")
                qz = quantise(orc, "nvfp4" if nv else "fp8", W, rows, gs)
                del W
                out.append(gemv_ref(orc, qz, x_bits))
            (gr, ag), (ur, au) = out
            href, bound = orc.swiglu(gr, ur, ag, au)
            y = e.y if rows is None else e.y[:, rows]
            err = np.abs(y.float().cpu().numpy().astype(np.float64) - href)
            worst = float((err / bound).max())
            assert worst <= 1.0, f"{e.name}: worst error / bound {worst:.3g}"
            if rows is None:
                produced[e.y.data_ptr()] = bf16_of(orc, href)


@pytest.mark.parametrize("N", [1, 8])
@pytest.mark.parametrize("mlp_fmt", ["nvfp4", "fp8"])
def test_fused_stack_small(vg, orc, N, mlp_fmt):
    from verify_gemm_gb300.workloads import build_fused_stack

    fs = build_fused_stack(N, layers=2, hidden=512, inter=1408, vocab=1000, seed=31,
                           mlp_fmt=mlp_fmt)
    plan = fs.plan()
    for rep in range(2):
        for e in fs.entries:
            e.y.fill_(CANARY)              # every output, so every produced x, starts as a canary
        plan.run()
        assert plan.check() == 0
        oracle_chain(orc, fs, 31)
    plan.close()


def test_fused_stack_width_word(vg):
    """One fused plan made for 8 columns, run at widths 1, 3, 5 and 8 read
    from its device word: every entry's first w rows equal, bit for bit,
    those of a plan made for width w alone over the same inputs (the norms'
    rows and the gated activation included), and its other rows are not
    written."""
    from verify_gemm_gb300.workloads import build_fused_stack

    fs = build_fused_stack(8, layers=2, hidden=512, inter=1408, vocab=1000, seed=33)
    plan = fs.plan()
    width = torch.zeros(1, dtype=torch.int32, device="cuda")
    plan.set_width(width)
    for w in (1, 3, 5, 8):
        for e in fs.entries:
            e.y.fill_(CANARY)
        width.fill_(w)
        plan.run()
        assert plan.check() == 0, w
        # the same pass made for width w: inputs are the first w rows, and
        # every x written by the pass is the narrow plan's own output
        outs = {}
        narrow = []
        for e in fs.entries:
            x = outs[e.x.data_ptr()] if e.after else e.x[:w].contiguous()
            y = torch.full((w, e.y.shape[1]), CANARY, dtype=torch.bfloat16, device="cuda")
            outs[e.y.data_ptr()] = y
            narrow.append((e.op, x, y, e.group, e.after))
        ref = vg.VerifyPlan(narrow, w)
        ref.run()
        assert ref.check() == 0
        ref.close()
        for e, (_, _, yn, _, _) in zip(fs.entries, narrow):
            assert torch.equal(e.y[:w].view(torch.int16), yn.view(torch.int16)), (e.name, w)
            assert torch.all(e.y[w:] == CANARY), (e.name, w)
    plan.close()


def test_fused_stack_full_size_first_layer_and_head(vg, orc):
    """The 64-layer fused stack at N = 8 as the bench times it: every entry
    of layer 0 (the gated pair and the down projection over all rows, since
    down's x is the whole activation), the last layer's norms, and the head
    on sampled rows."""
    from verify_gemm_gb300.workloads import FusedStack, build_fused_stack

    fs = build_fused_stack(8)
    plan = fs.plan()
    plan.run()
    assert plan.check() == 0
    plan.close()
    rng = np.random.default_rng(5)
    first = [e for e in fs.entries if e.layer == 0]
    oracle_chain(orc, FusedStack(first, 8), 4,
                 rows_for=lambda e: None if e.kind == "swiglu" or e.name.endswith("down")
                 else np.unique(np.concatenate([[0], rng.integers(0, e.op.M, 256)])))
    tail = [e for e in fs.entries if e.layer == 64]     # final norm + head
    oracle_chain(orc, FusedStack(tail, 8), 4,
                 rows_for=lambda e: np.unique(np.concatenate([[0, e.op.M - 1],
                                                              rng.integers(0, e.op.M, 512)])))
    last = [e for e in fs.entries if e.layer == 63 and e.kind == "norm"]
    oracle_chain(orc, FusedStack(last, 8), 4)
