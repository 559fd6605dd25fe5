"""Width dispatch on the device, and the draft step.

* One verify plan created for N = 8 columns serves every width 1..8 read
  from a device word at launch (engine card, Design table, Decode row: one
  graph per round, the verify pass run for the drafts made, 2-8 columns, no
  host wait mid-round).  For each width the written columns equal, bit for
  bit, those of a plan made for that width alone (a column's result does not
  depend on the others), the columns past the width are left untouched, and
  one captured CUDA graph replays correctly for every width.  A width
  outside 1..8 writes nothing and reports device error 5.
* The draft step at N = 1 (engine card, Model section: the drafting layer as
  row-scaled FP8, the head as NVFP4; Measured section: about 0.8 ms per
  draft step on the card's GPU): every product within the tolerance of the
  oracle, on a reduced-size layer in full and on the full-size step on
  sampled rows.
"""
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1
CANARY = 1280.0   # exact in BF16


@pytest.fixture(scope="module")
def vg():
    from verify_gemm_gb300 import build

    build.build()
    import verify_gemm_gb300 as vg

    torch.cuda.init()
    return vg


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _stack(N=8):
    from verify_gemm_gb300.workloads import build_stack

    # multi-chunk items (hidden 1024) and one-chunk items (the head, K 1024:
    # rt 16 for 1000 rows) in one stack
    return build_stack(N, layers=2, hidden=1024, inter=2048, vocab=1000, seed=21)


def _fixed_width_outputs(vg, st, w):
    """y of a plan made for width w alone over the first w rows of each x."""
    ys = [torch.zeros((w, m.M), dtype=torch.bfloat16, device="cuda") for m in st.mats]
    plan = vg.VerifyPlan([(wt, x[:w], y, m.group) for m, wt, x, y in
                          zip(st.mats, st.weights, st.xs, ys)], w, ordered=True)
    plan.run()
    assert plan.check() == 0
    plan.close()
    return ys


def test_width_read_on_the_device(vg):
    st = _stack()
    plan = st.plan(ordered=True)
    width = torch.zeros(1, dtype=torch.int32, device="cuda")
    plan.set_width(width)
    for w in range(1, 9):
        width.fill_(w)
        st.y_all.fill_(CANARY)
        plan.run()
        assert plan.check() == 0, w
        want = _fixed_width_outputs(vg, st, w)
        for m, y, yw in zip(st.mats, st.ys, want):
            assert torch.equal(bits_t(y[:w]), bits_t(yw)), (m.name, w)
            assert torch.all(y[w:] == CANARY), (m.name, w)
    plan.close()


def bits_t(t):
    return t.view(torch.int16)


def test_one_graph_serves_every_width(vg):
    """The pass is captured once; before each replay a device-side fill sets
    the width (as a drafting kernel would), and no host value changes."""
    st = _stack()
    plan = st.plan(ordered=True)
    width = torch.full((1,), 8, dtype=torch.int32, device="cuda")
    plan.set_width(width)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        plan.run()
    for w in (3, 8, 1, 6, 2):
        width.fill_(w)
        st.y_all.fill_(CANARY)
        graph.replay()
        torch.cuda.synchronize()
        want = _fixed_width_outputs(vg, st, w)
        for m, y, yw in zip(st.mats, st.ys, want):
            assert torch.equal(bits_t(y[:w]), bits_t(yw)), (m.name, w)
            assert torch.all(y[w:] == CANARY), (m.name, w)
    assert plan.check() == 0
    plan.close()


@pytest.mark.parametrize("bad", [0, 9, -1])
def test_width_out_of_range_writes_nothing(vg, bad):
    st = _stack()
    plan = st.plan(ordered=True)
    width = torch.full((1,), bad, dtype=torch.int32, device="cuda")
    plan.set_width(width)
    st.y_all.fill_(CANARY)
    plan.run()
    assert plan.check() == 5
    assert torch.all(st.y_all == CANARY)
    # the plan is clean afterwards: a valid width runs normally
    width.fill_(4)
    plan.run()
    assert plan.check() == 0
    plan.set_width(None)
    plan.run()
    assert plan.check() == 0
    plan.close()


def _check_stack(orc, st, seed, rows_per=None):
    from verify_gemm_gb300.inputs import draw_stack_matrix

    rng = np.random.default_rng(seed)
    for m, wt, x, y in zip(st.mats, st.weights, st.xs, st.ys):
        W, _ = draw_stack_matrix(m, st.N, seed, "cuda")
        Wh = W.cpu().numpy()
        del W
        rows = (np.arange(m.M) if rows_per is None else
                np.unique(np.concatenate([[0, m.M - 1], rng.integers(0, m.M, rows_per)])))
        if m.fmt == "nvfp4":
            assert wt.gscale == np.float32(orc.amax(Wh)) / np.float32(2688.0)
            nib, sc = orc.nvfp4_quantise_gs(Wh[rows], wt.gscale)
            yref, a = orc.gemv_nvfp4(nib, sc, wt.gscale, bits(x), threads=THREADS)
        else:
            q, rs = orc.fp8_quantise(Wh[rows])
            yref, a = orc.gemv_fp8(q, rs, bits(x), threads=THREADS)
        bad, worst = orc.check(bits(y[:, rows]), yref, a)
        assert bad == 0, f"{m.name}: {bad} out of tolerance (worst {worst:.3g})"


def test_draft_step_small(vg, orc):
    from verify_gemm_gb300.inputs import DRAFT_SEED, draft_mats
    from verify_gemm_gb300.workloads import build_stack

    mats = draft_mats(hidden=512, inter=1408, vocab=3000)
    st = build_stack(1, mats=mats, seed=DRAFT_SEED)
    plan = st.plan(ordered=True)
    plan.run()
    assert plan.check() == 0
    _check_stack(orc, st, DRAFT_SEED)
    plan.close()


def test_draft_step_full_size_sampled(vg, orc):
    from verify_gemm_gb300.inputs import DRAFT_SEED, draft_mats
    from verify_gemm_gb300.workloads import build_stack

    st = build_stack(1, mats=draft_mats(), seed=DRAFT_SEED)
    assert st.bytes == 810_061_828
    plan = st.plan(ordered=True)
    plan.run()
    assert plan.check() == 0
    _check_stack(orc, st, DRAFT_SEED, rows_per=256)
    plan.close()
