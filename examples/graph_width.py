"""One CUDA graph per decode round, the verify width chosen on the device.

A speculative-decoding round drafts a variable number of tokens and then
verifies them in one pass over the weights.  Here the verify pass (a small
two-group stack) is captured once in a CUDA graph; before each replay a
kernel on the stream writes how many columns to verify (standing in for the
drafting step, which knows how many drafts it made), and the pass reads that
width from device memory at launch.  The host never waits between the two.

Run from the repository root on a GB300: ``python examples/graph_width.py``.
"""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch
import verify_gemm_gb300 as vg

torch.manual_seed(0)
N_MAX, H = 8, 2048
dev = "cuda"
w1 = vg.nvfp4_pack(torch.randn(H, H, device=dev) * 0.02)
w2 = vg.nvfp4_pack(torch.randn(H, H, device=dev) * 0.02)
x = torch.randn(N_MAX, H, device=dev).to(torch.bfloat16)
y1 = torch.zeros(N_MAX, H, dtype=torch.bfloat16, device=dev)
y2 = torch.zeros(N_MAX, H, dtype=torch.bfloat16, device=dev)

plan = vg.VerifyPlan([(w1, x, y1, 0), (w2, y1, y2, 1, True)], N_MAX)   # y2 = f(f(x))
width = torch.full((1,), N_MAX, dtype=torch.int32, device=dev)
plan.set_width(width)                      # each pass reads its width from here

# warm up on a side stream, then capture one pass
side = torch.cuda.Stream()
side.wait_stream(torch.cuda.current_stream())
with torch.cuda.stream(side):
    plan.run()
torch.cuda.current_stream().wait_stream(side)
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph):
    plan.run()

width.fill_(N_MAX)
graph.replay()
y_full = y2.clone()                        # all N_MAX columns

for drafts in (3, 1, 7):
    width.fill_(drafts + 1)                # a device-side write, ordered before the replay
    y2.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert plan.check() == 0               # device error word
    w = drafts + 1
    # a column's result does not depend on the others, and the rows past the
    # width are not written
    assert torch.equal(y2[:w], y_full[:w])
    assert torch.count_nonzero(y2[w:]) == 0
    print(f"verified {w} of {N_MAX} columns with one captured graph")
plan.set_width(None)
plan.close()
