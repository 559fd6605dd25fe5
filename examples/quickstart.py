"""Quick start: pack a weight, run one GEMV and a two-group verify pass.

Run from the repository root on a GB300: ``python examples/quickstart.py``.
Device tensors come from torch; every step runs in libvgemm.so.
"""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch
import verify_gemm_gb300 as vg

W = torch.randn(5120, 5120, device="cuda") * 0.02          # FP32 weights
wt = vg.nvfp4_pack(W)                                        # or vg.fp8_pack(W)
x = torch.randn(8, 5120, device="cuda").to(torch.bfloat16)   # N = 8 columns
ws = vg.workspace_for(wt)                                    # zero-filled once, reused
y = vg.gemv(wt, x, workspace=ws)                             # BF16 [8, 5120]

# a fused pass over many matrices: (weight, x, y, group); group g waits for g - 1
plan = vg.VerifyPlan([(wt, x, y, 0), (wt, x, torch.empty_like(y), 1)], N=8)
plan.run()
assert plan.check() == 0                                     # device error word
plan.close()

print("y", tuple(y.shape), y.dtype)
