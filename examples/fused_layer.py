"""A transformer layer's weight-streaming work as one fused verify pass.

Groups, each waiting for the one before it:
  0  RMS norm of the layer input              (no weights)
  1  q, k, v projections of the norm's y      (NVFP4; x written by group 0)
  2  o projection of the attention output     (NVFP4; x given, not in this path)
  3  RMS norm of the MLP input
  4  gate and up with the SiLU-gated epilogue (NVFP4 pair; x written by group 3)
  5  down projection of the activation        (row-scaled FP8; x written by group 4)
and, for one width, the same pass read from a device word.

Run from the repository root on a GB300: ``python examples/fused_layer.py``.
Device tensors come from torch; every step runs in libvgemm.so.  The check
at the end compares the gated activation with plain PyTorch arithmetic on
the weights as packed (unpacked to the canonical codes and dequantised
here), which agrees within a BF16 rounding or two.
"""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch
import verify_gemm_gb300 as vg

torch.manual_seed(0)
N, H, I = 8, 1024, 2816            # columns (drafts), hidden size, MLP width
dev = "cuda"


def bf16(*shape):
    return torch.empty(shape, dtype=torch.bfloat16, device=dev)


x_attn = torch.randn(N, H, device=dev).to(torch.bfloat16)   # layer input
x_o = torch.randn(N, H, device=dev).to(torch.bfloat16)      # attention output
x_mlp = torch.randn(N, H, device=dev).to(torch.bfloat16)    # MLP input
gamma1 = (1 + 0.1 * torch.randn(H, device=dev)).to(torch.bfloat16)
gamma2 = (1 + 0.1 * torch.randn(H, device=dev)).to(torch.bfloat16)

wq, wk, wv, wo = (vg.nvfp4_pack(torch.randn(H, H, device=dev) * 0.02) for _ in range(4))
Wg, Wu = torch.randn(I, H, device=dev) * 0.02, torch.randn(I, H, device=dev) * 0.02
gate_up = vg.nvfp4_pack_gated(Wg, Wu)                        # I gate + I up rows
down = vg.fp8_pack(torch.randn(H, I, device=dev) * 0.02)

n1, q, k, v, o, n2, h, y = bf16(N, H), bf16(N, H), bf16(N, H), bf16(N, H), bf16(N, H), \
    bf16(N, H), bf16(N, I), bf16(N, H)
entries = [
    (vg.RMSNorm(gamma1), x_attn, n1, 0),
    (wq, n1, q, 1, True), (wk, n1, k, 1, True), (wv, n1, v, 1, True),
    (wo, x_o, o, 2),
    (vg.RMSNorm(gamma2), x_mlp, n2, 3),
    (gate_up, n2, h, 4, True),                               # h = SiLU(x Wg^T) * (x Wu^T)
    (down, h, y, 5, True),
]
plan = vg.VerifyPlan(entries, N)
plan.run()
assert plan.check() == 0                                     # device error word

# the same plan at width 3, chosen on the device (e.g. by a drafting kernel)
width = torch.full((1,), 3, dtype=torch.int32, device=dev)
plan.set_width(width)
plan.run()
assert plan.check() == 0
plan.set_width(None)
plan.close()

# check the gated activation against PyTorch arithmetic on the packed weights
nib, sc = vg.nvfp4_unpack(gate_up)                           # canonical codes, gate/up interleaved
e2m1 = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6], device=dev)


def e4m3(b):
    b = b.to(torch.int32)
    e, f = (b >> 3) & 15, (b & 7).to(torch.float32)
    return torch.where(e == 0, f * 2.0 ** -9, (1 + f / 8) * 2.0 ** (e.float() - 7))


codes = torch.stack([nib & 15, nib >> 4], dim=-1).reshape(2 * I, H).to(torch.int64)
w_hat = torch.where(codes >= 8, -1.0, 1.0) * e2m1[codes & 7] * e4m3(sc).repeat_interleave(16, 1)
tiles = w_hat.reshape(I // 8, 2, 8, H)                       # tiles of 8 gate + 8 up rows
wg_hat = tiles[:, 0].reshape(I, H) * gate_up.gscale
wu_hat = tiles[:, 1].reshape(I, H) * gate_up.gscale_up
g = n2.float() @ wg_hat.T
u = n2.float() @ wu_hat.T
h_ref = torch.nn.functional.silu(g) * u
err = ((h.float() - h_ref).abs() / (h_ref.abs() + 1e-3)).max().item()
print(f"gated activation: max relative difference {err:.2e} (BF16 output)")
assert err < 3e-2
print("q", tuple(q.shape), "h", tuple(h.shape), "y", tuple(y.shape))
