"""Build the synthetic verify-stack workload on the device: draw each
matrix (seeded, see ``inputs``), quantise it with the library's packer and
lay out x and y for all matrices in two contiguous buffers, so that an
end-to-end step can move every input and output with one copy each."""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (FP8Weight, NVFP4Weight, RMSNorm, VerifyPlan, fp8_pack, fp8_pack_gated, int4g_pack,
               mxfp8_pack, nvfp4_pack, nvfp4_pack_gated)
from .inputs import (HIDDEN, INTERMEDIATE, LAYERS, VOCAB, Mat, draw_norm_inputs, draw_stack_matrix,
                     stack_mats)


@dataclass
class StackSetup:
    mats: list            # Mat per matrix
    weights: list         # NVFP4Weight | FP8Weight per matrix
    xs: list              # BF16 [N, K] views into x_all
    ys: list              # BF16 [N, M] views into y_all
    x_all: torch.Tensor   # flat BF16
    y_all: torch.Tensor   # flat BF16
    N: int

    @property
    def bytes(self) -> int:
        return sum(w.nbytes for w in self.weights)

    def with_new_buffers(self) -> "StackSetup":
        """The same matrices and packed weights over a second pair of x / y
        buffers (x copied): a pass on one pair can run while the other pair's
        x is uploaded and its y read back."""
        x_all = self.x_all.clone()
        y_all = torch.zeros_like(self.y_all)
        xs = [x_all[(x.data_ptr() - self.x_all.data_ptr()) // 2:][:x.numel()].view(x.shape)
              for x in self.xs]
        ys = [y_all[(y.data_ptr() - self.y_all.data_ptr()) // 2:][:y.numel()].view(y.shape)
              for y in self.ys]
        return StackSetup(self.mats, self.weights, xs, ys, x_all, y_all, self.N)

    def plan(self, ordered: bool = True, **kw) -> VerifyPlan:
        entries = [(w, x, y, m.group) for m, w, x, y in zip(self.mats, self.weights, self.xs,
                                                              self.ys)]
        return VerifyPlan(entries, self.N, ordered=ordered, **kw)


PACKERS = {"nvfp4": nvfp4_pack, "fp8": fp8_pack, "mxfp8": mxfp8_pack, "int4g": int4g_pack}


def pack(W: torch.Tensor, fmt: str):
    return PACKERS[fmt](W)


def build_stack(N: int, device="cuda", layers: int = LAYERS, seed: int = 4,
                attn_fmt: str = "nvfp4", down_fmt: str = "fp8", hidden: int = HIDDEN,
                inter: int = INTERMEDIATE, vocab: int = VOCAB, mats=None,
                all_fmt: str | None = None) -> StackSetup:
    """Quantised layer stack (+ head) with x drawn per matrix (BF16 N(0,1)).
    all_fmt: every matrix in that format instead."""
    if mats is None:
        mats = stack_mats(layers, attn_fmt, down_fmt)
        if all_fmt is not None:
            mats = [Mat(m.name, all_fmt, m.M, m.K, m.group, m.layer, m.idx) for m in mats]
        if (hidden, inter, vocab) != (HIDDEN, INTERMEDIATE, VOCAB):
            def resize(m: Mat) -> Mat:
                dims = {HIDDEN: hidden, INTERMEDIATE: inter, VOCAB: vocab}
                return Mat(m.name, m.fmt, dims[m.M], dims[m.K], m.group, m.layer, m.idx)
            mats = [resize(m) for m in mats]
    x_off, y_off = [], []
    nx = ny = 0
    for m in mats:
        x_off.append(nx)
        y_off.append(ny)
        nx += N * m.K
        ny += N * m.M
    x_all = torch.empty(nx, dtype=torch.bfloat16, device=device)
    y_all = torch.zeros(ny, dtype=torch.bfloat16, device=device)
    weights, xs, ys = [], [], []
    for m, xo, yo in zip(mats, x_off, y_off):
        W, x = draw_stack_matrix(m, N, seed, device)
        weights.append(pack(W, m.fmt))
        del W
        xv = x_all[xo:xo + N * m.K].view(N, m.K)
        xv.copy_(x)
        xs.append(xv)
        ys.append(y_all[yo:yo + N * m.M].view(N, m.M))
    return StackSetup(mats, weights, xs, ys, x_all, y_all, N)


def weight_bytes(w) -> int:
    assert isinstance(w, (NVFP4Weight, FP8Weight))
    return w.nbytes


@dataclass
class FusedEntry:
    kind: str             # "norm", "gemv", "swiglu"
    name: str
    layer: int
    op: object            # packed weight or RMSNorm
    x: torch.Tensor
    y: torch.Tensor
    group: int
    after: bool           # x is written by the previous group
    mats: tuple = ()      # the stack matrices (Mat) behind a weight entry


@dataclass
class FusedStack:
    entries: list
    N: int

    @property
    def bytes(self) -> int:
        return sum(e.op.nbytes for e in self.entries)

    def plan(self, **kw) -> VerifyPlan:
        return VerifyPlan([(e.op, e.x, e.y, e.group, e.after) for e in self.entries], self.N,
                          ordered=True, **kw)


def build_fused_stack(N: int, device="cuda", layers: int = LAYERS, seed: int = 4,
                      attn_fmt: str = "nvfp4", mlp_fmt: str = "nvfp4", down_fmt: str = "fp8",
                      hidden: int = HIDDEN, inter: int = INTERMEDIATE, vocab: int = VOCAB,
                      eps: float = 1e-6) -> FusedStack:
    """The layer stack with its GEMV neighbours fused into the pass and real
    data dependencies.  Per layer: RMS norm -> {q, k, v} (x = the norm's y)
    -> {o} (x drawn: the attention output is not part of this path) -> RMS
    norm -> {gate+up, gated activation} (x = the norm's y) -> {down} (x = the
    activation's y); after the layers an RMS norm -> head.  The weights are
    the same draws as the plain stack's (same derived seeds); norm inputs and
    weights come from their own derived seeds."""
    def resize(m: Mat) -> Mat:
        dims = {HIDDEN: hidden, INTERMEDIATE: inter, VOCAB: vocab}
        return Mat(m.name, m.fmt, dims[m.M], dims[m.K], m.group, m.layer, m.idx)

    base = [resize(m) for m in stack_mats(layers, attn_fmt, down_fmt)]
    by_name = {m.name: m for m in base}
    entries = []
    g = 0

    def bf16(shape):
        return torch.zeros(shape, dtype=torch.bfloat16, device=device)

    def norm(layer, which, name):
        nonlocal g
        x, gamma = draw_norm_inputs(seed, layer, which, N, hidden, device)
        y = bf16((N, hidden))
        entries.append(FusedEntry("norm", name, layer, RMSNorm(gamma.contiguous(), eps), x, y, g,
                                  False))
        g += 1
        return y

    def gemv(m: Mat, x, after):
        W, xd = draw_stack_matrix(m, N, seed, device)
        wt = nvfp4_pack(W) if m.fmt == "nvfp4" else fp8_pack(W)
        del W
        if x is None:
            x = xd
        return FusedEntry("gemv", m.name, m.layer, wt, x, bf16((N, m.M)), g, after, (m,))

    for layer in range(layers):
        xn = norm(layer, 0, f"L{layer}.norm1")
        for nm in ("q", "k", "v"):
            entries.append(gemv(by_name[f"L{layer}.{nm}"], xn, True))
        g += 1
        entries.append(gemv(by_name[f"L{layer}.o"], None, False))
        g += 1
        xn2 = norm(layer, 1, f"L{layer}.norm2")
        mg, mu = by_name[f"L{layer}.gate"], by_name[f"L{layer}.up"]
        Wg, _ = draw_stack_matrix(mg, N, seed, device)
        Wu, _ = draw_stack_matrix(mu, N, seed, device)
        pair = nvfp4_pack_gated(Wg, Wu) if mlp_fmt == "nvfp4" else fp8_pack_gated(Wg, Wu)
        del Wg, Wu
        h = bf16((N, inter))
        entries.append(FusedEntry("swiglu", f"L{layer}.gate_up", layer, pair, xn2, h, g, True,
                                  (mg, mu)))
        g += 1
        entries.append(gemv(by_name[f"L{layer}.down"], h, True))
        g += 1
    xf = norm(layers, 0, "final_norm")
    entries.append(gemv(by_name["head"], xf, True))
    return FusedStack(entries, N)
