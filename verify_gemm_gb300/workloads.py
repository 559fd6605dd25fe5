"""Build the synthetic verify-stack workload on the device: draw each
matrix (seeded, see ``inputs``), quantise it with the library's packer and
lay out x and y for all matrices in two contiguous buffers, so that an
end-to-end step can move every input and output with one copy each."""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import FP8Weight, NVFP4Weight, VerifyPlan, fp8_pack, nvfp4_pack
from .inputs import HIDDEN, INTERMEDIATE, LAYERS, VOCAB, Mat, draw_stack_matrix, stack_mats


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


def pack(W: torch.Tensor, fmt: str):
    return nvfp4_pack(W) if fmt == "nvfp4" else fp8_pack(W)


def build_stack(N: int, device="cuda", layers: int = LAYERS, seed: int = 4,
                attn_fmt: str = "nvfp4", down_fmt: str = "fp8", hidden: int = HIDDEN,
                inter: int = INTERMEDIATE, vocab: int = VOCAB, mats=None) -> StackSetup:
    """Quantised layer stack (+ head) with x drawn per matrix (BF16 N(0,1))."""
    if mats is None:
        mats = stack_mats(layers, attn_fmt, down_fmt)
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
