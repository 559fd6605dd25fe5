"""Seeded synthetic inputs for the verify GEMV workloads.

This module holds no arithmetic of the method (no quantisation, no decode,
no product): it only draws seeded FP32 weights and BF16 activations with the
shapes and distributions of the workloads, so that the CUDA path and the CPU
oracle see the same inputs.  The workloads stand in for the Qwen3.8-27B
checkpoint shapes that the mtp7-device-confidence engine card (crit-hub,
Model section) runs: hidden 5120, intermediate 17408, vocabulary 151936,
64 layers, verify width 2-8 (card, Design table, Decode row).

Recipe:
  * W = 0.02 * randn (FP32), x = randn (FP32) rounded to BF16 (RNE).
  * One ``torch.Generator`` per workload seeded with the workload's seed;
    draw order: every weight matrix in listed order, then x.
  * Outliers: after drawing x, ``randperm(K)[:8]`` picks 8 channels whose
    columns are multiplied by 20 before the BF16 rounding.
  * The 64-layer stack is too large to hold in FP32 at once: each matrix is
    drawn from its own generator seeded with seed*1000003 + layer*16 + idx,
    and each matrix gets its own x from seed*1000003 + layer*16 + 8 + idx.
  * The draft step (one row-scaled FP8 layer + the NVFP4 head, N = 1) is
    drawn the same way from seed 5, a seed of its own.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

HIDDEN = 5120
INTERMEDIATE = 17408
VOCAB = 151936
LAYERS = 64
W_STD = 0.02


@dataclass(frozen=True)
class Mat:
    """One weight matrix of a workload: name, format ('nvfp4'|'fp8'), M, K,
    dependency group (matrices of one group may run concurrently)."""

    name: str
    fmt: str
    M: int
    K: int
    group: int = 0
    layer: int = -1
    idx: int = 0


@dataclass
class Workload:
    key: str
    title: str
    seed: int
    mats: list
    Ns: tuple
    outliers: int = 0


def stack_mats(layers: int = LAYERS, attn_fmt: str = "nvfp4", down_fmt: str = "fp8"):
    """Matrices of the layer stack in verify order, with dependency groups:
    per layer {q,k,v} -> {o} -> {gate, up} -> {down}; then the head."""
    mats = []
    g = 0
    for layer in range(layers):
        for i, nm in enumerate(("q", "k", "v")):
            mats.append(Mat(f"L{layer}.{nm}", attn_fmt, HIDDEN, HIDDEN, g, layer, i))
        g += 1
        mats.append(Mat(f"L{layer}.o", attn_fmt, HIDDEN, HIDDEN, g, layer, 3))
        g += 1
        mats.append(Mat(f"L{layer}.gate", "nvfp4", INTERMEDIATE, HIDDEN, g, layer, 4))
        mats.append(Mat(f"L{layer}.up", "nvfp4", INTERMEDIATE, HIDDEN, g, layer, 5))
        g += 1
        mats.append(Mat(f"L{layer}.down", down_fmt, HIDDEN, INTERMEDIATE, g, layer, 6))
        g += 1
    mats.append(Mat("head", "nvfp4", VOCAB, HIDDEN, g, layers, 0))
    return mats


DRAFT_SEED = 5


def draft_mats(hidden: int = HIDDEN, inter: int = INTERMEDIATE, vocab: int = VOCAB):
    """Matrices of one draft step (engine card, Model section: the drafting
    layer re-encoded as row-scaled FP8, the output head as NVFP4; Measured
    section: each draft step adds about 0.8 ms).  One layer's q, k, v, o,
    gate, up and down, all row-scaled FP8, then the NVFP4 head; the same
    groups as a stack layer.  Drawn like the stack (derived seeds, layer 0
    and 1 for the head) from DRAFT_SEED."""
    mats = [Mat(f"D.{nm}", "fp8", hidden, hidden, 0, 0, i) for i, nm in enumerate("qkv")]
    mats.append(Mat("D.o", "fp8", hidden, hidden, 1, 0, 3))
    mats.append(Mat("D.gate", "fp8", inter, hidden, 2, 0, 4))
    mats.append(Mat("D.up", "fp8", inter, hidden, 2, 0, 5))
    mats.append(Mat("D.down", "fp8", hidden, inter, 3, 0, 6))
    mats.append(Mat("head", "nvfp4", vocab, hidden, 4, 1, 0))
    return mats


WORKLOADS = {
    "tiny": Workload("tiny", "tiny NVFP4 GEMV 256x512", 0,
                     [Mat("w", "nvfp4", 256, 512)], (1,)),
    "proj": Workload("proj", "single projection NVFP4 5120x5120, outlier x", 1,
                     [Mat("w", "nvfp4", HIDDEN, HIDDEN)], (1,), outliers=8),
    "gateup": Workload("gateup", "fused gate+up NVFP4 34816x5120 (two halves, own scales)",
                       2, [Mat("gate", "nvfp4", INTERMEDIATE, HIDDEN),
                           Mat("up", "nvfp4", INTERMEDIATE, HIDDEN)], (1, 2, 4, 8)),
    "down_head": Workload("down_head",
                          "row-scaled FP8 down 5120x17408 + NVFP4 head 151936x5120", 3,
                          [Mat("down", "fp8", HIDDEN, INTERMEDIATE),
                           Mat("head", "nvfp4", VOCAB, HIDDEN, 1)], (1, 8)),
    "stack": Workload("stack", "64-layer verify stack + NVFP4 head", 4, stack_mats(),
                      (8, 1, 2, 4)),
}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def stack_seed(seed: int, layer: int, idx: int) -> int:
    """Derived seed of matrix ``idx`` of ``layer`` in the layer stack."""
    return seed * 1000003 + layer * 16 + idx


def draw_weight(gen: torch.Generator, M: int, K: int, device="cpu") -> torch.Tensor:
    """FP32 [M, K] ~ N(0, 0.02^2)."""
    w = torch.randn((M, K), generator=gen, dtype=torch.float32, device=device)
    return w.mul_(W_STD)


def draw_x(gen: torch.Generator, N: int, K: int, outliers: int = 0,
           device="cpu") -> torch.Tensor:
    """BF16 [N, K] ~ N(0, 1) with ``outliers`` channels scaled by 20."""
    x = torch.randn((N, K), generator=gen, dtype=torch.float32, device=device)
    if outliers:
        idx = torch.randperm(K, generator=gen, device=device)[:outliers]
        x[:, idx] *= 20.0
    return x.to(torch.bfloat16)


def draw_norm_inputs(seed: int, layer: int, which: int, N: int, K: int, device="cpu"):
    """x [N, K] BF16 ~ N(0, 1) and gamma [K] BF16 ~ 1 + 0.1 N(0, 1) of one
    RMS normalisation of a fused layer (which: 0 before q/k/v, 1 before the
    MLP), from the derived seeds of indices 12 + which and 14 + which."""
    gx = generator(stack_seed(seed, layer, 12 + which), device)
    x = torch.randn((N, K), generator=gx, dtype=torch.float32, device=device).to(torch.bfloat16)
    gg = generator(stack_seed(seed, layer, 14 + which), device)
    gamma = (1.0 + 0.1 * torch.randn((K,), generator=gg, dtype=torch.float32, device=device))
    return x, gamma.to(torch.bfloat16)


def bf16_bits(x: torch.Tensor):
    """BF16 tensor -> numpy uint16 bit patterns (host copy)."""
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def draw_workload(key: str, N: int, device="cpu"):
    """Weights (FP32) and x (BF16) of a single-pass workload in draw order.
    Returns ([W per matrix], [x per distinct K], ...) as (Ws, xs) where xs
    maps K -> x[N, K]."""
    wl = WORKLOADS[key]
    gen = generator(wl.seed, device)
    Ws = [draw_weight(gen, m.M, m.K, device) for m in wl.mats]
    xs = {}
    for m in wl.mats:
        if m.K not in xs:
            xs[m.K] = draw_x(gen, N, m.K, wl.outliers, device)
    return Ws, xs


def draw_stack_matrix(mat: Mat, N: int, seed: int = 4, device="cpu"):
    """FP32 weight and BF16 x of one matrix of the layer stack."""
    gw = generator(stack_seed(seed, mat.layer, mat.idx), device)
    W = draw_weight(gw, mat.M, mat.K, device)
    gx = generator(stack_seed(seed, mat.layer, 8 + mat.idx), device)
    x = draw_x(gx, N, mat.K, 0, device)
    return W, x
