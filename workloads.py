"""Seeded synthetic inputs for the INT4 weight-only linear layer.

This module only draws random numbers and names shapes.  It holds none of the
layer's arithmetic (no quantisation, packing or matmul), so that both the CPU
oracle and the CUDA path can take their inputs from it without sharing any of
the computation they are compared on.

Workload recipe (the shapes and distributions are the LLM projections the
pages measure; there is no dataset, the Gaussian draws stand in for trained
weights and real activations):

* W  ~ N(0, 0.02^2) fp32, shape [N, K] (out x in).  Optionally a fixed
  fraction of input columns is multiplied by an outlier factor before any
  quantisation ("1% of input columns x20").
* x  ~ N(0, 1) drawn in fp32 and rounded to bf16 (round-to-nearest-even),
  shape [M, K].  Optionally a fraction of positions per token is multiplied
  by an outlier factor before the rounding ("0.5% outliers x50").
* bias ~ N(0, 0.1^2) fp32, shape [N], where a config asks for one.

Every linear gets its own ``torch.Generator('cpu')`` seeded with
``seed``; draws happen in the order W, W-outlier columns, x, x-outlier
positions, bias.

Expert (mixture-of-experts) layers at decode: E = 128 experts with 8 active
per token and 32-wide groups, as on the Gemma 4 26B-A4B TPU page; the expert
matrix sizes are not on the pages and are chosen here (hidden 2048, expert
width 1024: gate|up 2048 x 2048, down 2048 x 1024), symmetric int4.  A batch
of B tokens routes each token to 8 distinct experts drawn uniformly (seeded),
so the grouped call sees T = 8 B rows sorted by expert, most experts holding
0-3 of them.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch


@dataclass(frozen=True)
class Linear:
    """One linear layer instance of a workload."""
    name: str
    M: int
    N: int
    K: int
    group_size: int
    symmetric: bool
    seed: int
    w_outlier_frac: float = 0.0     # fraction of input columns scaled
    w_outlier_scale: float = 20.0
    x_outlier_frac: float = 0.0     # fraction of positions per token scaled
    x_outlier_scale: float = 50.0
    bias: bool = False
    kind: str = "w4a16"             # "w4a16" or "w4a8"


@dataclass
class Inputs:
    W: torch.Tensor                 # fp32 [N, K]
    x: torch.Tensor                 # bf16 [M, K]
    bias: Optional[torch.Tensor]    # fp32 [N] or None


def make_inputs(lin: Linear, M: Optional[int] = None) -> Inputs:
    """Draw W, x and bias for ``lin`` on the CPU (seeded, deterministic).

    ``M`` overrides the token count (the weights do not depend on it)."""
    M = lin.M if M is None else M
    g = torch.Generator(device="cpu")
    g.manual_seed(lin.seed)
    W = torch.randn(lin.N, lin.K, generator=g, dtype=torch.float32) * 0.02
    n_wcols = int(round(lin.w_outlier_frac * lin.K))
    if n_wcols > 0:
        cols = torch.randperm(lin.K, generator=g)[:n_wcols]
        W[:, cols] *= lin.w_outlier_scale
    x = torch.randn(M, lin.K, generator=g, dtype=torch.float32)
    n_xpos = int(round(lin.x_outlier_frac * lin.K))
    if n_xpos > 0:
        for m in range(M):
            pos = torch.randperm(lin.K, generator=g)[:n_xpos]
            x[m, pos] *= lin.x_outlier_scale
    x = x.to(torch.bfloat16)
    bias = None
    if lin.bias:
        bias = torch.randn(lin.N, generator=g, dtype=torch.float32) * 0.1
    return Inputs(W=W, x=x, bias=bias)


def make_activations(K: int, M: int, seed: int, outlier_frac: float = 0.0,
                     outlier_scale: float = 50.0) -> torch.Tensor:
    """Fresh bf16 activations [M, K] ~ N(0,1), independent of any weight."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn(M, K, generator=g, dtype=torch.float32)
    n_xpos = int(round(outlier_frac * K))
    if n_xpos > 0:
        for m in range(M):
            pos = torch.randperm(K, generator=g)[:n_xpos]
            x[m, pos] *= outlier_scale
    return x.to(torch.bfloat16)


# --------------------------------------------------------------------------
# The five workloads.
# --------------------------------------------------------------------------

def tiny() -> List[Linear]:
    """Single tiny linear: M=1, K=512, N=256, G=32, symmetric, seed 0."""
    return [Linear("tiny", 1, 256, 512, 32, True, seed=0)]


# 7B decode shapes: hidden 3584, KV dim 512 (Q + K + V = 3584 + 2*512),
# intermediate 18944 (gate|up fused = 2*18944).
DECODE_7B = [("qkv", 4608, 3584), ("o", 3584, 3584),
             ("gate_up", 37888, 3584), ("down", 3584, 18944)]


def decode_7b(M: int = 1) -> List[Linear]:
    """Decode GEMV set at 7B shapes, symmetric, G=128."""
    return [Linear(f"decode7b_{nm}", M, N, K, 128, True, seed=100 + i)
            for i, (nm, N, K) in enumerate(DECODE_7B)]


def decode_12b(M: int) -> List[Linear]:
    """Batched decode at 12B-class shapes: D=3840, F=15360, asymmetric, G=32,
    1% of W input columns x20."""
    shapes = [("up", 15360, 3840), ("down", 3840, 15360)]
    return [Linear(f"decode12b_{nm}_m{M}", M, N, K, 32, False, seed=200 + i,
                   w_outlier_frac=0.01, w_outlier_scale=20.0)
            for i, (nm, N, K) in enumerate(shapes)]


def prefill_7b(M: int) -> List[Linear]:
    """Prefill GEMM at 7B MLP shapes, symmetric, G=128."""
    shapes = [("gate_up", 37888, 3584), ("down", 3584, 18944)]
    return [Linear(f"prefill7b_{nm}_m{M}", M, N, K, 128, True, seed=300 + i)
            for i, (nm, N, K) in enumerate(shapes)]


def w4a8_7b() -> List[Linear]:
    """W4A8 integer path, M=1: per-row INT4 weights (group = padded K),
    per-token dynamic INT8 activations with 0.5% outliers x50, bias
    ~N(0, 0.1^2).  The third linear is the padding case K=3580 -> 3584."""
    out = []
    for i, (nm, N, K, Kp) in enumerate([("up", 18944, 3584, 3584),
                                        ("down", 3584, 18944, 18944),
                                        ("pad", 18944, 3580, 3584)]):
        out.append(Linear(f"w4a8_{nm}", 1, N, K, Kp, True, seed=400 + i,
                          x_outlier_frac=0.005, x_outlier_scale=50.0,
                          bias=True, kind="w4a8"))
    return out


def padding_w4a16() -> List[Linear]:
    """The K=3580 shape through the W4A16 path with G=128 (Kp=3584)."""
    return [Linear("pad_w4a16", 1, 18944, 3580, 128, True, seed=500,
                   bias=True)]


WORKLOADS = {
    "tiny": tiny,
    "decode_7b": decode_7b,
    "decode_12b": decode_12b,
    "prefill_7b": prefill_7b,
    "w4a8_7b": w4a8_7b,
}


def make_random_format(N: int, K: int, group_size: int, symmetric: bool, seed: int):
    """Arbitrary valid packed weights (every nibble value 0..15 occurs,
    including the code 0 that round-to-nearest with s = max/7 never emits),
    positive fp32 scales and, for asymmetric groups, zero points in
    [0, 15].  Returns (packed uint8 [N, Kp/2], scales fp32 [N, Ng],
    zeros uint8 [N, Ng] or None) as CPU tensors."""
    Kp = -(-K // group_size) * group_size
    Ng = Kp // group_size
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    packed = torch.randint(0, 256, (N, Kp // 2), generator=g, dtype=torch.int64).to(torch.uint8)
    scales = (torch.rand(N, Ng, generator=g, dtype=torch.float32) * 0.01 + 1e-4)
    zeros = None
    if not symmetric:
        zeros = torch.randint(0, 16, (N, Ng), generator=g, dtype=torch.int64).to(torch.uint8)
    return packed, scales, zeros


# --------------------------------------------------------------------------
# Expert layers (grouped decode).
# --------------------------------------------------------------------------

MOE_EXPERTS, MOE_TOPK, MOE_HIDDEN, MOE_WIDTH, MOE_GROUP = 128, 8, 2048, 1024, 32


def moe_route_counts(batch: int, experts: int = MOE_EXPERTS, topk: int = MOE_TOPK,
                     seed: int = 0) -> List[int]:
    """Tokens per expert when each of `batch` tokens picks `topk` distinct
    experts uniformly at random (seeded)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    counts = [0] * experts
    for _ in range(batch):
        for e in torch.randperm(experts, generator=g)[:topk].tolist():
            counts[e] += 1
    return counts


def moe_decode(batch: int = 16) -> List[Linear]:
    """The two projections of an expert layer, one matrix per expert
    (N x K per expert; the grouped call stacks the 128 of them)."""
    return [Linear(f"moe_gate_up_b{batch}", batch * MOE_TOPK, 2 * MOE_WIDTH, MOE_HIDDEN,
                   MOE_GROUP, True, seed=600),
            Linear(f"moe_down_b{batch}", batch * MOE_TOPK, MOE_HIDDEN, MOE_WIDTH,
                   MOE_GROUP, True, seed=601)]
