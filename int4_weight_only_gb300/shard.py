"""One INT4 weight-only linear layer split across the GPUs of a process group.

The layer y = x W_hat^T + b shards two ways, one process per GPU:

* column-parallel (split of the N output rows): rank r owns rows
  [n0, n1) of the packed codes, scales, zero points and bias, computes
  y[:, n0:n1] with w4a16_linear and exchanges nothing (the next layer can
  consume the slice, or the caller gathers it);
* row-parallel (split of the K input columns into group-aligned slices):
  rank r owns columns [k0, k1), k0 and k1 multiples of group_size (the last
  rank also the ragged end), and the matching slice of the activations;
  each rank computes its fp32 partial sum with w4a16_linear_partial, one
  all-reduce adds the partials, and w4a16_partial_finish adds the bias and
  rounds to bf16 once.

Because round-to-nearest quantization is per (row, group), packing a
rank's slice of W gives exactly the rows or groups of the whole layer's
packing, so a shard can be packed on its own GPU from its own slice.  The
pages define the layer and its quantization ("Lab 5: Gemma4 端到端推理优化",
section "INT4 线性量化"); the split is the usual tensor-parallel one.

Only the host logic lives here (ranges, which slice goes where, the one
collective); every arithmetic step runs in libw4's kernels or in the
process group's all-reduce.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Tuple

import torch

from . import _lib as L


def column_range(N: int, world: int, rank: int) -> Tuple[int, int]:
    """Output rows [n0, n1) of `rank` when N rows are split over `world`
    ranks as evenly as possible (the first N % world ranks take one more)."""
    if world < 1 or not 0 <= rank < world or N < 0:
        raise ValueError("need 0 <= rank < world and N >= 0")
    q, r = divmod(N, world)
    n0 = rank * q + min(rank, r)
    return n0, n0 + q + (1 if rank < r else 0)


def k_range(K: int, group_size: int, world: int, rank: int) -> Tuple[int, int]:
    """Input columns [k0, k1) of `rank`: the ceil(K / group_size) groups are
    split as evenly as possible into contiguous runs, so k0 is a multiple of
    group_size; the last rank's slice ends at K (the padded tail belongs to
    it).  A rank can be left with no columns when there are fewer groups than
    ranks."""
    if group_size <= 0:
        raise ValueError("group_size must be positive")
    ng = -(-K // group_size)
    g0, g1 = column_range(ng, world, rank)
    return min(g0 * group_size, K), min(g1 * group_size, K)


@dataclass
class Shard:
    """This rank's part of one layer, packed on its device."""
    mode: str                           # "n" (column-parallel) or "k" (row-parallel)
    N: int                              # rows of the whole layer
    K: int                              # columns of the whole layer
    group_size: int
    lo: int                             # first owned row (n) or column (k)
    hi: int                             # one past the last
    packed: torch.Tensor
    scales: torch.Tensor
    zeros: Optional[torch.Tensor]
    bias: Optional[torch.Tensor]        # n: the owned rows' bias; k: the whole bias

    @property
    def width(self) -> int:
        return self.hi - self.lo


def pack_shard(W: torch.Tensor, group_size: int, symmetric: bool, mode: str, world: int,
               rank: int, bias: Optional[torch.Tensor] = None) -> Shard:
    """Pack rank `rank`'s slice of the fp32 weights W [N, K] (on this rank's
    device) with w4_pack_rtn.  mode "n": rows column_range(N); mode "k":
    columns k_range(K, group_size)."""
    N, K = W.shape
    if mode == "n":
        lo, hi = column_range(N, world, rank)
        Ws = W[lo:hi].contiguous()
        b = None if bias is None else bias[lo:hi].contiguous()
    elif mode == "k":
        lo, hi = k_range(K, group_size, world, rank)
        Ws = W[:, lo:hi].contiguous()
        b = bias
    else:
        raise ValueError("mode must be 'n' or 'k'")
    if Ws.numel() == 0:
        dev = W.device
        return Shard(mode, N, K, group_size, lo, hi, torch.empty(0, 0, dtype=torch.uint8, device=dev),
                     torch.empty(0, 0, device=dev), None, b)
    p, s, z = L.w4_pack_rtn(Ws, group_size, symmetric)
    return Shard(mode, N, K, group_size, lo, hi, p, s, z, b)


def column_parallel_linear(x: torch.Tensor, sh: Shard, y=None) -> torch.Tensor:
    """y[:, lo:hi] of the layer for this rank's rows: w4a16_linear on the
    shard; no exchange."""
    if sh.mode != "n":
        raise ValueError("not a column-parallel shard")
    M = x.shape[0]
    if sh.width == 0:
        return torch.empty(M, 0, dtype=torch.bfloat16, device=x.device)
    return L.w4a16_linear(x, sh.packed, sh.scales, sh.zeros, sh.bias, sh.width, sh.K,
                          sh.group_size, y=y)


def row_parallel_linear(x_local: torch.Tensor, sh: Shard, group=None, y=None,
                        y32=None) -> torch.Tensor:
    """The whole layer's y [M, N] on every rank from this rank's activation
    slice x_local [M, hi - lo]: fp32 partial (w4a16_linear_partial), one
    all-reduce (sum) over `group` when it has more than one rank, then bias
    and one bf16 rounding (w4a16_partial_finish)."""
    if sh.mode != "k":
        raise ValueError("not a row-parallel shard")
    M = x_local.shape[0]
    if y32 is None:
        y32 = torch.empty(M, sh.N, dtype=torch.float32, device=x_local.device)
    if sh.width > 0:
        L.w4a16_linear_partial(x_local, sh.packed, sh.scales, sh.zeros, sh.N, sh.width,
                               sh.group_size, y32=y32)
    else:
        y32.zero_()
    if torch.distributed.is_available() and torch.distributed.is_initialized() and \
            torch.distributed.get_world_size(group) > 1:
        torch.distributed.all_reduce(y32, op=torch.distributed.ReduceOp.SUM, group=group)
    return L.w4a16_partial_finish(y32, sh.bias, y=y)
