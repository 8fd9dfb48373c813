"""One layer split across ranks, through the kernels (w4a16_linear on row
slices; w4a16_linear_partial + w4a16_partial_finish on group-aligned column
slices), checked against the fp64 oracle of the unsharded layer.

The ranks run one after another on the one GPU; in place of the all-reduce
the test adds their fp32 partials (a harness step, exact up to fp32
rounding).  The CPU test test_shard_multirank.py covers the same split with
real gloo ranks and the oracle; bench.py --shard runs it on N GPUs with
NCCL."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, ensure_built, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


CASES = [  # M, N, K, G, sym, world
    (1, 3584, 18944, 128, True, 2),      # 7B down projection, decode, split-K inside a shard
    (4, 640, 3840, 32, False, 3),        # asymmetric G = 32, ragged split of 120 groups
    (1, 200, 1000, 32, True, 4),         # K not a multiple of G: the last rank holds the tail
    (64, 1024, 4096, 128, True, 2),      # prefill (tensor-core path)
    (300, 512, 8192, 64, False, 2),      # prefill, asymmetric, two token tiles
]


@pytest.mark.parametrize("M,N,K,G,sym,world", CASES)
def test_row_parallel_matches_unsharded(w4, M, N, K, G, sym, world):
    from int4_weight_only_gb300.shard import k_range, pack_shard, row_parallel_linear
    lin = WL.Linear("rowpar", M, N, K, G, sym, seed=M + N + K, bias=True)
    inp = WL.make_inputs(lin)
    op, os_, oz = O.pack_rtn(inp.W.numpy(), G, sym)
    ref = O.w4a16_linear(inp.x, op, os_, oz, inp.bias.numpy(), K, G)
    Wd, xd, bd = inp.W.cuda(), inp.x.cuda(), inp.bias.cuda()
    total = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    for r in range(world):
        sh = pack_shard(Wd, G, sym, "k", world, r, bias=bd)
        k0, k1 = k_range(K, G, world, r)
        assert (sh.lo, sh.hi) == (k0, k1)
        if k1 > k0:
            # the shard's codes and scales are the whole layer's columns / groups
            g0 = k0 // G
            assert np.array_equal(to_np(sh.packed), op[:, k0 // 2:k0 // 2 + sh.packed.shape[1]])
            assert np.array_equal(to_np(sh.scales).view(np.uint32),
                                  os_[:, g0:g0 + sh.scales.shape[1]].view(np.uint32))
            part = w4.w4a16_linear_partial(xd[:, k0:k1].contiguous(), sh.packed, sh.scales,
                                           sh.zeros, N, k1 - k0, G)
            pref = O.w4a16_linear(inp.x[:, k0:k1], op[:, k0 // 2:k0 // 2 + sh.packed.shape[1]],
                                  os_[:, g0:g0 + sh.scales.shape[1]],
                                  None if sym else oz[:, g0:g0 + sh.scales.shape[1]], None,
                                  k1 - k0, G)
            d = to_np(part).astype(np.float64) - pref
            assert np.linalg.norm(d) <= 5e-3 * np.linalg.norm(pref), f"rank {r} partial"
            total += part
    y = w4.w4a16_partial_finish(total, bd)
    assert_close(y, ref, f"row-parallel x{world}")
    # the same through the module's helper on a single rank (no process group)
    sh1 = pack_shard(Wd, G, sym, "k", 1, 0, bias=bd)
    assert_close(row_parallel_linear(xd, sh1), ref, "row-parallel x1")
    assert w4.w4_get_device_error() == 0


@pytest.mark.parametrize("M,N,K,G,sym,world", CASES[:3] + CASES[4:])
def test_column_parallel_matches_unsharded(w4, M, N, K, G, sym, world):
    from int4_weight_only_gb300.shard import column_parallel_linear, column_range, pack_shard
    lin = WL.Linear("colpar", M, N, K, G, sym, seed=N + K, bias=True)
    inp = WL.make_inputs(lin)
    op, os_, oz = O.pack_rtn(inp.W.numpy(), G, sym)
    ref = O.w4a16_linear(inp.x, op, os_, oz, inp.bias.numpy(), K, G)
    Wd, xd, bd = inp.W.cuda(), inp.x.cuda(), inp.bias.cuda()
    parts = []
    for r in range(world):
        sh = pack_shard(Wd, G, sym, "n", world, r, bias=bd)
        n0, n1 = column_range(N, world, r)
        assert np.array_equal(to_np(sh.packed), op[n0:n1])
        parts.append(column_parallel_linear(xd, sh))
    assert_close(torch.cat(parts, dim=1), ref, f"column-parallel x{world}")


def test_partial_finish_rounding(w4):
    """bf16(ysum + bias) with one rounding, both the 4-wide and the scalar
    path (N % 4 != 0), bit for bit against the same fp32 sum rounded on the
    host."""
    g = torch.Generator().manual_seed(3)
    for M, N in ((3, 1024), (5, 1001), (1, 4)):
        ys = torch.randn(M, N, generator=g) * 10
        b = torch.randn(N, generator=g)
        y = w4.w4a16_partial_finish(ys.cuda(), b.cuda())
        want = (ys + b[None, :]).to(torch.bfloat16)
        assert torch.equal(y.cpu().view(torch.int16), want.view(torch.int16))
        y0 = w4.w4a16_partial_finish(ys.cuda(), None)
        assert torch.equal(y0.cpu().view(torch.int16), ys.to(torch.bfloat16).view(torch.int16))
