"""Sharding one layer across ranks, on the CPU: the host logic of
int4_weight_only_gb300.shard and the decomposition itself, with two gloo
ranks on 127.0.0.1 that each compute their shard with the oracle.

* column-parallel: the gathered row slices equal the unsharded oracle output;
* row-parallel: the all-reduced fp64 partials plus the bias equal it too;
* packing a rank's slice of W gives exactly its rows / groups of the whole
  layer's packing (round-to-nearest is per row and group), which is what lets
  each rank pack its own shard.
No GPU and no library call: the kernels' side of the same split is the
-m gpu test in test_gpu_shard.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from int4_weight_only_gb300.shard import column_range, k_range


def test_column_range_covers_rows_once():
    for N in (0, 1, 7, 3584, 37888):
        for world in (1, 2, 3, 8):
            rs = [column_range(N, world, r) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == N
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
            sizes = [hi - lo for lo, hi in rs]
            assert max(sizes) - min(sizes) <= 1


def test_k_range_is_group_aligned():
    for K, G in ((3584, 128), (18944, 128), (3580, 128), (100, 32), (15360, 32), (64, 64)):
        for world in (1, 2, 3, 4, 8):
            rs = [k_range(K, G, world, r) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == K
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
            assert all(lo % G == 0 for lo, hi in rs if hi > lo)
            # every slice that does not end at K is a whole number of groups
            assert all((hi - lo) % G == 0 for lo, hi in rs if hi < K)


def test_ranges_reject_bad_arguments():
    with pytest.raises(ValueError):
        column_range(10, 2, 2)
    with pytest.raises(ValueError):
        k_range(10, 0, 2, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    import workloads as WL
    lin = WL.Linear("shard", 3, 96, 1000, 32, False, seed=77, w_outlier_frac=0.01, bias=True)
    return WL.make_inputs(lin), lin


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        inp, lin = _case()
        W = inp.W.numpy()
        b = inp.bias.numpy()
        G, sym = lin.group_size, lin.symmetric
        full_p, full_s, full_z = O.pack_rtn(W, G, sym)
        # column-parallel: this rank's rows
        n0, n1 = column_range(lin.N, world, rank)
        p, s, z = O.pack_rtn(W[n0:n1], G, sym)
        same_rows = (np.array_equal(p, full_p[n0:n1]) and np.array_equal(s, full_s[n0:n1])
                     and np.array_equal(z, full_z[n0:n1]))
        y_loc = O.w4a16_linear(inp.x, p, s, z, b[n0:n1], lin.K, G)
        parts = [torch.zeros(lin.M, hi - lo, dtype=torch.float64)
                 for lo, hi in (column_range(lin.N, world, r) for r in range(world))]
        torch.distributed.all_gather(parts, torch.from_numpy(np.ascontiguousarray(y_loc)))
        y_col = torch.cat(parts, dim=1).numpy()
        # row-parallel: this rank's group-aligned columns, partial without bias
        k0, k1 = k_range(lin.K, G, world, rank)
        pk, sk, zk = O.pack_rtn(W[:, k0:k1], G, sym)
        g0, g1 = k0 // G, -(-k1 // G)
        same_groups = (np.array_equal(pk, full_p[:, k0 // 2:k0 // 2 + pk.shape[1]])
                       and np.array_equal(sk, full_s[:, g0:g1]) and np.array_equal(zk, full_z[:, g0:g1]))
        xk = inp.x[:, k0:k1]
        part = O.w4a16_linear(xk, pk, sk, zk, None, k1 - k0, G)
        t = torch.from_numpy(np.ascontiguousarray(part))
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
        y_row = t.numpy() + b[None, :]
        q.put((rank, same_rows, same_groups, y_col, y_row))
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_ranks_reproduce_the_unsharded_layer(world):
    import oracle as O
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    mp.start_processes(_worker, args=(world, _free_port(), q), nprocs=world, join=True,
                       start_method="spawn")
    got = sorted((q.get() for _ in range(world)), key=lambda g: g[0])
    inp, lin = _case()
    p, s, z = O.pack_rtn(inp.W.numpy(), lin.group_size, lin.symmetric)
    ref = O.w4a16_linear(inp.x, p, s, z, inp.bias.numpy(), lin.K, lin.group_size)
    for rank, same_rows, same_groups, y_col, y_row in got:
        assert same_rows, f"rank {rank}: row shard packs differently"
        assert same_groups, f"rank {rank}: column shard packs differently"
        np.testing.assert_allclose(y_col, ref, rtol=1e-12, atol=1e-12)
        # the partials are added in a different order: fp64 rounding only
        np.testing.assert_allclose(y_row, ref, rtol=1e-10, atol=1e-12)
