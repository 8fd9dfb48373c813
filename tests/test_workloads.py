"""The seeded input recipe (no GPU): routing of the expert layer, and the
determinism every parity test relies on."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402


def test_moe_routing_counts():
    for batch in (1, 4, 16):
        counts = WL.moe_route_counts(batch, seed=batch)
        assert len(counts) == WL.MOE_EXPERTS
        assert sum(counts) == batch * WL.MOE_TOPK           # 8 experts per token
        assert max(counts) <= batch                          # distinct experts per token
        assert counts == WL.moe_route_counts(batch, seed=batch)
    assert WL.moe_route_counts(16, seed=1) != WL.moe_route_counts(16, seed=2)


def test_inputs_are_seeded():
    lin = WL.tiny()[0]
    a, b = WL.make_inputs(lin), WL.make_inputs(lin)
    assert torch.equal(a.W, b.W) and torch.equal(a.x, b.x)
    assert a.x.dtype == torch.bfloat16 and a.W.dtype == torch.float32
    p1 = WL.make_random_format(64, 100, 32, False, 3)
    p2 = WL.make_random_format(64, 100, 32, False, 3)
    assert all(torch.equal(u, v) for u, v in zip(p1, p2))
    assert p1[0].shape == (64, 64) and p1[1].shape == (64, 4) and p1[2].shape == (64, 4)
    assert int(p1[2].max()) <= 15 and float(p1[1].min()) > 0


def test_expert_layer_shapes():
    up, down = WL.moe_decode(16)
    assert (up.N, up.K) == (2 * WL.MOE_WIDTH, WL.MOE_HIDDEN)
    assert (down.N, down.K) == (WL.MOE_HIDDEN, WL.MOE_WIDTH)
    assert up.M == 16 * WL.MOE_TOPK and up.group_size == WL.MOE_GROUP == 32
