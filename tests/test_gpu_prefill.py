"""GPU parity of the tensor-core prefill path (M > 16) through the C ABI,
against the CPU oracle on identical seeded inputs."""
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


@pytest.mark.parametrize("M,N,K,G,sym", [
    (17, 1, 64, 32, True), (32, 100, 96, 32, False), (64, 129, 200, 64, True),
    (100, 384, 1000, 128, False), (256, 128, 512, 128, True), (257, 256, 256, 32, True),
    (300, 200, 3584, 128, False), (512, 640, 2048, 256, True), (33, 130, 18944, 18944, True),
])
def test_prefill_edge_shapes_random_codes(w4, M, N, K, G, sym):
    """Arbitrary codes (0..15), ragged token, row and column counts, odd
    group sizes, bias."""
    seed = M * 11 + N * 5 + K + G
    packed, scales, zeros = WL.make_random_format(N, K, G, sym, seed)
    x = WL.make_activations(K, M, seed + 1)
    b = torch.randn(N, generator=torch.Generator().manual_seed(seed + 2)) * 0.1
    args = (packed.cuda(), scales.cuda(), None if zeros is None else zeros.cuda(), b.cuda(),
            N, K, G)
    y = w4.w4a16_linear(x.cuda(), *args)
    torch.cuda.synchronize()
    yref = O.w4a16_linear(x, packed.numpy(), scales.numpy(),
                          None if zeros is None else zeros.numpy(), b.numpy(), K, G)
    assert_close(y, yref, f"M{M} N{N} K{K} G{G} sym{sym}")
    y2 = w4.w4a16_linear(x.cuda(), *args)
    assert torch.equal(y, y2), "prefill is not deterministic"


@pytest.mark.parametrize("M", [512, 2048])
@pytest.mark.parametrize("which", [0, 1], ids=["gate_up", "down"])
def test_prefill_workloads(w4, M, which):
    lin = WL.prefill_7b(M)[which]
    inp = WL.make_inputs(lin)
    p, s, z = w4.w4_pack_rtn(inp.W.cuda(), lin.group_size, True)
    y = w4.w4a16_linear(inp.x.cuda(), p, s, z, None, lin.N, lin.K, lin.group_size)
    torch.cuda.synchronize()
    rng = np.random.default_rng(lin.seed)
    rows = np.unique(np.concatenate([rng.choice(lin.N, 384, replace=False), [0, lin.N - 1]]))
    op, os_, _ = O.pack_rtn(inp.W.numpy()[rows], lin.group_size, True)
    assert np.array_equal(to_np(p)[rows], op)
    yref = O.w4a16_linear(inp.x, op, os_, None, None, lin.K, lin.group_size)
    assert_close(y[:, torch.as_tensor(rows, device=y.device)], yref, lin.name)


@pytest.mark.parametrize("pair,bn,split,kb", [
    (1, 256, 1, 1), (1, 256, 2, 1), (1, 256, 3, 1), (0, 256, 1, 1), (0, 256, 2, 1), (0, 128, 1, 1),
    (0, 128, 4, 1), (1, 256, 1, 2), (1, 256, 2, 2), (0, 256, 1, 2), (0, 256, 3, 2),
    (0, 64, 1, 1), (0, 64, 3, 1), (0, 64, 1, 2), (0, 64, 2, 2),
])
@pytest.mark.parametrize("M,N,K,G,sym", [
    (300, 520, 1000, 64, False), (700, 384, 3584, 128, True), (40, 1000, 512, 32, True),
])
def test_prefill_every_variant(w4, monkeypatch, pair, bn, split, kb, M, N, K, G, sym):
    """Each tile variant (CTA pair 256 x 256, one CTA 128 x 256 / 128 x 128,
    64 or 128 columns per stage) and K split, pinned through the planner's
    tuning variables, on ragged shapes: same tolerance, deterministic, no
    device error."""
    if kb == 2 and G % 64:
        pytest.skip("128-column stages need group sizes that are multiples of 64")
    monkeypatch.setenv("W4_GEMM_KB", str(kb))
    monkeypatch.setenv("W4_GEMM_PAIR", str(pair))
    monkeypatch.setenv("W4_GEMM_BN", str(bn))
    monkeypatch.setenv("W4_GEMM_SPLIT", str(split))
    seed = M + 3 * N + 7 * K + G + split
    packed, scales, zeros = WL.make_random_format(N, K, G, sym, seed)
    x = WL.make_activations(K, M, seed + 1)
    b = torch.randn(N, generator=torch.Generator().manual_seed(seed + 2)) * 0.1
    args = (packed.cuda(), scales.cuda(), None if zeros is None else zeros.cuda(), b.cuda(),
            N, K, G)
    y = w4.w4a16_linear(x.cuda(), *args)
    y2 = w4.w4a16_linear(x.cuda(), *args)
    torch.cuda.synchronize()
    assert w4.w4_get_device_error() == 0
    yref = O.w4a16_linear(x, packed.numpy(), scales.numpy(),
                          None if zeros is None else zeros.numpy(), b.numpy(), K, G)
    assert_close(y, yref, f"pair{pair} BN{bn} S{split} KB{kb} M{M} N{N} K{K}")
    assert torch.equal(y, y2), "prefill is not deterministic"


def test_prefill_rejects_k_not_multiple_of_8(w4):
    N, K, G = 64, 100, 32
    packed, scales, _ = WL.make_random_format(N, K, G, True, 1)
    x = WL.make_activations(K, 40, 2).cuda()
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_linear(x, packed.cuda(), scales.cuda(), None, None, N, K, G)
    assert e.value.code == -8


def test_prefill_no_device_error(w4):
    assert w4.w4_get_device_error() == 0
