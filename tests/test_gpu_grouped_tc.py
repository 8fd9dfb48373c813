"""GPU parity of the grouped W4A16 linear for groups of many tokens (the
prefill side of a mixture-of-experts layer) on the tensor-core kernel:
w4a16_grouped_linear with tile_tokens 17..256 runs token tiles of 64 or 256
on tcgen05, each tile dequantizing its group's weights once ("Yeniden
paketlenmiş QAT Gemma 4 26B-A4B, tek bir TPU v6e'de FP8 işlemenin 1.9 katı
verimle sunuluyor", section "vLLM'in TPU backend'inde değişen ne oldu": the
grouped matmul over the experts).  Against the fp64 oracle on identical
seeded inputs, tolerance as for the linear (rel. Frobenius <= 5e-3,
max|diff| <= 1e-2 max|y|): groups of 0, 1, 17, 200 and 1000 tokens, empty
groups, ragged row blocks, both stage widths, offsets computed on the
device, bad offsets flagged with their rows left untouched, and the
128-expert layer at batch 512 x top-8."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _run(w4, E, N, K, G, sym, counts, seed, tile, bias=True, cols=None):
    packed, scales, zeros = WL.make_random_format(E * N, K, G, sym, seed)
    T = int(sum(counts))
    x = WL.make_activations(K, T, seed + 1)
    b = (torch.randn(E * N, generator=torch.Generator().manual_seed(seed + 2)) * 0.1
         if bias else None)
    goff = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    cnt = torch.tensor(counts, dtype=torch.int32, device="cuda")
    goff_d = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    goff_d[1:] = torch.cumsum(cnt, 0, dtype=torch.int32)      # as a router kernel would
    args = (x.cuda(), goff_d, packed.cuda(), scales.cuda(),
            None if zeros is None else zeros.cuda(), None if b is None else b.cuda(),
            E, N, K, G)
    y = w4.w4a16_grouped_linear(*args, tile)
    torch.cuda.synchronize()
    assert w4.w4_get_device_error() == 0
    yref = O.w4a16_grouped_linear(x, goff, packed.numpy(), scales.numpy(),
                                  None if zeros is None else zeros.numpy(),
                                  None if b is None else b.numpy(), E, N, K, G, cols=cols)
    yg = y if cols is None else y[:, torch.as_tensor(cols, device=y.device)]
    assert_close(yg, yref, f"grouped tc E{E} N{N} K{K} G{G} sym{sym} tile{tile}")
    y2 = w4.w4a16_grouped_linear(*args, tile)
    assert torch.equal(y, y2), "not deterministic"
    return y, args


@pytest.mark.parametrize("tile", [64, 256])
@pytest.mark.parametrize("G,sym", [(64, True), (32, False), (128, True)])
def test_grouped_tc_group_sizes(w4, tile, G, sym):
    """Groups of 0, 1, 17, 200 and 1000 tokens (and more empty ones), N with
    a partial last row block; 128-column stages where G allows (64, 128),
    64-column stages for G = 32."""
    counts = [0, 1, 17, 0, 200, 1000, 0, 33]
    _run(w4, len(counts), 320, 512, G, sym, counts, seed=G + tile, tile=tile)


def test_grouped_tc_matches_decode_path(w4):
    """The same routing through the decode kernel (tiles of 16) and the
    tensor-core kernel agree within the tolerance of each against fp64."""
    counts = [5, 40, 0, 70, 3]
    y_tc, args = _run(w4, len(counts), 256, 1024, 128, True, counts, seed=3, tile=64)
    y_dec = w4.w4a16_grouped_linear(*args, 16)
    torch.cuda.synchronize()
    d = (y_tc.float() - y_dec.float()).norm() / y_dec.float().norm()
    assert float(d) < 5e-3


def test_grouped_tc_expert_layer_prefill(w4):
    """128 experts, 8 of them per token, batch 512 (4096 routed rows):
    gate|up 2048 x 2048, G = 32, symmetric; 96 sampled output columns."""
    B = 512
    counts = WL.moe_route_counts(B, seed=B)
    rng = np.random.default_rng(0)
    cols = np.sort(rng.choice(2048, 96, replace=False))
    _run(w4, WL.MOE_EXPERTS, 2048, 2048, 32, True, counts, seed=11, tile=64, bias=False,
         cols=cols)


def test_grouped_tc_bad_offsets(w4):
    """Offsets past T leave that group out (its rows keep their contents),
    raise W4_ERR_GROUP_TOKENS, and keep the other groups right."""
    E, N, K, G = 4, 128, 256, 64
    counts = [30, 50, 0, 20]
    packed, scales, _ = WL.make_random_format(E * N, K, G, True, 21)
    T = sum(counts)
    x = WL.make_activations(K, T, 22)
    goff = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    yref = O.w4a16_grouped_linear(x, goff, packed.numpy(), scales.numpy(), None, None, E, N, K, G)
    bad = torch.tensor([0, 30, 80, 80, 130], dtype=torch.int32, device="cuda")   # last past T=100
    y = torch.full((T, N), 7.0, dtype=torch.bfloat16, device="cuda")
    w4.w4a16_grouped_linear(x.cuda(), bad, packed.cuda(), scales.cuda(), None, None, E, N, K, G,
                            64, y=y)
    assert w4.w4_get_device_error() == -11
    assert torch.all(y[80:] == 7.0)
    assert_close(y[:80], yref[:80], "valid groups")
    assert w4.w4_get_device_error() == 0
