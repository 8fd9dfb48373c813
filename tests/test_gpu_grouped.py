"""GPU parity of the grouped W4A16 linear (experts of a mixture-of-experts
layer, decode sizes) through the C ABI, against the CPU oracle on identical
seeded inputs ("Yeniden paketlenmiş QAT Gemma 4 26B-A4B, tek bir TPU v6e'de
FP8 işlemenin 1.9 katı verimle sunuluyor": 128 experts, 8 active per token,
int4 with 32-wide groups, a grouped matmul).  Tolerance as for the linear:
rel. Frobenius <= 5e-3 and max|diff| <= 1e-2 max|y| against fp64."""
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


def _case(E, N, K, G, sym, counts, seed, bias=True):
    packed, scales, zeros = WL.make_random_format(E * N, K, G, sym, seed)
    T = int(sum(counts))
    x = WL.make_activations(K, T, seed + 1)
    b = (torch.randn(E * N, generator=torch.Generator().manual_seed(seed + 2)) * 0.1
         if bias else None)
    goff = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return packed, scales, zeros, x, b, goff


def _run(w4, E, N, K, G, sym, counts, seed, gmax, bias=True, cols=None):
    packed, scales, zeros, x, b, goff = _case(E, N, K, G, sym, counts, seed, bias)
    # offsets computed on the device just before the call, as a router would
    cnt = torch.tensor(counts, dtype=torch.int32, device="cuda")
    goff_d = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    goff_d[1:] = torch.cumsum(cnt, 0, dtype=torch.int32)
    y = w4.w4a16_grouped_linear(x.cuda(), goff_d, packed.cuda(), scales.cuda(),
                                None if zeros is None else zeros.cuda(),
                                None if b is None else b.cuda(), E, N, K, G, gmax)
    torch.cuda.synchronize()
    assert w4.w4_get_device_error() == 0
    yref = O.w4a16_grouped_linear(x, goff, packed.numpy(), scales.numpy(),
                                  None if zeros is None else zeros.numpy(),
                                  None if b is None else b.numpy(), E, N, K, G, cols=cols)
    yg = y if cols is None else y[:, torch.as_tensor(cols, device=y.device)]
    assert_close(yg, yref, f"grouped E{E} N{N} K{K} G{G} sym{sym}")
    return y


@pytest.mark.parametrize("E,N,K,G,sym,gmax", [
    (8, 256, 1024, 32, True, 4), (16, 200, 1000, 32, False, 8), (4, 64, 4096, 128, True, 16),
    (32, 384, 768, 64, False, 16), (3, 40, 96, 32, True, 2), (64, 128, 2048, 128, True, 12),
])
def test_grouped_random_routing(w4, E, N, K, G, sym, gmax):
    """Random token counts 0..gmax per group (empty groups included),
    ragged N and K, symmetric and asymmetric, both token tiles (<= 8, <= 16)."""
    rng = np.random.default_rng(E + N + K)
    counts = rng.integers(0, gmax + 1, E).tolist()
    counts[0] = gmax                          # a full group
    counts[-1] = 0                            # an empty last group
    y = _run(w4, E, N, K, G, sym, counts, seed=E * 7 + N, gmax=gmax)
    y2 = _run(w4, E, N, K, G, sym, counts, seed=E * 7 + N, gmax=gmax)
    assert torch.equal(y, y2), "not deterministic"


@pytest.mark.parametrize("batch", [1, 16])
def test_grouped_expert_layer(w4, batch):
    """The expert-layer workload: 128 experts, 8 per token, G = 32, gate|up
    2048 x 2048 and down 2048 x 1024 per expert; sampled output columns."""
    counts = WL.moe_route_counts(batch, seed=batch)
    gmax = max(1, max(counts))
    for lin in WL.moe_decode(batch):
        cols = np.unique(np.concatenate([np.arange(0, lin.N, 61), [lin.N - 1]]))
        _run(w4, WL.MOE_EXPERTS, lin.N, lin.K, lin.group_size, True, counts, seed=lin.seed,
             gmax=gmax, cols=cols)


def test_grouped_single_group_matches_linear(w4):
    """E = 1 with all tokens: the same numbers as w4a16_linear's oracle."""
    _run(w4, 1, 512, 3584, 128, True, [7], seed=3, gmax=7)


@pytest.mark.parametrize("tile", [1, 4, 16])
def test_grouped_tiles_larger_groups(w4, tile):
    """Groups larger than the token tile are taken in several passes: counts
    up to 41 with tiles of 1, 4 and 16 tokens (ragged last tiles)."""
    counts = [41, 0, 16, 17, 3, 0, 33, 1]
    _run(w4, 8, 192, 1024, 64, False, counts, seed=70 + tile, gmax=tile)


def test_grouped_bad_offsets(w4):
    """Offsets past T are skipped (those rows keep their old contents), flag
    W4_ERR_GROUP_TOKENS, and leave the other groups right."""
    E, N, K, G = 4, 64, 256, 32
    counts = [2, 5, 0, 3]
    packed, scales, _, x, b, goff = _case(E, N, K, G, True, counts, 21)
    y = torch.full((10, N), 7.0, dtype=torch.bfloat16, device="cuda")
    yref = O.w4a16_grouped_linear(x, goff, packed.numpy(), scales.numpy(), None, b.numpy(),
                                  E, N, K, G)
    # offsets running past T (the last group claims rows 7..11 of 10)
    bad = torch.tensor([0, 2, 7, 7, 12], dtype=torch.int32, device="cuda")
    w4.w4a16_grouped_linear(x.cuda(), bad, packed.cuda(), scales.cuda(), None, b.cuda(),
                            E, N, K, G, 8, y=y)
    assert w4.w4_get_device_error() == -11
    assert torch.all(y[7:] == 7.0)
    assert_close(y[:7], yref[:7], "valid groups")
    assert w4.w4_get_device_error() == 0
    # overlapping offsets, each group valid on its own: more tiles than T
    # allows; the list keeps what fits and the error is flagged
    lap = torch.tensor([0, 10, 0, 10, 10], dtype=torch.int32, device="cuda")
    w4.w4a16_grouped_linear(x.cuda(), lap, packed.cuda(), scales.cuda(), None, b.cuda(),
                            E, N, K, G, 1, y=y)
    assert w4.w4_get_device_error() == -11
    assert w4.w4_get_device_error() == 0


def test_grouped_empty_and_argument_errors(w4):
    E, N, K, G = 4, 64, 256, 32
    packed, scales, _ = WL.make_random_format(E * N, K, G, True, 1)
    goff = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    x0 = torch.zeros(0, K, dtype=torch.bfloat16, device="cuda")
    y0 = w4.w4a16_grouped_linear(x0, goff, packed.cuda(), scales.cuda(), None, None, E, N, K,
                                 G, 4)
    assert y0.shape == (0, N)
    x = WL.make_activations(K, 4, 2).cuda()
    goff = torch.tensor([0, 4, 4, 4, 4], dtype=torch.int32, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_grouped_linear(x, goff, packed.cuda(), scales.cuda(), None, None, E, N, K, G, 257)
    assert e.value.code == -1
    # every token in group 0, the rest idle
    y = w4.w4a16_grouped_linear(x, goff, packed.cuda(), scales.cuda(), None, None, E, N, K, G, 4)
    yref = O.w4a16_linear(x.cpu(), packed.numpy()[:N], scales.numpy()[:N], None, None, K, G)
    assert_close(y, yref, "one busy group")
    assert w4.w4_get_device_error() == 0
