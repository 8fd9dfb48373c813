"""GPU parity of the fused gate|up projection with SiLU (decode, M <= 16)
through the C ABI, against the CPU oracle on identical seeded inputs.

The fused matrix is [2F, K]: 16-row tiles of 8 gate rows followed by the
same 8 up rows; y[m, f] = SiLU(g[m, f]) * u[m, f] with each projection's
bias added first ("Lab 5: Gemma4 端到端推理优化", section 基础).  The
output is bf16 from fp32 accumulators, held to the same bar as the linear
itself: rel. Frobenius <= 5e-3 and max|diff| <= 1e-2 max|y| against fp64."""
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


def _run(w4, M, F, K, G, sym, seed, bias=True, cols=None, ws=None):
    packed, scales, zeros = WL.make_random_format(2 * F, K, G, sym, seed)
    x = WL.make_activations(K, M, seed + 1)
    b = (torch.randn(2 * F, generator=torch.Generator().manual_seed(seed + 2)) * 0.5
         if bias else None)
    y = w4.w4a16_linear_swiglu(x.cuda(), packed.cuda(), scales.cuda(),
                               None if zeros is None else zeros.cuda(),
                               None if b is None else b.cuda(), F, K, G, workspace=ws)
    torch.cuda.synchronize()
    yref = O.w4a16_linear_swiglu(x, packed.numpy(), scales.numpy(),
                                 None if zeros is None else zeros.numpy(),
                                 None if b is None else b.numpy(), F, K, G, cols=cols)
    yg = y if cols is None else y[:, torch.as_tensor(cols, device=y.device)]
    assert_close(yg, yref, f"swiglu M{M} F{F} K{K} G{G} sym{sym}")
    return y


@pytest.mark.parametrize("M,F,K,G,sym", [
    (1, 8, 32, 32, True), (3, 24, 100, 32, False), (8, 64, 4096, 128, True),
    (16, 200, 768, 32, False), (5, 136, 1000, 96, True), (1, 512, 16384, 128, True),
    (2, 1000, 3584, 128, False), (16, 768, 2048, 64, True),
])
def test_swiglu_edge_shapes_random_codes(w4, M, F, K, G, sym):
    """Arbitrary codes (0 included, i.e. q = -8), ragged K, odd group sizes,
    several row tiles with a partial last block, split-K shapes, bias."""
    seed = M * 5 + F * 3 + K + G
    y = _run(w4, M, F, K, G, sym, seed)
    y2 = _run(w4, M, F, K, G, sym, seed)
    assert torch.equal(y, y2), "not deterministic"


@pytest.mark.parametrize("rows", ["16", "32", "64", "128"])
@pytest.mark.parametrize("split", ["1", "2"])
@pytest.mark.parametrize("M", [1, 16])
def test_swiglu_pinned_plans(w4, monkeypatch, rows, split, M):
    """Every stage height and both the unsplit and the split-K hand-off."""
    monkeypatch.setenv("W4_GEMV_ROWS", rows)
    monkeypatch.setenv("W4_GEMV_SPLIT", split)
    _run(w4, M, 320, 3072, 128, M == 1, seed=int(rows) + int(split) + M,
         bias=M == 16)


@pytest.mark.parametrize("M", [1, 16])
def test_swiglu_7b_gate_up(w4, M):
    """7B gate|up (F = 18944, K = 3584, G = 128, symmetric): realistic
    weights paired on the GPU side by the binding and on the CPU side by the
    oracle, packed by each side (bit-exact), outputs sampled."""
    F, K, G = 18944, 3584, 128
    lin = WL.Linear("gate_up_fused", M, 2 * F, K, G, True, seed=102, bias=True)
    inp = WL.make_inputs(lin)
    Wg, Wu = inp.W[:F], inp.W[F:]
    fused_gpu = w4.pair_gate_up(Wg.cuda(), Wu.cuda())
    p, s, z = w4.w4_pack_rtn(fused_gpu, G, True)
    op, os_, oz = O.pack_rtn(O.pair_rows(Wg.numpy(), Wu.numpy()), G, True)
    assert np.array_equal(to_np(p), op) and z is None
    assert np.array_equal(to_np(s).view(np.uint32), os_.view(np.uint32))
    bg, bu = inp.bias[:F], inp.bias[F:]
    y = w4.w4a16_linear_swiglu(inp.x.cuda(), p, s, None,
                               w4.pair_gate_up(bg.cuda(), bu.cuda()), F, K, G)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    cols = np.unique(np.concatenate([rng.choice(F, 1024, replace=False), [0, 7, 8, F - 1]]))
    yref = O.w4a16_linear_swiglu(inp.x, op, os_, oz, O.pair_rows(bg.numpy(), bu.numpy()),
                                 F, K, G, cols=cols)
    assert_close(y[:, torch.as_tensor(cols, device=y.device)], yref, f"7B gate_up M{M}")


def test_swiglu_12b_asym_g32(w4):
    """12B-class up projection (F = 15360, K = 3840) asymmetric, G = 32, M = 4."""
    F = 15360
    rng = np.random.default_rng(3)
    cols = np.unique(np.concatenate([rng.choice(F, 768, replace=False), [0, F - 1]]))
    _run(w4, 4, F, 3840, 32, False, seed=303, cols=cols)


def test_swiglu_shape_errors(w4):
    F, K, G = 64, 512, 32
    packed, scales, _ = WL.make_random_format(2 * F, K, G, True, 9)
    x17 = WL.make_activations(K, 17, 10).cuda()
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_linear_swiglu(x17, packed.cuda(), scales.cuda(), None, None, F, K, G)
    assert e.value.code == -8
    # F not a multiple of 8
    p12, s12, _ = WL.make_random_format(24, K, G, True, 11)
    x1 = WL.make_activations(K, 1, 12).cuda()
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_linear_swiglu(x1, p12.cuda(), s12.cuda(), None, None, 12, K, G)
    assert e.value.code == -1
    # M = 0 returns an empty output without a launch
    y0 = w4.w4a16_linear_swiglu(x1[:0], packed.cuda(), scales.cuda(), None, None, F, K, G)
    assert y0.shape == (0, F)
    y0 = w4.w4a16_linear(x1[:0], packed.cuda(), scales.cuda(), None, None, 2 * F, K, G)
    assert y0.shape == (0, 2 * F)
    assert w4.w4_get_device_error() == 0


def test_swiglu_shares_workspace_with_linear(w4, monkeypatch):
    """A split-K fused call and a split-K linear call alternate on one
    zero-filled workspace."""
    monkeypatch.setenv("W4_GEMV_ROWS", "64")
    monkeypatch.setenv("W4_GEMV_SPLIT", "4")
    need = max(w4.w4a16_workspace_bytes(8, 2 * 256, 8192, 128),
               w4.w4a16_workspace_bytes(8, 4096, 8192, 128))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for i in range(2):
        _run(w4, 8, 256, 8192, 128, True, seed=400 + i, ws=ws)
        packed, scales, _ = WL.make_random_format(4096, 8192, 128, True, 410 + i)
        x = WL.make_activations(8192, 8, 420 + i)
        y = w4.w4a16_linear(x.cuda(), packed.cuda(), scales.cuda(), None, None, 4096, 8192,
                            128, workspace=ws)
        torch.cuda.synchronize()
        rows = np.arange(0, 4096, 13)
        yref = O.w4a16_linear(x, packed.numpy()[rows], scales.numpy()[rows], None, None,
                              8192, 128)
        assert_close(y[:, torch.as_tensor(rows, device=y.device)], yref, f"linear {i}")
    assert w4.w4_get_device_error() == 0
