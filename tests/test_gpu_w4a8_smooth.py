"""GPU parity of group-wise W4A8 and of SmoothQuant smoothing through the C
ABI against the CPU oracle ("【infra之路】12-投机解码、量化与推理引擎对比",
sections 2.2 and 2.4; "LLM 模型壓縮與推理加速實踐-陳磊.pdf", W8A8 slides).

Bit-exact: INT8 activations and their scales, smoothed or not (the factors
are seeded inputs there).  Within fp32 accuracy: the smoothing factors
(powf on the device, fp64 in the oracle).  Float tolerance (rel. Frobenius
5e-3, max|diff| 1e-2 max|y|): group-wise outputs and the smoothed layer."""
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


def _grouped(w4, M, N, K, G, seed, rows=None):
    lin = WL.Linear("w4a8g", M, N, K, G, True, seed=seed, bias=True, x_outlier_frac=0.005,
                    kind="w4a8")
    inp = WL.make_inputs(lin)
    p, s, _ = w4.w4_pack_rtn(inp.W.cuda(), G, True)
    op, os_, _ = O.pack_rtn(inp.W.numpy(), G, True)
    assert np.array_equal(to_np(p), op)
    qx, sx = w4.w4a8_quantize_act(inp.x.cuda(), G)
    oq, osx = O.w4a8_quantize_act(inp.x, O.padded_k(K, G))
    assert np.array_equal(to_np(qx), oq)
    y, acc = w4.w4a8_linear(qx, sx, p, s, inp.bias.cuda(), N, K, G)
    torch.cuda.synchronize()
    assert acc is None
    _, oy = O.w4a8_linear_grouped(oq, osx, op, os_, G, bias=inp.bias.numpy(), rows=rows)
    yg = y if rows is None else y[:, torch.as_tensor(rows, device=y.device)]
    assert_close(yg, oy, f"w4a8 grouped M{M} N{N} K{K} G{G}")
    return y


@pytest.mark.parametrize("M,N,K,G", [
    (1, 4096, 3584, 128), (4, 1000, 3580, 128), (16, 512, 2048, 32), (8, 300, 1024, 64),
    (2, 256, 4096, 256), (3, 640, 6144, 512), (16, 129, 4096, 128), (1, 3584, 18944, 128),
    (5, 200, 96, 32),
])
def test_w4a8_groupwise(w4, M, N, K, G):
    rows = None if N <= 4096 else np.arange(0, N, 7)
    y = _grouped(w4, M, N, K, G, seed=M + N + K + G, rows=rows)
    y2 = _grouped(w4, M, N, K, G, seed=M + N + K + G, rows=rows)
    assert torch.equal(y, y2), "not deterministic"


@pytest.mark.parametrize("rows,split", [("16", "1"), ("64", "3"), ("128", "8")])
def test_w4a8_groupwise_pinned_plans(w4, monkeypatch, rows, split):
    """Unsplit and split-K plans (float partials added in split order)."""
    monkeypatch.setenv("W4_GEMV_ROWS", rows)
    monkeypatch.setenv("W4_GEMV_SPLIT", split)
    _grouped(w4, 4, 640, 8192, 128, seed=int(rows) * 10 + int(split))


def test_w4a8_groupwise_errors(w4):
    K, N = 192, 64
    qx = torch.zeros(1, K, dtype=torch.int8, device="cuda")
    sx = torch.ones(1, device="cuda")
    p = torch.zeros(N, K // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.w4a8_linear(qx, sx, p, torch.ones(N, 2, device="cuda"), None, N, K, 96)
    assert e.value.code == -4
    with pytest.raises(w4.W4Error) as e:
        w4.w4a8_linear(qx, sx, p, torch.ones(N, 6, device="cuda"), None, N, K, 32, want_acc=True)
    assert e.value.code == -1


@pytest.mark.parametrize("M,K,G", [(1, 3584, 3584), (3, 3580, 3584), (2, 1001, 1024),
                                   (4, 18944, 18944), (2, 40000, 40000), (16, 512, 128)])
def test_smoothed_act_quant_bit_exact(w4, M, K, G):
    """Factors drawn as seeded inputs, spanning 2^-6 .. 2^6 with arbitrary
    mantissas; every load path of the quantizer."""
    x = WL.make_activations(K, M, seed=K + M, outlier_frac=0.01)
    g = torch.Generator().manual_seed(K)
    inv_s = torch.exp2((torch.rand(K, generator=g) - 0.5) * 12.0).float()
    qx, sx = w4.w4a8_quantize_act_smooth(x.cuda(), inv_s.cuda(), G)
    oq, osx = O.w4a8_quantize_act(x, O.padded_k(K, G), inv_s=inv_s.numpy())
    assert np.array_equal(to_np(sx).view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(to_np(qx), oq)


def _outlier_layer(T, K, N, seed):
    """Calibration and test activations with 1% outlier channels x50 (the same
    channels in both), weights N(0, 0.02^2)."""
    g = torch.Generator().manual_seed(seed)
    hot = torch.randperm(K, generator=g)[: max(1, K // 100)]
    def acts(rows):
        x = torch.randn(rows, K, generator=g)
        x[:, hot] *= 50.0
        return x.to(torch.bfloat16)
    W = torch.randn(N, K, generator=g) * 0.02
    return acts(T), acts(8), W


def test_smooth_factors_and_weights(w4):
    Xc, _, W = _outlier_layer(256, 1024, 384, 5)
    W[:, 3] = 0.0                                    # a dead weight column: s = 1
    Wd = W.cuda()
    s, inv_s = w4.w4_smooth(Xc.cuda(), Wd, 0.5)
    torch.cuda.synchronize()
    os_ = O.smooth_factors(Xc, W.numpy(), 0.5)
    assert np.allclose(to_np(s), os_, rtol=4e-6, atol=0)
    assert to_np(s)[3] == 1.0
    assert np.allclose(to_np(inv_s), 1.0 / os_, rtol=4e-6, atol=0)
    assert np.allclose(to_np(Wd), W.numpy() * os_[None, :], rtol=5e-6, atol=0)
    # no calibration tokens: s = 1, W unchanged
    W2 = W.cuda()
    s0, _ = w4.w4_smooth(torch.zeros(0, 1024, dtype=torch.bfloat16, device="cuda"), W2, 0.5)
    assert torch.all(s0 == 1.0) and torch.equal(W2.cpu(), W)


@pytest.mark.parametrize("alpha", [0.5, 0.75])
def test_smoothquant_layer(w4, alpha):
    """Calibrate, smooth, pack and run the W4A8 layer on the GPU; the oracle
    runs the same steps in its own arithmetic, and both agree.  Smoothing
    does what it is for: the INT8 activations of the ordinary channels lose
    far less than without it.  (Whether the whole layer gains depends on the
    weights: with 4-bit weights the scaled-up outlier columns cost the weight
    groups precision, so this test does not assert it.)"""
    T, K, N, G = 256, 2048, 512, 128
    Xc, x, W = _outlier_layer(T, K, N, 11)
    # GPU
    Wd = W.cuda()
    s, inv_s = w4.w4_smooth(Xc.cuda(), Wd, alpha)
    p, sc, _ = w4.w4_pack_rtn(Wd, G, True)
    qx, sx = w4.w4a8_quantize_act_smooth(x.cuda(), inv_s, G)
    y, _ = w4.w4a8_linear(qx, sx, p, sc, None, N, K, G)
    # plain INT8 activations for comparison
    qx0, sx0 = w4.w4a8_quantize_act(x.cuda(), G)
    torch.cuda.synchronize()
    # oracle
    os_ = O.smooth_factors(Xc, W.numpy(), alpha)
    oinv = (np.float32(1.0) / os_.astype(np.float32)).astype(np.float32)
    op, osc, _ = O.pack_rtn((W.numpy() * os_.astype(np.float32)).astype(np.float32), G, True)
    oq, osx = O.w4a8_quantize_act(x, K, inv_s=oinv)
    _, oy = O.w4a8_linear_grouped(oq, osx, op, osc, G)
    assert_close(y, oy, f"smoothquant alpha {alpha}")
    # activation error on the channels without outliers
    xs = x.float().numpy().astype(np.float64)
    cold = np.abs(xs).max(axis=0) < 10.0
    deq0 = to_np(qx0).astype(np.float64)[:, :K] * to_np(sx0)[:, None]
    deq = to_np(qx).astype(np.float64)[:, :K] * to_np(sx)[:, None] * to_np(s)[None, :]
    e0 = np.linalg.norm((deq0 - xs)[:, cold]) / np.linalg.norm(xs[:, cold])
    e1 = np.linalg.norm((deq - xs)[:, cold]) / np.linalg.norm(xs[:, cold])
    assert e1 < 0.5 * e0, (e1, e0)
