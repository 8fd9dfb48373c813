"""GPU GPTQ (fp32, blocked) against the CPU oracle (fp64, column by column),
"Lab 5: Gemma4 端到端推理优化", section 从 RTN 到 GPTQ.

Exact where nothing propagates (an isotropic Hessian: the codes and scales
are RTN's) and for dead and padded columns (exact zeros).  Elsewhere the two
sides propagate in different precisions, which can flip a code near a
rounding boundary and then take slightly different paths; the comparison
is on the quantities GPTQ optimises: the share of identical codes, the
predicted loss L_pred and the calibration objective ||X (W - W_hat)^T||."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import ensure_built, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _unpack(packed):
    return O.unpack_nibbles(to_np(packed))


def _dequant(codes, scales, zeros, G):
    N, Kp = codes.shape
    z = np.full((N, Kp // G), 8.0) if zeros is None else zeros.astype(np.float64)
    return (scales.astype(np.float64)[:, :, None]
            * (codes.reshape(N, Kp // G, G).astype(np.float64) - z[:, :, None])).reshape(N, Kp)


def _hadamard(n):
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def _correlated(T, K, N, seed):
    g = np.random.default_rng(seed)
    A = g.standard_normal((K, K)) * 0.4 + np.eye(K)
    X = torch.from_numpy((g.standard_normal((T, K)) @ A).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy((g.standard_normal((N, K)) * 0.05).astype(np.float32))
    return X, W


@pytest.mark.parametrize("symmetric,G", [(True, 32), (False, 32), (True, 64), (False, 128)])
def test_gptq_isotropic_is_rtn_exactly(w4, symmetric, G):
    K = 128
    X = torch.from_numpy(_hadamard(K).astype(np.float32)).to(torch.bfloat16)
    W = torch.from_numpy((np.random.default_rng(G).standard_normal((40, K)) * 0.1).astype(np.float32))
    p, s, z, loss = w4.w4_gptq(X.cuda(), W.cuda(), G, symmetric)
    torch.cuda.synchronize()
    assert w4.w4_get_device_error() == 0
    rc, rs, rz = O.rtn_quantize(W.numpy(), G, symmetric)
    assert np.array_equal(_unpack(p), rc)
    assert np.array_equal(to_np(s).view(np.uint32), rs.view(np.uint32))
    if not symmetric:
        assert np.array_equal(to_np(z), rz)


@pytest.mark.parametrize("symmetric", [True, False])
def test_gptq_dead_and_padded_columns(w4, symmetric):
    T, K, N, G = 96, 200, 24, 64                       # Kp = 256: 56 padded columns
    X, W = _correlated(T, K, N, 3)
    X[:, [5, 77]] = 0
    p, s, z, loss = w4.w4_gptq(X.cuda(), W.cuda(), G, symmetric)
    torch.cuda.synchronize()
    Wq = _dequant(_unpack(p), to_np(s), None if symmetric else to_np(z), G)
    assert np.all(Wq[:, [5, 77]] == 0) and np.all(Wq[:, K:] == 0)
    assert np.all(np.isfinite(to_np(loss)))
    assert w4.w4_get_device_error() == 0


def _compare(w4, X, W, G, symmetric, rows=None, min_same=0.97):
    p, s, z, loss = w4.w4_gptq(X.cuda(), W.cuda(), G, symmetric)
    torch.cuda.synchronize()
    assert w4.w4_get_device_error() == 0
    codes = _unpack(p)
    sc = to_np(s)
    zz = None if symmetric else to_np(z)
    lg = to_np(loss).astype(np.float64)
    Wr = W.numpy() if rows is None else W.numpy()[rows]
    if rows is not None:
        codes, sc, lg = codes[rows], sc[rows], lg[rows]
        zz = None if zz is None else zz[rows]
    oc, os_, oz, ol, Hd, W0 = O.gptq_quantize(Wr, X, G, symmetric)
    same = np.mean(codes == oc)
    assert same >= min_same, same
    assert abs(lg.sum() - ol.sum()) <= 0.02 * ol.sum(), (lg.sum(), ol.sum())
    # the GPU's codes carry the loss they claim, under the oracle's Hessian
    D = W0 - _dequant(codes, sc, zz, G)
    quad = 0.5 * np.einsum("nk,kj,nj->n", D, Hd, D)
    assert abs(quad.sum() - lg.sum()) <= 0.02 * quad.sum(), (quad.sum(), lg.sum())
    # calibration objective against the oracle's and RTN's
    K = W.shape[1]
    Xd = X.float().numpy().astype(np.float64)
    obj = lambda Wq: np.linalg.norm(Xd @ (Wr.astype(np.float64) - Wq[:, :K]).T)
    o_gpu = obj(_dequant(codes, sc, zz, G))
    o_orc = obj(_dequant(oc, os_, oz, G))
    rc, rs, rz = O.rtn_quantize(Wr, G, symmetric)
    o_rtn = obj(_dequant(rc, rs, rz, G))
    assert abs(o_gpu - o_orc) <= 0.02 * o_orc, (o_gpu, o_orc)
    assert o_gpu < 0.9 * o_rtn, (o_gpu, o_rtn)


@pytest.mark.parametrize("T,K,N,G,sym", [(256, 256, 96, 32, True), (512, 512, 64, 128, False),
                                         (300, 640, 48, 64, True), (128, 1024, 32, 1024, True)])
def test_gptq_matches_oracle(w4, T, K, N, G, sym):
    X, W = _correlated(T, K, N, K + G)
    _compare(w4, X, W, G, sym)


def test_gptq_7b_qkv_shape_sampled_rows(w4):
    """4608 x 3584 (the 7B fused QKV projection), G = 128, 512 calibration
    tokens; the oracle quantizes a sample of the rows (rows are independent
    given U)."""
    g = torch.Generator().manual_seed(9)
    K, N, T = 3584, 4608, 512
    mix = torch.randn(K, 64, generator=g) * 0.3
    X = (torch.randn(T, K, generator=g) + torch.randn(T, 64, generator=g) @ mix.T).to(torch.bfloat16)
    W = torch.randn(N, K, generator=g) * 0.02
    rows = np.sort(np.random.default_rng(1).choice(N, 64, replace=False))
    _compare(w4, X, W, 128, True, rows=rows, min_same=0.95)


def test_gptq_argument_errors(w4):
    X = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(8, 64, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.w4_gptq(X, W, 32, True)                  # no calibration tokens
    assert e.value.code in (-1, -2)
    with pytest.raises(w4.W4Error) as e:
        w4.w4_gptq(torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda"), W, 48, True)
    assert e.value.code == -4
