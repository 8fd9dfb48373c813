"""GPU parity of the bf16 parameter layout (bf16 scales and, asymmetric, bf16
(8 - z) s offsets; "Yeniden paketlenmiş QAT Gemma 4 26B-A4B, tek bir TPU
v6e'de …", section 26B'deki boşluk; "Lab 5: Gemma4 端到端推理优化",
section 融合INT4反量化与矩阵乘) through the C ABI, against the CPU oracle.

Bit-exact: the packed codes and the bf16 bits of every scale and offset.
Float tolerance (rel. Frobenius 5e-3, max|diff| 1e-2 max|y|): decode and
prefill outputs against the oracle's fp64 product with the same bf16
parameters."""
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


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy().astype(np.uint16)


def _pack_both(w4, W, G, sym):
    p, sb, ob = w4.w4_pack_rtn_bf16(W.cuda(), G, sym)
    op, osb, oob = O.pack_rtn_bf16(W.numpy(), G, sym)
    assert np.array_equal(to_np(p), op), "codes differ"
    assert np.array_equal(_bits(sb), (osb.view(np.uint32) >> 16).astype(np.uint16)), "scales differ"
    if sym:
        assert ob is None and oob is None
    else:
        assert np.array_equal(_bits(ob), (oob.view(np.uint32) >> 16).astype(np.uint16))
    return (p, sb, ob), (op, osb, oob)


def _run(w4, M, N, K, G, sym, seed, rows=None, wout=0.0):
    lin = WL.Linear("bf16p", M, N, K, G, sym, seed=seed, bias=True, w_outlier_frac=wout)
    inp = WL.make_inputs(lin)
    (p, sb, ob), (op, osb, oob) = _pack_both(w4, inp.W, G, sym)
    y = w4.w4a16_linear_bf16p(inp.x.cuda(), p, sb, ob, inp.bias.cuda(), N, K, G)
    torch.cuda.synchronize()
    yref = O.w4a16_linear_bf16_params(inp.x, op, osb, oob, inp.bias.numpy(), K, G, rows=rows)
    yg = y if rows is None else y[:, torch.as_tensor(rows, device=y.device)]
    assert_close(yg, yref, f"bf16p M{M} N{N} K{K} G{G} sym{sym}")
    assert w4.w4_get_device_error() == 0
    return y


@pytest.mark.parametrize("M,N,K,G,sym", [
    (1, 256, 512, 32, True), (3, 300, 1000, 32, False), (8, 512, 4096, 128, True),
    (16, 384, 2048, 32, False), (5, 200, 960, 96, False), (1, 130, 40960, 128, False),
    (12, 1000, 3584, 64, True),
])
def test_bf16p_decode_shapes(w4, M, N, K, G, sym):
    """Both scale load paths (eight bf16 scales per 16-byte load at G = 32,
    scalar otherwise), split-K shapes, ragged N and K, bias."""
    _run(w4, M, N, K, G, sym, seed=M + N + K + G)


@pytest.mark.parametrize("rows,split", [("16", "1"), ("64", "3"), ("128", "6")])
def test_bf16p_decode_pinned_plans(w4, monkeypatch, rows, split):
    monkeypatch.setenv("W4_GEMV_ROWS", rows)
    monkeypatch.setenv("W4_GEMV_SPLIT", split)
    _run(w4, 4, 640, 6144, 32, False, seed=int(rows) + int(split))


@pytest.mark.parametrize("M", [1, 16])
def test_bf16p_7b_and_12b_shapes(w4, M):
    rows = np.unique(np.concatenate([np.arange(0, 4608, 9), [4607]]))
    _run(w4, M, 4608, 3584, 128, True, seed=100 + M, rows=rows)
    rows = np.unique(np.concatenate([np.arange(0, 15360, 31), [15359]]))
    _run(w4, M, 15360, 3840, 32, False, seed=200 + M, rows=rows, wout=0.01)


@pytest.mark.parametrize("M,N,K,G,sym", [(64, 1024, 2048, 128, False), (512, 768, 1024, 32, True),
                                         (300, 512, 3584, 64, False)])
def test_bf16p_prefill(w4, M, N, K, G, sym):
    """M > 16: the tensor-core kernel dequantizes with the bf16 parameters."""
    _run(w4, M, N, K, G, sym, seed=M + N)
