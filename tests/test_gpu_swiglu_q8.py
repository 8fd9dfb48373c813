"""GPU parity of the fused gate|up + SiLU call that also emits the INT8
activations of the W4A8 layer after it (w4a16_linear_swiglu_q8): the
per-token dynamic quantization folded into the op before the integer GEMV
("Jetson Orin AGX INT4 推理优化实践", section 后续还能继续优化什么, item 2).

* y matches the fp64 oracle of the SwiGLU layer within the layer's
  tolerance, and equals w4a16_linear_swiglu's output bit for bit;
* qx and sx are bit-exact against the oracle's INT8 rule applied to the
  kernel's own bf16 y (the rounding of y to bf16 is the layer's; from there
  on the rule is exact), and equal the two-launch path
  (w4a16_linear_swiglu, then w4a8_quantize_act) bit for bit;
* padded columns F .. Fp-1 are zero; split and unsplit plans, every stage
  height, a zero token, two calls in a row on one workspace."""
import os

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


def _case(M, F, K, G, sym, seed, zero_token=False, bias=True):
    packed, scales, zeros = WL.make_random_format(2 * F, K, G, sym, seed)
    x = WL.make_activations(K, M, seed + 1)
    if zero_token:
        x[M - 1] = 0
    b = (torch.randn(2 * F, generator=torch.Generator().manual_seed(seed + 2)) * 0.5
         if bias else None)
    return packed, scales, zeros, x, b


def _check(w4, M, F, K, G, sym, Gq, seed, zero_token=False, bias=True):
    packed, scales, zeros, x, b = _case(M, F, K, G, sym, seed, zero_token, bias)
    args = (x.cuda(), packed.cuda(), scales.cuda(), None if zeros is None else zeros.cuda(),
            None if b is None else b.cuda(), F, K, G)
    y, qx, sx = w4.w4a16_linear_swiglu_q8(*args, Gq)
    torch.cuda.synchronize()
    yref = O.w4a16_linear_swiglu(x, packed.numpy(), scales.numpy(),
                                 None if zeros is None else zeros.numpy(),
                                 None if b is None else b.numpy(), F, K, G)
    assert_close(y, yref, f"swiglu_q8 y M{M} F{F} K{K}")
    Fp = O.padded_k(F, Gq)
    oq, osx = O.w4a8_quantize_act(y.cpu(), Fp)
    assert np.array_equal(to_np(sx).view(np.uint32), osx.view(np.uint32)), "s_x differs"
    assert np.array_equal(to_np(qx), oq), "q_x differs"
    assert not to_np(qx)[:, F:].any(), "padded columns not zero"
    # the two-launch path, bit for bit
    y2 = w4.w4a16_linear_swiglu(*args)
    q2, s2 = w4.w4a8_quantize_act(y2, Gq)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(qx, q2) and torch.equal(sx, s2)
    return y, qx, sx


@pytest.mark.parametrize("coop", ["1", "0"])
@pytest.mark.parametrize("M,F,K,G,sym,Gq", [
    (1, 18944, 3584, 128, True, 18944),     # 7B MLP: the W4A8 down projection per row
    (8, 18944, 3584, 128, True, 128),       # the same, 8 tokens, group-wise W4A8
    (1, 1000, 3584, 128, False, 128),       # F padded to 1024
    (16, 768, 2048, 64, True, 256),
    (3, 200, 100, 32, False, 64),           # ragged K, asymmetric
    (1, 512, 16384, 128, True, 512),        # split-K plan
])
def test_swiglu_q8_matches_oracle_and_two_launches(w4, monkeypatch, coop, M, F, K, G, sym, Gq):
    """Both hand-offs of the quantization: every CTA quantizes its share
    after a grid-wide barrier (cooperative launch, the default), or the last
    CTA quantizes all of y (W4_GEMV_COOP=0)."""
    monkeypatch.setenv("W4_GEMV_COOP", coop)
    _check(w4, M, F, K, G, sym, Gq, seed=M + F + K)
    _check(w4, M, F, K, G, sym, Gq, seed=M + F + K + 1)     # a second call: next generation


@pytest.mark.parametrize("rows,split", [("16", "1"), ("16", "2"), ("16", "4"),
                                        ("128", "1"), ("128", "3")])
def test_swiglu_q8_every_plan(w4, rows, split):
    """Forced stage heights and K splits (K = 8192: four 2048-column stages
    of 16 rows, thirty-two 256-column stages of 128 rows)."""
    old = {k: os.environ.get(k) for k in ("W4_GEMV_ROWS", "W4_GEMV_SPLIT")}
    os.environ["W4_GEMV_ROWS"], os.environ["W4_GEMV_SPLIT"] = rows, split
    try:
        _check(w4, 4, 1024, 8192, 128, True, 128, seed=int(rows) + int(split))
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def test_swiglu_q8_zero_token_and_reuse(w4):
    """A token of zeros (no bias, so its y is zero) gets s_x = 0 and q_x = 0;
    two calls in a row on the same workspace (its completion counter and
    token maxima return to zero)."""
    for _ in range(2):
        y, qx, sx = _check(w4, 3, 256, 1024, 128, True, 128, seed=5, zero_token=True,
                           bias=False)
        assert float(sx[2]) == 0.0 and not to_np(qx)[2].any()
    assert w4.w4_get_device_error() == 0


@pytest.mark.parametrize("coop", ["1", "0", "alt"])
def test_swiglu_q8_maxima_do_not_carry_over(w4, monkeypatch, coop):
    """The per-token maxima live in the shared workspace: a call whose y is
    a thousand times smaller (or larger) than the previous call's still gets
    its own s_x (a stale maximum would give larger scales and mostly-zero
    codes), for either hand-off and for the two alternating."""
    packed, scales, zeros, x, b = _case(16, 512, 1024, 128, True, 9, bias=False)
    for i, xs in enumerate((x, x * 1e-3, x * 1e3, x)):
        # alt: the two hand-offs in turn on the same workspace
        monkeypatch.setenv("W4_GEMV_COOP", str(i % 2) if coop == "alt" else coop)
        xs = xs.to(torch.bfloat16)
        args = (xs.cuda(), packed.cuda(), scales.cuda(), None, None, 512, 1024, 128)
        y, qx, sx = w4.w4a16_linear_swiglu_q8(*args, 128)
        oq, osx = O.w4a8_quantize_act(y.cpu(), 512)
        assert np.array_equal(to_np(sx).view(np.uint32), osx.view(np.uint32))
        assert np.array_equal(to_np(qx), oq)


def test_swiglu_q8_argument_errors(w4):
    packed, scales, _, x, _ = _case(1, 64, 256, 128, True, 1)
    args = (x.cuda(), packed.cuda(), scales.cuda(), None, None, 64, 256, 128)
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_linear_swiglu_q8(*args, 48)
    assert e.value.code == -4
    x17 = WL.make_activations(256, 17, 2).cuda()
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_linear_swiglu_q8(x17, *args[1:], 128)
    assert e.value.code == -8
