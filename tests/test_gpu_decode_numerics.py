"""Decode-kernel numerics on activations that stress its fp16 operand form.

The decode GEMV feeds the tensor cores exact fp16 words 1024 + c (even
columns) and 1024 + 16 c (odd columns) and activations scaled by a power of
two per segment; the offset terms are removed at each group's flush.  The
offsets are exact, but the fp32 accumulation inside the MMA sees terms about
130 times larger than (c - z) x, so its rounding error scales with
sum |x| rather than with sum |(c - z) x|.  These inputs make that difference
as large as it gets, and the results must still meet the layer's tolerance
(relative Frobenius error <= 5e-3, max |diff| <= 1e-2 max |y|) against the
fp64 oracle ("Lab 5: Gemma4 端到端推理优化", sections "INT4 线性量化" and
"融合INT4反量化与矩阵乘"):

(a) activations all positive, at the large end of the supported range,
    with full 8-bit mantissas, and rows whose codes are balanced around the
    zero point (pairs c, 2z - c), so y is small against sum |x| |w_hat|;
(b) per 256-column segment one activation 10^4 above the rest, so the
    segment's power-of-two scale is set by the outlier and the others keep
    few bits above the fp16 range's bottom;
(c) alternating signs with a scale per 32-column block drawn from
    2^-40 .. 2^40, so groups span many binades.

Each runs at M = 1 and 16, G = 32 asymmetric and G = 128 symmetric, K = 3584
(the 7B hidden size), and also on the split-K 7B down-projection shape."""
import numpy as np
import pytest
import torch

import oracle as O
from helpers import assert_close, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _codes(rng, N, K, G, sym, balanced_rows):
    """Codes [N, K] in 0..15 and zero points [N, K/G] (8 when symmetric);
    every other row of `balanced_rows` pairs each even column's code c with
    2z - c (clipped) in the next column."""
    Ng = K // G
    z = np.full((N, Ng), 8, np.int64) if sym else rng.integers(3, 13, (N, Ng))
    c = rng.integers(0, 16, (N, K))
    if balanced_rows:
        zc = np.repeat(z, G, axis=1)
        mirror = np.clip(2 * zc[:, 0::2] - c[:, 0::2], 0, 15)
        rows = np.arange(N) % 2 == 0
        c[rows, 1::2] = mirror[rows]
    return c, z


def _activations(case, rng, M, K):
    if case == "a":
        # positive, 2^90 .. 2^91 with random mantissas
        x = rng.uniform(1.0, 2.0, (M, K)) * 2.0 ** 90
    elif case == "b":
        x = rng.standard_normal((M, K))
        for m in range(M):
            for s0 in range(0, K, 256):
                x[m, s0 + rng.integers(0, 256)] *= 1e4
    else:
        scale = 2.0 ** rng.integers(-40, 41, (M, K // 32))
        sign = np.where(np.arange(K) % 2 == 0, 1.0, -1.0)
        x = rng.uniform(0.5, 1.0, (M, K)) * sign * np.repeat(scale, 32, axis=1)
    return _bf16(x)


def _run(w4, case, M, N, K, G, sym, seed):
    rng = np.random.default_rng(seed)
    codes, z = _codes(rng, N, K, G, sym, balanced_rows=(case == "a"))
    packed = O.pack_nibbles(codes.astype(np.uint8))
    scales = rng.uniform(0.002, 0.02, (N, K // G)).astype(np.float32)
    zeros = None if sym else z.astype(np.uint8)
    x = _activations(case, rng, M, K)
    y = w4.w4a16_linear(x.cuda(), torch.from_numpy(packed).cuda(), torch.from_numpy(scales).cuda(),
                        None if sym else torch.from_numpy(zeros).cuda(), None, N, K, G)
    yref = O.w4a16_linear(x, packed, scales, zeros, None, K, G)
    assert np.all(np.isfinite(yref))
    return assert_close(y, yref, f"case {case} M{M} N{N} K{K} G{G} sym{sym}")


@pytest.mark.parametrize("case", ["a", "b", "c"])
@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("G,sym", [(32, False), (128, True)])
def test_decode_stress_activations(w4, case, M, G, sym):
    _run(w4, case, M, 512, 3584, G, sym, seed=ord(case) * 100 + M + G)


@pytest.mark.parametrize("case", ["a", "b", "c"])
def test_decode_stress_split_k(w4, case):
    """The 7B down-projection width (K = 18944, split over CTAs) at M = 1."""
    _run(w4, case, 1, 256, 18944, 128, True, seed=ord(case))


def test_balanced_rows_are_small(w4):
    """Guard on the construction of case (a): the balanced rows' exact
    results are much smaller than sum |x| |w_hat| (so the case does stress
    the cancellation), and the other rows are not."""
    rng = np.random.default_rng(1)
    N, K, G = 64, 3584, 128
    codes, z = _codes(rng, N, K, G, True, balanced_rows=True)
    x = rng.uniform(1.0, 2.0, K)
    w = (codes - 8).astype(np.float64)
    y = w @ x
    mag = np.abs(w) @ x
    assert np.all(np.abs(y[0::2]) < 0.2 * mag[0::2])
    assert np.median(np.abs(y[1::2]) / mag[1::2]) > 0.05
