"""Pins for the CPU oracle: closed forms, invariants, worked numbers from the
pages, and brute force on tiny inputs.  Every check here is computed
independently of the oracle's own code path, so a dropped term, a wrong sign,
a swapped nibble or a transposed operand in the oracle fails at least one.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_w(N, K, seed, std=0.02, outlier_cols=0):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * std).astype(np.float32)
    if outlier_cols:
        cols = rng.permutation(K)[:outlier_cols]
        W[:, cols] *= np.float32(20.0)
    return W


def _bf16_round(a):
    """Round fp32 values to bf16 (nearest-even) and return them as fp32."""
    a = np.asarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


# ---------------------------------------------------------------------------
# Quantisation closed forms (page "Lab 5: Gemma4 端到端推理优化", INT4 线性量化)
# ---------------------------------------------------------------------------

def test_symmetric_closed_form_and_ties():
    # One group of 32 with max|r| = 7/8, so s = 1/8 exactly; r = k/8 gives
    # q = k exactly, r = +-1.5/8 and 0.5/8 are ties (half to even).
    r = np.zeros(32, np.float32)
    r[:8] = [0.875, -0.875, 0.125, -0.25, 0.0625, 0.1875, -0.1875, -0.3125]
    codes, s, z = O.rtn_quantize(r[None, :], 32, True)
    assert z is None
    assert s[0, 0] == np.float32(0.125)
    q = codes[0].astype(int) - 8
    assert list(q[:8]) == [7, -7, 1, -2, 0, 2, -2, -2]
    assert all(q[8:] == 0)


def test_asymmetric_closed_form():
    # rmin = -1, rmax = 2: s = 3/15 (fp32), z = round(1/s) = 5.
    r = np.linspace(-1.0, 2.0, 32).astype(np.float32)
    codes, s, z = O.rtn_quantize(r[None, :], 32, False)
    assert s[0, 0] == np.float32(3.0) / np.float32(15.0)
    assert z[0, 0] == 5
    assert codes[0, 0] == 0 and codes[0, -1] == 15
    r2 = r.copy()
    r2[7] = 0.0
    c2, s2, z2 = O.rtn_quantize(r2[None, :], 32, False)
    assert c2[0, 7] == z2[0, 0]           # zero maps onto the zero point
    W = O.dequantize_f64(O.pack_nibbles(c2), s2, z2, 32)
    assert W[0, 7] == 0.0


def test_asymmetric_positive_group_includes_zero():
    # Reading (v): the range is widened to contain 0, so z stays in [0, 15].
    r = np.linspace(0.5, 1.5, 32).astype(np.float32)
    codes, s, z = O.rtn_quantize(r[None, :], 32, False)
    assert z[0, 0] == 0
    assert s[0, 0] == np.float32(1.5) / np.float32(15.0)
    r = -r
    codes, s, z = O.rtn_quantize(r[None, :], 32, False)
    assert z[0, 0] == 15


@pytest.mark.parametrize("symmetric", [True, False])
def test_zero_group(symmetric):
    W = np.zeros((2, 64), np.float32)
    W[1, 40] = 0.5
    codes, s, z = O.rtn_quantize(W, 32, symmetric)
    assert s[0, 0] == 0 and s[0, 1] == 0 and s[1, 0] == 0
    Wd = O.dequantize_f64(O.pack_nibbles(codes), s, z, 32)
    assert np.all(Wd[0] == 0.0) and np.all(Wd[1, :32] == 0.0)
    assert Wd[1, 40] == pytest.approx(0.5, rel=1e-6)


@pytest.mark.parametrize("symmetric", [True, False])
@pytest.mark.parametrize("G", [32, 128])
def test_codes_are_nearest_grid_point(symmetric, G):
    """Brute force: every code is the grid point s*(c - z), c in 0..15,
    nearest to r (ties, and values within fp32 rounding of a tie, may go
    either way)."""
    W = _rand_w(24, 256, seed=G + symmetric, outlier_cols=3)
    codes, s, z = O.rtn_quantize(W, G, symmetric)
    N, Kp = codes.shape
    Ng = Kp // G
    zz = np.full((N, Ng), 8) if z is None else z.astype(int)
    grid_c = np.arange(16)
    for n in range(N):
        for g in range(Ng):
            sg = float(s[n, g])
            r = W[n, g * G:(g + 1) * G].astype(np.float64)
            dist = np.abs(r[:, None] - sg * (grid_c[None, :] - zz[n, g]))
            best = dist.argmin(axis=1)
            got = codes[n, g * G:(g + 1) * G].astype(int)
            d_got = dist[np.arange(G), got]
            d_best = dist[np.arange(G), best]
            # equal distance (a tie) is fine; anything else must match
            assert np.all(d_got <= d_best + 1e-6 * sg), (n, g)


@pytest.mark.parametrize("symmetric", [True, False])
def test_rtn_error_at_most_half_step(symmetric):
    """|r - r_hat| <= s/2 for every element (the half-step bound of
    symmetric INT8 on page 2, section 2.2, carried to the INT4 grid)."""
    W = _rand_w(64, 384, seed=7, outlier_cols=4)
    packed, s, z = O.pack_rtn(W, 32, symmetric)
    Wd = O.dequantize_f64(packed, s, z, 32)[:, :384]
    step = np.repeat(s.astype(np.float64), 32, axis=1)[:, :384]
    assert np.all(np.abs(W - Wd) <= step / 2 * (1 + 1e-6))


# ---------------------------------------------------------------------------
# Packing
# ---------------------------------------------------------------------------

def test_pack_bit_layout_and_round_trip():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 16, size=(5, 64)).astype(np.uint8)
    p = O.pack_nibbles(codes)
    assert p.shape == (5, 32)
    for n in range(5):
        for j in range(32):
            assert int(p[n, j]) == int(codes[n, 2 * j]) | (int(codes[n, 2 * j + 1]) << 4)
    # a little-endian uint32 holds eight codes [w7 ... w0] (page 4, DP4A 做了什么)
    words = p.view("<u4")
    for n in range(5):
        for w in range(8):
            expect = sum(int(codes[n, 8 * w + i]) << (4 * i) for i in range(8))
            assert int(words[n, w]) == expect
    assert np.array_equal(O.unpack_nibbles(p), codes)


def test_unpack_in_place_mistake_is_caught():
    """Page 'Lab 5', section 量化正确性修正: interleaving into the packed uint8
    storage itself corrupts the codes; the oracle's unpack does not."""
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 16, size=(3, 64)).astype(np.uint8)
    packed = O.pack_nibbles(codes)

    def naive_in_place(pk):
        buf = np.zeros((pk.shape[0], pk.shape[1] * 2), np.uint8)
        buf[:, :pk.shape[1]] = pk          # codes live in the same storage
        view = buf
        src = view[:, :pk.shape[1]]
        view[:, 0::2] = src & 0x0F         # overwrites bytes still to be read
        view[:, 1::2] = src >> 4
        return view

    assert not np.array_equal(naive_in_place(packed), codes)
    assert np.array_equal(O.unpack_nibbles(packed), codes)


def test_bytes_per_row_matches_page_table():
    g = _golden("p4_bytes_per_row.json")
    H = g["H"]
    W = _rand_w(2, H, seed=3)
    packed, s, _ = O.pack_rtn(W, 128, True)
    assert packed.shape[1] == g["int4_row_bytes"]
    assert 2 * H == g["fp16_row_bytes"] and H == g["int8_row_bytes"]


# ---------------------------------------------------------------------------
# Padding (page 'Lab 5', INT4 线性量化: padded positions dequantize to zero)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("symmetric", [True, False])
def test_padding_dequantizes_to_zero_and_changes_nothing(symmetric):
    K, G = 100, 32          # Kp = 128
    W = _rand_w(8, K, seed=4)
    packed, s, z = O.pack_rtn(W, G, symmetric)
    assert packed.shape[1] == 64
    Wd = O.dequantize_f64(packed, s, z, G)
    assert np.all(Wd[:, K:] == 0.0)
    assert not np.any(np.signbit(Wd[:, K:]))
    # appending explicit zero columns to W and x leaves y unchanged
    Wz = np.zeros((8, 128), np.float32)
    Wz[:, :K] = W
    p2, s2, z2 = O.pack_rtn(Wz, G, symmetric)
    assert np.array_equal(p2, packed) and np.array_equal(s2, s)
    rng = np.random.default_rng(5)
    x = _bf16_round(rng.standard_normal((3, K)))
    xz = np.zeros((3, 128), np.float32)
    xz[:, :K] = x
    y1 = O.w4a16_linear(x, packed, s, z, None, K, G)
    y2 = O.w4a16_linear(xz, p2, s2, z2, None, 128, G)
    assert np.array_equal(y1, y2)


def test_additive_offset_identity():
    """Page 'Lab 5', 融合INT4反量化与矩阵乘: with codes read as (q - 8), an
    asymmetric group needs the additive offset (8 - z) s:
    s (q - z) == s (q - 8) + (8 - z) s, exactly in fp64."""
    W = _rand_w(16, 256, seed=6, outlier_cols=2)
    codes, s, z = O.rtn_quantize(W, 32, False)
    sf = np.repeat(s.astype(np.float64), 32, axis=1)
    zf = np.repeat(z.astype(np.float64), 32, axis=1)
    c = codes.astype(np.float64)
    lhs = O.dequantize_f64(O.pack_nibbles(codes), s, z, 32)
    rhs = sf * (c - 8) + (8 - zf) * sf
    assert np.array_equal(lhs, rhs)
    assert np.array_equal(lhs, sf * (c - zf))


# ---------------------------------------------------------------------------
# Matmul
# ---------------------------------------------------------------------------

def test_dyadic_inputs_give_exact_integer_result():
    """x in {0, +-1/4, +-1/2, +-1}, group maxima 7 * 2^-e so that s = 2^-e:
    every product and partial sum is exact in fp64, so the oracle must equal
    an integer computation done here with Python ints."""
    rng = np.random.default_rng(8)
    M, N, K, G = 3, 5, 64, 32
    qs = rng.integers(-7, 8, size=(N, K))
    e = rng.integers(2, 6, size=(N, K // G))
    W = np.zeros((N, K), np.float32)
    for n in range(N):
        for g in range(K // G):
            qs[n, g * G] = 7                        # pin the group max to 7 s
            W[n, g * G:(g + 1) * G] = qs[n, g * G:(g + 1) * G] * 2.0 ** -int(e[n, g])
    x4 = rng.integers(-4, 5, size=(M, K))
    x4[np.abs(x4) == 3] = 0
    x = (x4 / 4.0).astype(np.float32)
    packed, s, z = O.pack_rtn(W, G, True)
    y = O.w4a16_linear(x, packed, s, z, None, K, G)
    # exact: y * 4 * 2^emax is an integer
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for k in range(K):
                tot += Fraction(int(x4[m, k]), 4) * Fraction(int(qs[n, k]), 2 ** int(e[n, k // G]))
            assert Fraction(y[m, n]) == tot


@pytest.mark.parametrize("symmetric", [True, False])
def test_tiny_brute_force_triple_loop(symmetric):
    """Independent triple loop with exact rationals, from the codes, scales
    and zeros, for M, N, K in 1..3 x 1..5 x 32..64, with bias."""
    rng = np.random.default_rng(9)
    for (M, N, K, G) in [(1, 1, 32, 32), (2, 3, 40, 32), (3, 5, 64, 32), (1, 4, 64, 64)]:
        W = _rand_w(N, K, seed=M * 100 + N * 10 + K)
        x = _bf16_round(rng.standard_normal((M, K)))
        b = rng.standard_normal(N).astype(np.float32)
        codes, s, z = O.rtn_quantize(W, G, symmetric)
        packed = O.pack_nibbles(codes)
        y = O.w4a16_linear(x, packed, s, z, b, K, G)
        for m in range(M):
            for n in range(N):
                tot = Fraction(float(b[n]))
                for k in range(K):
                    g = k // G
                    zp = 8 if z is None else int(z[n, g])
                    w = Fraction(float(s[n, g])) * (int(codes[n, k]) - zp)
                    tot += Fraction(float(x[m, k])) * w
                assert abs(y[m, n] - float(tot)) <= 1e-12 * max(1.0, abs(float(tot)))


# ---------------------------------------------------------------------------
# W4A8 (page 'Jetson Orin AGX INT4 推理优化实践')
# ---------------------------------------------------------------------------

def test_int32_bound_worked_number_and_worst_case():
    g = _golden("p4_int32_bound.json")
    assert g["max_abs_qw"] * g["max_abs_qx"] == g["per_term"]
    assert O.int32_worst_case(g["H"]) == g["bound"]
    assert g["bound"] < g["int32_max"] == 2 ** 31 - 1
    # worst-case synthetic input: all codes 0 (q = -8) and all qx = 127
    K = 18944
    packed = np.zeros((2, K // 2), np.uint8)
    qx = np.full((1, K), 127, np.int8)
    acc, y = O.w4a8_linear(qx, np.ones(1, np.float32), packed,
                           np.ones(2, np.float32), None)
    assert acc[0, 0] == -O.int32_worst_case(K) == -8 * 127 * K
    assert abs(acc[0, 0]) < 2 ** 31 - 1


def test_w4a8_reduction_sums_codes():
    """With qx = 1 and s_x = s_W = 1, acc_j is the row sum of the signed
    codes q = code - 8."""
    rng = np.random.default_rng(10)
    codes = rng.integers(0, 16, size=(7, 96)).astype(np.uint8)
    packed = O.pack_nibbles(codes)
    qx = np.ones((1, 96), np.int8)
    acc, y = O.w4a8_linear(qx, np.ones(1, np.float32), packed,
                           np.ones(7, np.float32), None)
    assert np.array_equal(acc[0], codes.astype(np.int64).sum(axis=1) - 8 * 96)
    assert np.array_equal(y[0], acc[0].astype(np.float64))


def test_w4a8_matches_its_definition_by_loop():
    rng = np.random.default_rng(11)
    N, K = 6, 64
    W = _rand_w(N, K, seed=12)
    packed, ws, _ = O.pack_rtn(W, K, True)          # per-row scale
    x = _bf16_round(rng.standard_normal((2, K)))
    qx, sx = O.w4a8_quantize_act(x, K)
    b = rng.standard_normal(N).astype(np.float32)
    acc, y = O.w4a8_linear(qx, sx, packed, ws, b)
    codes = O.unpack_nibbles(packed).astype(int)
    for m in range(2):
        for n in range(N):
            a = sum((codes[n, k] - 8) * int(qx[m, k]) for k in range(K))
            assert acc[m, n] == a
            expect = float(ws[n, 0]) * float(sx[m]) * a + float(b[n])
            assert y[m, n] == pytest.approx(expect, rel=1e-15, abs=1e-15)


def test_int8_activation_examples_from_page_2():
    g = _golden("p2_int8_examples.json")
    rng = np.random.default_rng(13)
    # max 1.0: scale ~ 0.0078, error <= 0.0039
    x = _bf16_round(np.clip(rng.standard_normal((1, 512)) * 0.3, -0.99, 0.99))
    x[0, 17] = g["int8_symmetric"]["max"]
    qx, sx = O.w4a8_quantize_act(x, 512)
    assert sx[0] == np.float32(1.0) / np.float32(127.0)
    assert abs(float(sx[0]) - g["int8_symmetric"]["scale_approx"]) < 1e-4
    err = np.abs(qx[0].astype(np.float64) * float(sx[0]) - x[0])
    assert err.max() <= float(sx[0]) / 2 * (1 + 1e-6)
    assert err.max() <= g["int8_symmetric"]["max_error_approx"] + 1e-4
    assert qx[0, 17] == 127
    # one outlier of 5.0 among small values: scale ~ 0.039, 0.05 -> 1 -> 0.039
    ex = g["outlier_example"]
    x = _bf16_round(np.full((1, 64), ex["normal_value"], np.float32))
    x[0, 3] = ex["outlier"]
    qx, sx = O.w4a8_quantize_act(x, 64)
    assert abs(float(sx[0]) - ex["scale_approx"]) < 5e-4
    assert qx[0, 0] == ex["code"]
    assert abs(qx[0, 0] * float(sx[0]) - ex["dequant_approx"]) < 5e-4
    rel = abs(qx[0, 0] * float(sx[0]) - float(x[0, 0])) / float(x[0, 0])
    assert abs(rel - ex["rel_error_approx"]) < 0.015


def test_activation_quantize_closed_form_and_padding():
    x = np.zeros((2, 30), np.float32)
    x[0, :4] = [1.0, -0.5, 0.25, 0.0]
    qx, sx = O.w4a8_quantize_act(x, 32)
    assert qx.shape == (2, 32) and qx.dtype == np.int8
    assert sx[0] == np.float32(1.0) / np.float32(127.0)
    assert list(qx[0, :4]) == [127, -64, 32, 0]    # 63.5 -> 64 (half-even), 31.75 -> 32
    assert np.all(qx[:, 30:] == 0)
    assert sx[1] == 0 and np.all(qx[1] == 0)       # all-zero token


# ---------------------------------------------------------------------------
# Fused gate|up projection with SiLU ("Lab 5", section 基础)
# ---------------------------------------------------------------------------

def test_silu_closed_forms():
    import math
    v = np.array([0.0, math.log(3.0), -math.log(3.0), 1.0, -1.0, 40.0, -800.0, 800.0])
    s = O.silu_f64(v)
    assert s[0] == 0.0
    # sigma(ln 3) = 3/4 and sigma(-ln 3) = 1/4
    assert abs(s[1] - 0.75 * math.log(3.0)) < 1e-15
    assert abs(s[2] + 0.25 * math.log(3.0)) < 1e-15
    # SiLU(v) - SiLU(-v) = v sigma(v) + v sigma(-v) = v
    assert abs((s[3] - s[4]) - 1.0) < 1e-15
    assert abs(s[3] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    # saturation: SiLU(v) -> v for large v, -> 0 for very negative v, no NaN
    assert abs(s[5] - 40.0) < 1e-15 and s[7] == 800.0
    assert s[6] == 0.0 and np.all(np.isfinite(s))


def test_swiglu_row_pairing():
    F = 24
    g_idx, u_idx = O.swiglu_rows(F)
    assert sorted(np.concatenate([g_idx, u_idx]).tolist()) == list(range(2 * F))
    assert list(g_idx[:10]) == [0, 1, 2, 3, 4, 5, 6, 7, 16, 17]
    assert list(u_idx[:10]) == [8, 9, 10, 11, 12, 13, 14, 15, 24, 25]
    gate = np.arange(F) + 1000
    up = np.arange(F) + 2000
    fused = O.pair_rows(gate, up)
    assert list(fused[:17]) == ([1000 + i for i in range(8)] + [2000 + i for i in range(8)]
                                + [1008])
    with pytest.raises(ValueError):
        O.pair_rows(np.zeros(12), np.zeros(12))


@pytest.mark.parametrize("symmetric", [True, False])
def test_swiglu_brute_force_loops(symmetric):
    """Pure-Python loops over bytes and nibbles of the separately packed gate
    and up matrices: SiLU(sum x w_gate + b_gate) * (sum x w_up + b_up)."""
    import math
    F, K, G, M = 16, 40, 16, 2
    rng = np.random.default_rng(11)
    Wg = _rand_w(F, K, 1, std=0.5)
    Wu = _rand_w(F, K, 2, std=0.5)
    bg = rng.standard_normal(F).astype(np.float32)
    bu = rng.standard_normal(F).astype(np.float32)
    x = _bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    pg, sg, zg = O.pack_rtn(Wg, G, symmetric)
    pu, su, zu = O.pack_rtn(Wu, G, symmetric)
    # quantization is row-wise: packing the fused matrix equals fusing the packs
    pf, sf, zf = O.pack_rtn(O.pair_rows(Wg, Wu), G, symmetric)
    assert np.array_equal(pf, O.pair_rows(pg, pu))
    assert np.array_equal(sf, O.pair_rows(sg, su))
    if not symmetric:
        assert np.array_equal(zf, O.pair_rows(zg, zu))
    y = O.w4a16_linear_swiglu(x, pf, sf, zf, O.pair_rows(bg, bu), F, K, G)

    def proj(p, s, z, b, m, f):
        acc = 0.0
        for k in range(K):
            byte = int(p[f, k // 2])
            code = (byte >> 4) if k % 2 else (byte & 15)
            zero = 8 if z is None else int(z[f, k // G])
            acc += float(x[m, k]) * float(s[f, k // G]) * (code - zero)
        return acc + float(b[f])

    for m in range(M):
        for f in range(F):
            g = proj(pg, sg, zg, bg, m, f)
            u = proj(pu, su, zu, bu, m, f)
            want = g / (1.0 + math.exp(-g)) * u
            assert abs(y[m, f] - want) <= 1e-12 * (1.0 + abs(want))
    cols = np.array([3, 9, 15])
    assert np.array_equal(O.w4a16_linear_swiglu(x, pf, sf, zf, O.pair_rows(bg, bu), F, K, G,
                                                cols=cols), y[:, cols])


# ---------------------------------------------------------------------------
# Grouped linear over experts ("Yeniden paketlenmiş QAT Gemma 4 26B-A4B, tek
# bir TPU v6e'de ...", expert layers)
# ---------------------------------------------------------------------------

def _grouped_case(E, N, K, G, counts, symmetric, seed):
    rng = np.random.default_rng(seed)
    W = _rand_w(E * N, K, seed, std=0.1)
    packed, scales, zeros = O.pack_rtn(W, G, symmetric)
    T = int(sum(counts))
    x = _bf16_round(rng.standard_normal((T, K)).astype(np.float32))
    bias = rng.standard_normal(E * N).astype(np.float32)
    goff = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return x, goff, packed, scales, zeros, bias


@pytest.mark.parametrize("symmetric", [True, False])
def test_grouped_equals_dense_product_over_all_experts(symmetric):
    """Independent formulation: one fp64 product of every token with every
    expert's dequantized matrix, [T, E*N], from which each row keeps the
    block of its own expert (found by searching the offsets)."""
    E, N, K, G = 6, 16, 96, 32
    counts = [3, 0, 1, 5, 0, 2]
    x, goff, packed, scales, zeros, bias = _grouped_case(E, N, K, G, counts, symmetric, 4)
    y = O.w4a16_grouped_linear(x, goff, packed, scales, zeros, bias, E, N, K, G)
    Wd = O.dequantize_f64(packed, scales, zeros, G)[:, :K]
    full = x.astype(np.float64) @ Wd.T + bias.astype(np.float64)[None, :]
    for t in range(x.shape[0]):
        e = int(np.searchsorted(goff, t, side="right") - 1)
        assert np.allclose(y[t], full[t, e * N:(e + 1) * N], rtol=0, atol=1e-12)
    cols = np.array([0, 5, 15])
    yc = O.w4a16_grouped_linear(x, goff, packed, scales, zeros, bias, E, N, K, G, cols=cols)
    assert np.array_equal(yc, y[:, cols])


def test_grouped_token_order_and_offsets():
    """Permuting tokens inside a group permutes its rows of y; a group's
    result depends only on its own tokens; bad offsets are rejected."""
    E, N, K, G = 3, 8, 64, 32
    counts = [4, 0, 3]
    x, goff, packed, scales, zeros, bias = _grouped_case(E, N, K, G, counts, True, 9)
    y = O.w4a16_grouped_linear(x, goff, packed, scales, None, bias, E, N, K, G)
    perm = np.array([2, 0, 3, 1, 4, 5, 6])
    yp = O.w4a16_grouped_linear(x[perm], goff, packed, scales, None, bias, E, N, K, G)
    assert np.array_equal(yp, y[perm])
    x2 = x.copy()
    x2[4:] *= -3.0                       # change group 2's tokens only
    y2 = O.w4a16_grouped_linear(_bf16_round(x2), goff, packed, scales, None, bias, E, N, K, G)
    assert np.array_equal(y2[:4], y[:4]) and not np.allclose(y2[4:], y[4:])
    for bad in ([0, 5, 4, 7], [1, 4, 4, 7], [0, 4, 4, 8]):
        with pytest.raises(ValueError):
            O.w4a16_grouped_linear(x, np.array(bad), packed, scales, None, bias, E, N, K, G)


# ---------------------------------------------------------------------------
# Group-wise W4A8 and SmoothQuant smoothing ("【infra之路】12-…", section 2.4;
# "LLM 模型壓縮與推理加速實踐-陳磊.pdf", W8A8 slides)
# ---------------------------------------------------------------------------

def test_w4a8_grouped_one_group_is_per_row():
    rng = np.random.default_rng(3)
    N, K = 24, 256
    W = _rand_w(N, K, 5, std=0.3)
    packed, scales, _ = O.pack_rtn(W, K, True)
    x = _bf16_round(rng.standard_normal((3, K)).astype(np.float32))
    qx, sx = O.w4a8_quantize_act(x, K)
    acc, y = O.w4a8_linear(qx, sx, packed, scales, None)
    accg, yg = O.w4a8_linear_grouped(qx, sx, packed, scales, K)
    assert np.array_equal(accg[:, :, 0], acc)
    assert np.array_equal(yg, y)


def test_w4a8_grouped_brute_force_loops():
    """Pure-Python loops over bytes and nibbles, per group."""
    rng = np.random.default_rng(8)
    N, K, G = 5, 96, 32
    W = _rand_w(N, K, 6, std=0.3)
    packed, scales, _ = O.pack_rtn(W, G, True)
    x = _bf16_round(rng.standard_normal((2, K)).astype(np.float32))
    qx, sx = O.w4a8_quantize_act(x, K)
    b = rng.standard_normal(N).astype(np.float32)
    acc, y = O.w4a8_linear_grouped(qx, sx, packed, scales, G, bias=b)
    for m in range(2):
        for n in range(N):
            tot = 0.0
            for g in range(K // G):
                a = 0
                for k in range(g * G, (g + 1) * G):
                    byte = int(packed[n, k // 2])
                    code = (byte >> 4) if k % 2 else (byte & 15)
                    a += (code - 8) * int(qx[m, k])
                assert acc[m, n, g] == a
                tot += float(scales[n, g]) * a
            assert abs(y[m, n] - (float(sx[m]) * tot + float(b[n]))) <= 1e-12 * (1 + abs(y[m, n]))


def test_smooth_factors_closed_form():
    X = np.zeros((3, 4), np.float32)
    X[0] = [4.0, -1.0, 0.0, 2.0]
    X[2] = [-2.0, 0.5, 0.0, 1.0]
    W = np.array([[1.0, 4.0, 3.0, 0.0], [-0.5, -2.0, 1.0, 0.0]], np.float32)
    s = O.smooth_factors(X, W, 0.5)
    assert np.allclose(s, [2.0, 0.5, 1.0, 1.0], rtol=0, atol=1e-15)   # zero maxima -> 1
    # at alpha = 1/2 the smoothed maxima meet at sqrt(max|X_j| max|W_j|)
    xs = np.abs(X[:, :2] / s[:2]).max(axis=0)
    ws = np.abs(W[:, :2] * s[:2]).max(axis=0)
    assert np.allclose(xs, [2.0, 2.0]) and np.allclose(ws, [2.0, 2.0])
    # alpha = 1 moves all of max|X_j| into the weights, alpha = 0 none of it
    assert np.allclose(O.smooth_factors(X, W, 1.0)[:2], [4.0, 1.0])
    assert np.allclose(O.smooth_factors(X, W, 0.0)[:2], [1.0, 0.25])


def test_smoothing_keeps_the_product_and_tames_outlier_channels():
    """(X / s)(W s)^T = X W^T exactly in fp64, and with activation outliers in
    a few channels the smoothed W4A8 layer is closer to X W^T."""
    rng = np.random.default_rng(12)
    T, K, N = 64, 512, 128
    X = rng.standard_normal((T, K)).astype(np.float32)
    hot = rng.permutation(K)[:8]
    X[:, hot] *= 50.0
    X = _bf16_round(X)
    W = _rand_w(N, K, 13, std=0.05)
    s = O.smooth_factors(X, W, 0.5)
    exact = X.astype(np.float64) @ W.astype(np.float64).T
    moved = (X.astype(np.float64) / s) @ (W.astype(np.float64) * s).T
    assert np.allclose(moved, exact, rtol=1e-12, atol=1e-9)

    def w4a8_error(inv_s, Ws):
        p, sc, _ = O.pack_rtn(Ws.astype(np.float32), K, True)
        qx, sx = O.w4a8_quantize_act(X, K, inv_s=inv_s)
        _, y = O.w4a8_linear(qx, sx, p, sc, None)
        return np.linalg.norm(y - exact) / np.linalg.norm(exact)
    inv_s = (np.float32(1.0) / s.astype(np.float32)).astype(np.float32)
    plain = w4a8_error(None, W)
    smooth = w4a8_error(inv_s, (W * s.astype(np.float32)).astype(np.float32))
    assert smooth < 0.85 * plain, (smooth, plain)      # measured 0.112 vs 0.142


def test_smoothed_act_quant_with_power_of_two_factors():
    """inv_s a power of two: x * inv_s is exact, so the result is the plain
    rule on the exactly scaled activations; inv_s = 1 changes nothing."""
    rng = np.random.default_rng(2)
    x = _bf16_round(rng.standard_normal((3, 64)).astype(np.float32))
    q1, s1 = O.w4a8_quantize_act(x, 64)
    q2, s2 = O.w4a8_quantize_act(x, 64, inv_s=np.ones(64, np.float32))
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
    inv = np.where(np.arange(64) % 2 == 0, 0.25, 4.0).astype(np.float32)
    q3, s3 = O.w4a8_quantize_act(x, 64, inv_s=inv)
    q4, s4 = O.w4a8_quantize_act(_bf16_round(x * inv), 64)
    assert np.array_equal(q3, q4) and np.array_equal(s3, s4)


# ---------------------------------------------------------------------------
# GPTQ ("Lab 5: Gemma4 端到端推理优化", section 从 RTN 到 GPTQ)
# ---------------------------------------------------------------------------

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


@pytest.mark.parametrize("symmetric,G", [(True, 32), (False, 32), (True, 64)])
def test_gptq_loss_identity(symmetric, G):
    """The accumulated L_pred equals 1/2 (w0 - w_hat)^T H (w0 - w_hat) for
    every row: w0 - w_hat = U^T e and U H U^T = I, so the identity holds
    exactly for any codes, and breaks if the update, its sign, the row of U
    or the normalisation is wrong."""
    rng = np.random.default_rng(7)
    N, K, T = 12, 96, 80
    A = rng.standard_normal((K, K)) * 0.3 + np.eye(K)
    X = _bf16_round((rng.standard_normal((T, K)) @ A).astype(np.float32))
    W = _rand_w(N, K, 8, std=0.2)
    codes, scales, zeros, loss, Hd, W0 = O.gptq_quantize(W, X, G, symmetric)
    D = W0 - _dequant(codes, scales, zeros, G)
    quad = 0.5 * np.einsum("nk,kj,nj->n", D, Hd, D)
    assert np.allclose(loss, quad, rtol=1e-9, atol=0)


def test_gptq_with_isotropic_hessian_is_rtn():
    """X a Hadamard matrix (entries +-1, exact in bf16): H = c I, U is
    diagonal, nothing propagates, and GPTQ gives the RTN codes."""
    K = 64
    X = _hadamard(K).astype(np.float32)
    for symmetric in (True, False):
        W = _rand_w(10, K, 3, std=0.2)
        codes, scales, zeros, _, _, _ = O.gptq_quantize(W, X, 32, symmetric)
        rc, rs, rz = O.rtn_quantize(W, 32, symmetric)
        assert np.array_equal(codes, rc) and np.array_equal(scales, rs)
        if not symmetric:
            assert np.array_equal(zeros, rz)


def test_gptq_dead_columns_and_padding():
    """A channel that is zero in every calibration token, and the padded
    columns, have their weights zeroed and dequantize to exactly 0."""
    rng = np.random.default_rng(4)
    N, K, T, G = 6, 80, 64, 32                         # Kp = 96: 16 padded columns
    X = _bf16_round(rng.standard_normal((T, K)).astype(np.float32))
    X[:, 5] = 0.0
    W = _rand_w(N, K, 9, std=0.2)
    for symmetric in (True, False):
        codes, scales, zeros, loss, Hd, W0 = O.gptq_quantize(W, X, G, symmetric)
        Wq = _dequant(codes, scales, zeros, G)
        assert np.all(W0[:, 5] == 0) and np.all(Wq[:, 5] == 0)
        assert np.all(Wq[:, K:] == 0)
        lam = 0.01 * np.mean(np.diag(Hd)) / 1.01        # diag(Hd) = diag(H) + lam
        assert abs(Hd[5, 5] - (1.0 + lam)) < 1e-12       # dead: H_55 = 1 before damping
        assert np.all(np.isfinite(loss))


def test_gptq_beats_rtn_on_the_calibration_objective():
    """||X (W - W_hat)^T||_F is lower than RTN's for correlated activations."""
    rng = np.random.default_rng(21)
    N, K, T = 32, 128, 256
    A = rng.standard_normal((K, K)) * 0.5 + np.eye(K)
    X = _bf16_round((rng.standard_normal((T, K)) @ A).astype(np.float32))
    W = _rand_w(N, K, 22, std=0.05)
    Xd = X.astype(np.float64)
    for symmetric, G in ((True, 32), (False, 128)):
        codes, scales, zeros, _, _, _ = O.gptq_quantize(W, X, G, symmetric)
        rc, rs, rz = O.rtn_quantize(W, G, symmetric)
        err = lambda Wq: np.linalg.norm(Xd @ (W.astype(np.float64) - Wq[:, :K]).T)
        g_err = err(_dequant(codes, scales, zeros, G))
        r_err = err(_dequant(rc, rs, rz, G))
        assert g_err < 0.8 * r_err, (g_err, r_err)


# ---------------------------------------------------------------------------
# bf16 parameter layout: bf16 scales ("Yeniden paketlenmiş QAT Gemma 4 …",
# TPU W4A16 loads scales in bf16) and the (8 - z) s offset ("Lab 5",
# 融合INT4反量化与矩阵乘)
# ---------------------------------------------------------------------------

def test_round_bf16_closed_forms():
    v = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1 + 2 ** -8 + 2 ** -20,
                  3.0, 0.0, -2.5], np.float32)
    r = O.round_bf16(v)
    assert list(r) == [1.0, 1 + 2 ** -6, -1.0, 1 + 2 ** -7, 3.0, 0.0, -2.5]
    assert np.all(r.view(np.uint32) & 0xFFFF == 0)


def test_bf16_params_layout():
    rng = np.random.default_rng(5)
    W = _rand_w(24, 256, 31, std=0.3)
    W[3, :32] = np.abs(W[3, :32])                      # a one-signed group: z at a bound
    for symmetric in (True, False):
        packed, s_b, o_b = O.pack_rtn_bf16(W, 32, symmetric)
        p32, s, z = O.pack_rtn(W, 32, symmetric)
        assert np.array_equal(packed, p32)             # the codes are RTN's
        assert np.all(s_b.view(np.uint32) & 0xFFFF == 0)
        wb = O.dequantize_bf16_params(packed, s_b, o_b, 32)
        wf = O.dequantize_f64(p32, s, z, 32)
        # each stored parameter is within half a bf16 step: 8 significant
        # bits, unit roundoff 2^-8 relative; |code - 8| <= 8
        zz = np.full(s.shape, 8.0) if z is None else z.astype(np.float64)
        bound = 2.0 ** -8 * (8 * np.abs(s) + np.abs((8 - zz) * s)).astype(np.float64)
        assert np.all(np.abs(wb - wf) <= np.repeat(bound, 32, axis=1) * (1 + 1e-6))
        if symmetric:
            assert o_b is None
        else:
            assert np.all(o_b[z == 8] == 0)


def test_bf16_params_exact_for_power_of_two_scales():
    """When every s is a power of two, s_b = s and the offset is exact, so
    the two layouts dequantize identically."""
    rng = np.random.default_rng(6)
    W = rng.integers(-8, 8, size=(8, 64)).astype(np.float32) * 0.25
    W[:, ::32] = -8 * 0.25                              # every group spans -2 .. +1.75
    W[:, 1::32] = 7 * 0.25
    for symmetric in (True, False):
        packed, s_b, o_b = O.pack_rtn_bf16(W, 32, symmetric)
        p32, s, z = O.pack_rtn(W, 32, symmetric)
        if symmetric:
            continue                                    # max/7 is not a power of two
        assert np.array_equal(s_b, s)
        assert np.array_equal(O.dequantize_bf16_params(packed, s_b, o_b, 32),
                              O.dequantize_f64(p32, s, z, 32))


def test_gptq_hessian_closed_form():
    """X a Hadamard matrix (X^T X = T I): H = (2/T) X^T X = 2 I exactly, with
    zero rows and columns for the padded positions."""
    K = 64
    X = _hadamard(K).astype(np.float32)
    H = O.gptq_hessian(X, K)
    assert np.array_equal(H, 2.0 * np.eye(K))
    Hp = O.gptq_hessian(X[:, :48], 64)          # 48 real columns, 16 padded
    assert np.all(Hp[48:, :] == 0) and np.all(Hp[:, 48:] == 0)
    assert np.allclose(np.diag(Hp)[:48], 2.0)


def test_bf16_params_linear_reduces_to_the_linear():
    """With power-of-two scales both layouts describe the same weights, so
    the two linear oracles agree exactly."""
    rng = np.random.default_rng(8)
    W = rng.integers(-8, 8, size=(8, 64)).astype(np.float32) * 0.25
    W[:, ::32] = -2.0
    W[:, 1::32] = 1.75
    x = _bf16_round(rng.standard_normal((3, 64)).astype(np.float32))
    b = rng.standard_normal(8).astype(np.float32)
    packed, s_b, o_b = O.pack_rtn_bf16(W, 32, False)
    p32, s, z = O.pack_rtn(W, 32, False)
    assert np.array_equal(O.w4a16_linear_bf16_params(x, packed, s_b, o_b, b, 64, 32),
                          O.w4a16_linear(x, p32, s, z, b, 64, 32))
