"""CPU oracle for the group-wise INT4 weight-only linear layer (W4A16, W4A8).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
and the CPU-baseline leg of the benchmark may import this module.  It shares
no code, table or helper with the CUDA library; it is written from the pages'
formulas and checked against them by the pins in ``tests/test_oracle_*.py``.

Sources (page title, section):

[P1] "Lab 5: Gemma4 端到端推理优化", section "INT4 线性量化":
     q = clip(round(r/s + z), qmin, qmax), r_hat = s (q - z); one parameter set
     per output channel and per group_size input columns; symmetric codes
     stored as q+8 in [0,15] with s = max|r|/7; asymmetric s = (rmax-rmin)/15,
     z = round(-rmin/s); two codes per uint8, low nibble first; the input
     dimension is padded up to a multiple of group_size and padded positions
     must dequantize to zero.
[P1u] same page, section "量化正确性修正": unpack low and high nibbles
     independently, then interleave.
[P1g] same page, section "从 RTN 到 GPTQ": H = (2/N) X^T X; a dead column
     (zero diagonal) has its weights zeroed and H_ii = 1; then
     H <- H + lambda I, lambda = alpha mean(diag H); H^-1 = U^T U, U upper
     triangular; column i is quantized to q_i, e_i = (w_i - q_i) / U_ii and
     W[:, i:] <- W[:, i:] - e_i U[i, i:]; L_pred = 1/2 sum ||w_i - q_i||^2 / U_ii^2.
     The page's implementation works in FP32.
[P1a] same page, section "融合INT4反量化与矩阵乘": the additive offset of an
     asymmetric group is (8 - z) s when codes are read as (q - 8).
[P1f] same page, section "基础": the feed-forward block is
     W_down [SiLU(W_gate x) (*) (W_up x)] with SiLU(v) = v sigma(v).
[P3] "Yeniden paketlenmiş QAT Gemma 4 26B-A4B, tek bir TPU v6e'de FP8
     işlemenin 1.9 katı verimle sunuluyor", sections "26B'deki boşluk" and
     "vLLM'in TPU backend'inde değişen ne oldu": expert layers
     (128 experts, 8 active per token) whose int4 weights with 32-wide
     groups are multiplied by their tokens in a grouped matmul.
[P2] "【infra之路】12-投机解码、量化与推理引擎对比", section 2.2: symmetric INT8,
     scale = max/127, per-value error <= scale/2.  Section 2.4 (SmoothQuant):
     Y = (X diag(s)^-1)(diag(s) W) with s_j = max|X_j|^a / max|W_j|^(1-a),
     a = 0.5 typically, j an input channel.
[P5] "LLM 模型壓縮與推理加速實踐-陳磊.pdf", W8A8 slides (模型壓縮-W8A8量化): activation
     outliers sit in a few channels; a between 0.5 and 0.75, tuned per layer.
[P4] "Jetson Orin AGX INT4 推理优化实践：super 分支从 9 tok/s 到 24 tok/s",
     section "从 FP 线性层到 INT4 DP4A 的数学推导": per-row INT4 weights
     q^W = clip(round(W/s^W), -8, 7); dynamic per-token INT8 activations
     s^x = max|x|/127, q^x = clip(round(x/s^x), -127, 127);
     acc_j = sum_i q^W_ji q^x_i; y_j = s^W_j s^x acc_j + b_j.
     Section "INT32 accumulator 是否安全": worst case K * 8 * 127.
     Section "DP4A 做了什么": a uint32 holds eight codes [w7 ... w0].

Readings where the pages are silent (each is also listed in the design notes):
 (i)   round() is round-half-to-even (IEEE rint).
 (ii)  r/s, max/7, (rmax-rmin)/15, -rmin/s and r/s + z are each one IEEE
       fp32 operation with round-to-nearest-even (no reciprocal, no fusion).
 (iv)  padded positions take part in the group statistics as zeros.
 (v)   asymmetric: rmin = min(0, min r), rmax = max(0, max r), so z is in
       [0, 15] and 0 is exactly representable.
 (vi)  an all-zero group stores s = 0 (and z = 0); its codes are 8 (sym) or
       0 (asym) and dequantize to exactly 0; no division by zero happens.
 (ix)  fused gate|up weights: 16-row tiles of 8 gate rows then the same 8
       up rows (gate row f at 16 (f // 8) + f % 8, up row f 8 rows below);
       the bias of each projection is added before SiLU and the product.
 (x)   grouped linear: tokens arrive sorted by group with offsets
       goff[0] = 0 <= ... <= goff[E] = T; group e's weights are rows
       e N .. e N + N - 1 of the stacked matrix, its bias the same rows.
 (xi)  smoothing: channel maxima over the calibration tokens and over the
       output rows; a channel whose activation or weight maximum is 0 gets
       s = 1.  At inference x' = fp32(x * fp32(1 / s)) (one rounding each),
       then the INT8 rule of [P4] on x'.
 (xii) group-wise W4A8: acc_g = sum over the group's columns of
       (code - 8) q_x in integers; y = s_x * sum_g s_W[n, g] acc_g + b.
 (xiii) GPTQ: a group's parameters are fixed when the loop reaches the
       group's first column, from the group's current (already updated)
       weights, by the RTN rule; alpha (the damping ratio) defaults to 0.01;
       the padded columns K..Kp-1 are dead columns.  The oracle propagates
       in fp64 and takes every rounding decision by the fp32 rule, from the
       fp32 value of the current weight.
 (xiv) bf16 parameter layout: the codes are the RTN codes; the stored
       scale is bf16(s) and, for asymmetric groups, the stored offset is
       bf16(fp32((8 - z) s)) (round to nearest even each time);
       w_hat = s_b (code - 8) + o_b.
 (viii) the W4A8 weight scale is max|row|/7 (the symmetric rule of [P1]),
       codes stored as q+8 like W4A16.
 Matmuls are done in fp64 on exactly dequantized weights (s * (code - z) is
 exact in fp64), the W4A8 dot product in int64.

Functions that have no pin of their own: none (see the pins' module).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def padded_k(K: int, group_size: int) -> int:
    """K rounded up to a multiple of group_size [P1]."""
    return -(-K // group_size) * group_size


# ---------------------------------------------------------------------------
# Quantise [P1], readings (i), (ii), (iv)-(vi)
# ---------------------------------------------------------------------------

def rtn_params(R, symmetric: bool):
    """Group parameters of the last axis of R (fp32 [..., G]), readings
    (ii), (v), (vi): symmetric s = fp32(max|r| / 7), z = 8 (returned as
    None); asymmetric s = fp32((rmax - rmin) / 15) over the range widened to
    hold 0, z = rint(fp32(-rmin / s)) in [0, 15]; an all-zero group has s = 0
    (and z = 0)."""
    R = np.asarray(R, dtype=F32)
    if symmetric:
        maxabs = np.abs(R).max(axis=-1)             # exact in fp32
        return (maxabs / F32(7.0)).astype(F32), None
    rmin = np.minimum(R.min(axis=-1), F32(0.0))     # (v)
    rmax = np.maximum(R.max(axis=-1), F32(0.0))
    s = ((rmax - rmin).astype(F32) / F32(15.0)).astype(F32)
    nz = s != 0
    s_div = np.where(nz, s, F32(1.0)).astype(F32)
    z = np.clip(np.rint((-rmin) / s_div), 0, 15).astype(F32)
    z = np.where(nz, z, F32(0.0)).astype(F32)       # (vi)
    return s, z


def rtn_codes(R, s, z, symmetric: bool):
    """Codes in [0, 15] of fp32 values R [..., G] under group parameters s
    (and z) with one entry per group (the last axis of R is the group):
    symmetric q = clip(rint(fp32(r / s)), -8, 7) + 8, asymmetric
    q = clip(rint(fp32(fp32(r / s) + z)), 0, 15); 8 or 0 where s = 0."""
    R = np.asarray(R, dtype=F32)
    nz = s != 0
    s_div = np.where(nz, s, F32(1.0)).astype(F32)[..., None]
    if symmetric:
        q = np.clip(np.rint((R / s_div).astype(F32)), -8, 7)   # fp32 r/s, then rint (i)
        q = np.where(nz[..., None], q, 0)
        return (q + 8).astype(np.uint8)
    t = ((R / s_div).astype(F32) + z[..., None]).astype(F32)  # fp32 add
    q = np.clip(np.rint(t), 0, 15)
    q = np.where(nz[..., None], q, 0)
    return q.astype(np.uint8)


def rtn_quantize(W, group_size: int, symmetric: bool):
    """Round-to-nearest INT4 quantisation of W [N, K] (fp32).

    Returns (codes uint8 [N, Kp] in [0, 15], scales fp32 [N, Ng],
    zeros uint8 [N, Ng] or None when symmetric)."""
    W = np.asarray(W, dtype=F32)
    N, K = W.shape
    G = int(group_size)
    Kp = padded_k(K, G)
    Ng = Kp // G
    Wp = np.zeros((N, Kp), dtype=F32)
    Wp[:, :K] = W                                   # (iv) pads are zeros
    R = Wp.reshape(N, Ng, G)
    s, z = rtn_params(R, symmetric)
    codes = rtn_codes(R, s, z, symmetric)
    return codes.reshape(N, Kp), s, None if symmetric else z.astype(np.uint8)


# ---------------------------------------------------------------------------
# Pack / unpack [P1], [P1u], [P4] "DP4A 做了什么"
# ---------------------------------------------------------------------------

def pack_nibbles(codes):
    """Two codes per byte: column 2j in bits 0-3, column 2j+1 in bits 4-7."""
    codes = np.asarray(codes, dtype=np.uint8)
    even = codes[:, 0::2].astype(np.uint16)
    odd = codes[:, 1::2].astype(np.uint16)
    return (even | (odd << 4)).astype(np.uint8)


def unpack_nibbles(packed):
    """Inverse of pack_nibbles.  Low and high nibbles are computed from the
    packed bytes first and written into a fresh array [P1u]."""
    packed = np.asarray(packed, dtype=np.uint8)
    N, B = packed.shape
    out = np.empty((N, 2 * B), dtype=np.uint8)
    low = packed & np.uint8(0x0F)
    high = packed >> np.uint8(4)
    out[:, 0::2] = low
    out[:, 1::2] = high
    return out


def pack_rtn(W, group_size: int, symmetric: bool):
    """What w4_pack_rtn returns: (packed uint8 [N, Kp/2], scales fp32
    [N, Ng], zeros uint8 [N, Ng] or None)."""
    codes, s, z = rtn_quantize(W, group_size, symmetric)
    return pack_nibbles(codes), s, z


# ---------------------------------------------------------------------------
# Dequantise and matmul in fp64 [P1]
# ---------------------------------------------------------------------------

def round_bf16(a):
    """fp32 values rounded to the nearest bf16 (ties to even), as fp32."""
    b = np.asarray(a, dtype=F32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return (r & 0xFFFFFFFF).astype(np.uint32).view(F32)


def pack_rtn_bf16(W, group_size: int, symmetric: bool):
    """RTN codes with bf16 parameters, reading (xiv) ([P1a] offset (8 - z) s;
    [P3] bf16 scales): returns (packed, s_b fp32 [N, Ng] holding bf16
    values, o_b likewise or None when symmetric)."""
    codes, s, z = rtn_quantize(W, group_size, symmetric)
    s_b = round_bf16(s)
    o_b = None
    if not symmetric:
        o_b = round_bf16((F32(8.0) - z.astype(F32)) * s)      # fp32 product, then bf16
    return pack_nibbles(codes), s_b, o_b


def dequantize_bf16_params(packed, s_b, o_b, group_size: int, rows=None):
    """w_hat = s_b (code - 8) + o_b in fp64 (exact for bf16 s_b, o_b)."""
    packed = np.asarray(packed)
    s_b = np.asarray(s_b, dtype=F32)
    if rows is not None:
        rows = np.asarray(rows)
        packed, s_b = packed[rows], s_b[rows]
        o_b = None if o_b is None else np.asarray(o_b)[rows]
    codes = unpack_nibbles(packed).astype(np.float64)
    N, Kp = codes.shape
    G = int(group_size)
    Ng = Kp // G
    w = s_b.astype(np.float64)[:, :, None] * (codes.reshape(N, Ng, G) - 8.0)
    if o_b is not None:
        w = w + np.asarray(o_b, dtype=F32).astype(np.float64)[:, :, None]
    return w.reshape(N, Kp)


def w4a16_linear_bf16_params(x, packed, s_b, o_b, bias, K: int, group_size: int, rows=None):
    """w4a16_linear with the bf16 parameter layout, reading (xiv)."""
    xd = bf16_to_f64(x)
    Wd = dequantize_bf16_params(packed, s_b, o_b, group_size, rows=rows)[:, :K]
    y = xd @ Wd.T
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        y = y + (b if rows is None else b[np.asarray(rows)])[None, :]
    return y


def dequantize_f64(packed, scales, zeros, group_size: int, rows=None):
    """W_hat[n, k] = s[n, k // G] * (code[n, k] - z[n, k // G]) in fp64, with
    z = 8 for symmetric groups.  Exact: s is fp32 and code - z a small
    integer.  ``rows`` selects output channels (all when None)."""
    packed = np.asarray(packed)
    scales = np.asarray(scales, dtype=F32)
    if rows is not None:
        rows = np.asarray(rows)
        packed = packed[rows]
        scales = scales[rows]
        zeros = None if zeros is None else np.asarray(zeros)[rows]
    codes = unpack_nibbles(packed).astype(np.float64)
    N, Kp = codes.shape
    G = int(group_size)
    Ng = Kp // G
    if zeros is None:
        zf = np.full((N, Ng), 8.0)
    else:
        zf = np.asarray(zeros, dtype=np.float64)
    sf = scales.astype(np.float64)
    c3 = codes.reshape(N, Ng, G)
    return (sf[:, :, None] * (c3 - zf[:, :, None])).reshape(N, Kp)


def bf16_to_f64(x):
    """Accepts a torch bf16 tensor, or an fp32 array holding bf16 values,
    and returns the exact fp64 values."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu").float().numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x, dtype=F32)
    if np.any(x.view(np.uint32) & np.uint32(0xFFFF)):
        raise ValueError("activations are not bf16 values")
    return x.astype(np.float64)


def w4a16_linear(x, packed, scales, zeros, bias, K: int, group_size: int,
                 rows=None):
    """y[m, n] = sum_{k<K} x[m, k] * W_hat[n, k] + b[n] in fp64.

    ``x`` holds bf16 values [M, K].  ``rows`` restricts the output channels
    computed (returns y[:, rows]).  The contraction is a library fp64 matmul
    of the exactly dequantised weights."""
    xd = bf16_to_f64(x)
    Wd = dequantize_f64(packed, scales, zeros, group_size, rows=rows)[:, :K]
    y = xd @ Wd.T
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        y = y + (b if rows is None else b[np.asarray(rows)])[None, :]
    return y


# ---------------------------------------------------------------------------
# Fused gate|up projection with SiLU [P1f], reading (ix)
# ---------------------------------------------------------------------------

def swiglu_rows(F: int):
    """(gate_rows, up_rows) of the fused [2F] weight matrix, reading (ix)."""
    f = np.arange(F)
    gate = 16 * (f // 8) + f % 8
    return gate, gate + 8


def pair_rows(gate, up):
    """Stack two [F, ...] arrays into the fused [2F, ...] order of reading
    (ix): out[gate_rows] = gate, out[up_rows] = up."""
    gate = np.asarray(gate)
    up = np.asarray(up)
    F = gate.shape[0]
    if up.shape != gate.shape or F % 8:
        raise ValueError("gate and up need equal shapes and F % 8 == 0")
    g_idx, u_idx = swiglu_rows(F)
    out = np.empty((2 * F,) + gate.shape[1:], dtype=gate.dtype)
    out[g_idx] = gate
    out[u_idx] = up
    return out


def silu_f64(v):
    """SiLU(v) = v sigma(v) in fp64 [P1f]; sigma is evaluated on the side
    where exp does not overflow."""
    v = np.asarray(v, dtype=np.float64)
    e = np.exp(-np.abs(v))
    sig = np.where(v >= 0, 1.0 / (1.0 + e), e / (1.0 + e))
    return v * sig


def w4a16_linear_swiglu(x, packed, scales, zeros, bias, F: int, K: int,
                        group_size: int, cols=None):
    """y[m, f] = SiLU(g[m, f]) * u[m, f] in fp64, where g and u are the
    W4A16 linear outputs (bias included) of gate row f and up row f of the
    fused matrix.  ``cols`` restricts the f computed."""
    g_idx, u_idx = swiglu_rows(F)
    if cols is not None:
        cols = np.asarray(cols)
        g_idx, u_idx = g_idx[cols], u_idx[cols]
    g = w4a16_linear(x, packed, scales, zeros, bias, K, group_size, rows=g_idx)
    u = w4a16_linear(x, packed, scales, zeros, bias, K, group_size, rows=u_idx)
    return silu_f64(g) * u


# ---------------------------------------------------------------------------
# GPTQ [P1g], reading (xiii)
# ---------------------------------------------------------------------------

def gptq_hessian(X, Kp: int):
    """H = (2 / T) X^T X in fp64 for calibration activations X [T, K]
    (bf16 values), padded with zero columns to Kp."""
    Xd = bf16_to_f64(X)
    T, K = Xd.shape
    Xp = np.zeros((T, Kp))
    Xp[:, :K] = Xd
    return (2.0 / T) * (Xp.T @ Xp)


def gptq_quantize(W, X, group_size: int, symmetric: bool, damp: float = 0.01):
    """GPTQ of W [N, K] (fp32) with calibration X [T, K] (bf16 values), in
    the page's order: Hessian, dead columns, damping, U with H^-1 = U^T U,
    then column by column quantize, normalise the error and update the
    remaining columns.  Library primitives: the fp64 inverse and Cholesky.

    Returns (codes uint8 [N, Kp], scales fp32 [N, Ng], zeros uint8 [N, Ng]
    or None, loss fp64 [N] (L_pred per row), Hd fp64 [Kp, Kp] the damped
    Hessian that was factorized, W0 fp64 [N, Kp] the weights after the
    dead-column step)."""
    W = np.asarray(W, dtype=F32)
    N, K = W.shape
    G = int(group_size)
    Kp = padded_k(K, G)
    Ng = Kp // G
    Wc = np.zeros((N, Kp))
    Wc[:, :K] = W
    H = gptq_hessian(X, Kp)
    dead = np.diag(H) == 0
    H[dead, dead] = 1.0
    Wc[:, dead] = 0.0
    H = H + damp * np.mean(np.diag(H)) * np.eye(Kp)
    U = np.linalg.cholesky(np.linalg.inv(H)).T      # H^-1 = L L^T, U = L^T
    W0 = Wc.copy()
    codes = np.zeros((N, Kp), dtype=np.uint8)
    scales = np.zeros((N, Ng), dtype=F32)
    zeros = None if symmetric else np.zeros((N, Ng), dtype=np.uint8)
    loss = np.zeros(N)
    for i in range(Kp):
        g = i // G
        if i % G == 0:                               # (xiii) the group's parameters
            sg, zg = rtn_params(Wc[:, i:i + G].astype(F32), symmetric)
            scales[:, g] = sg
            if not symmetric:
                zeros[:, g] = zg.astype(np.uint8)
        sg = scales[:, g]
        zg = None if symmetric else zeros[:, g].astype(F32)
        c = rtn_codes(Wc[:, i:i + 1].astype(F32), sg, zg, symmetric)[:, 0]
        codes[:, i] = c
        zq = 8.0 if symmetric else zg.astype(np.float64)
        q = sg.astype(np.float64) * (c.astype(np.float64) - zq)     # dequantized q_i
        d = Wc[:, i] - q
        loss += 0.5 * d * d / U[i, i] ** 2
        e = d / U[i, i]
        Wc[:, i:] -= np.outer(e, U[i, i:])
    return codes, scales, zeros, loss, H, W0


# ---------------------------------------------------------------------------
# Grouped linear (experts) [P3], reading (x)
# ---------------------------------------------------------------------------

def w4a16_grouped_linear(x, goff, packed, scales, zeros, bias, E: int, N: int, K: int,
                         group_size: int, cols=None):
    """y[t, n] = sum_k x[t, k] W_hat_e[n, k] + b_e[n] for the group e with
    goff[e] <= t < goff[e+1], in fp64: each group's rows through
    w4a16_linear with that group's slice of the stacked weights.  ``cols``
    restricts the output columns n computed."""
    goff = np.asarray(goff, dtype=np.int64)
    T = np.asarray(x).shape[0] if not hasattr(x, "shape") else x.shape[0]
    if goff.shape != (E + 1,) or goff[0] != 0 or goff[-1] != T or np.any(np.diff(goff) < 0):
        raise ValueError("group offsets must rise from 0 to T")
    packed = np.asarray(packed).reshape(E, N, -1)
    scales = np.asarray(scales, dtype=F32).reshape(E, N, -1)
    zeros = None if zeros is None else np.asarray(zeros).reshape(E, N, -1)
    bias = None if bias is None else np.asarray(bias, dtype=np.float64).reshape(E, N)
    ncol = N if cols is None else len(cols)
    y = np.zeros((T, ncol))
    for e in range(E):
        t0, t1 = int(goff[e]), int(goff[e + 1])
        if t1 == t0:
            continue
        y[t0:t1] = w4a16_linear(x[t0:t1], packed[e], scales[e],
                                None if zeros is None else zeros[e],
                                None if bias is None else bias[e], K, group_size, rows=cols)
    return y


# ---------------------------------------------------------------------------
# W4A8 [P4]
# ---------------------------------------------------------------------------

def w4a8_quantize_act(x, Kp: int, inv_s=None):
    """Per-token dynamic INT8: s_x = fp32(max|x| / 127),
    q_x = clip(rint(fp32(x / s_x)), -127, 127); columns K..Kp-1 are 0.
    With ``inv_s`` (fp32 [K], reading (xi)) x is first smoothed:
    x' = fp32(x * inv_s).  Returns (qx int8 [M, Kp], sx fp32 [M])."""
    xf = bf16_to_f64(x).astype(F32)
    if inv_s is not None:
        xf = (xf * np.asarray(inv_s, dtype=F32)[None, :]).astype(F32)
    M, K = xf.shape
    maxabs = np.abs(xf).max(axis=1) if K > 0 else np.zeros(M, F32)
    sx = (maxabs.astype(F32) / F32(127.0)).astype(F32)
    nz = sx != 0
    s_div = np.where(nz, sx, F32(1.0)).astype(F32)
    q = np.clip(np.rint((xf / s_div[:, None]).astype(F32)), -127, 127)
    q = np.where(nz[:, None], q, 0)
    qx = np.zeros((M, Kp), dtype=np.int8)
    qx[:, :K] = q.astype(np.int8)
    return qx, sx


def smooth_factors(X, W, alpha: float):
    """SmoothQuant factors [P2] 2.4, reading (xi), in fp64:
    s_j = max_t |X[t, j]|^alpha / max_n |W[n, j]|^(1 - alpha), and 1 where
    either maximum is 0.  X: calibration activations [T, K] (bf16 values),
    W: fp32 [N, K]."""
    xm = np.abs(bf16_to_f64(X)).max(axis=0)
    wm = np.abs(np.asarray(W, dtype=np.float64)).max(axis=0)
    ok = (xm > 0) & (wm > 0)
    s = np.ones_like(xm)
    s[ok] = xm[ok] ** alpha / wm[ok] ** (1.0 - alpha)
    return s


def w4a8_linear_grouped(qx, sx, packed, scales, group_size: int, bias=None, rows=None):
    """Group-wise W4A8, reading (xii): per (token, row, group) the integer
    acc_g = sum_{k in g} (code - 8) q_x, then
    y = s_x * sum_g s_W[n, g] * acc_g + b in fp64.  Returns (acc [M, N, Ng]
    int64, y fp64 [M, N])."""
    packed = np.asarray(packed)
    scales = np.asarray(scales, dtype=F32)
    if rows is not None:
        rows = np.asarray(rows)
        packed = packed[rows]
        scales = scales[rows]
    q = unpack_nibbles(packed).astype(np.int64) - 8           # [N, Kp]
    N, Kp = q.shape
    G = int(group_size)
    Ng = Kp // G
    qx64 = np.asarray(qx, dtype=np.int64)                     # [M, Kp]
    acc = np.einsum("mgk,ngk->mng", qx64.reshape(-1, Ng, G), q.reshape(N, Ng, G))
    y = np.asarray(sx, np.float64)[:, None] * (acc.astype(np.float64)
                                                * scales.astype(np.float64)[None]).sum(axis=2)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        y = y + (b if rows is None else b[rows])[None, :]
    return acc, y


def w4a8_linear(qx, sx, packed, w_scales, bias, rows=None):
    """acc[m, n] = sum_k (code[n, k] - 8) * qx[m, k] over all Kp columns, in
    int64; y = s_W[n] * s_x[m] * acc + b[n] in fp64.  Per-row weight scale
    (one group spanning the padded row).  Returns (acc int64, y fp64)."""
    packed = np.asarray(packed)
    ws = np.asarray(w_scales, dtype=F32).reshape(packed.shape[0], -1)
    if ws.shape[1] != 1:
        raise ValueError("w4a8 oracle takes one weight scale per row")
    ws = ws[:, 0]
    if rows is not None:
        rows = np.asarray(rows)
        packed = packed[rows]
        ws = ws[rows]
    q = unpack_nibbles(packed).astype(np.int64) - 8
    qx64 = np.asarray(qx, dtype=np.int64)
    acc = qx64 @ q.T
    y = (ws.astype(np.float64)[None, :] * np.asarray(sx, np.float64)[:, None]
         * acc.astype(np.float64))
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        y = y + (b if rows is None else b[rows])[None, :]
    return acc, y


def int32_worst_case(K: int) -> int:
    """Largest |acc| of an INT4 x INT8 dot product of length K [P4]:
    |q^W| <= 8 and |q^x| <= 127."""
    return K * 8 * 127
