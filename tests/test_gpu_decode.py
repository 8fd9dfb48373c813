"""GPU parity of the decode path (M <= 16) and of the quantizer, through the
C ABI, against the CPU oracle on identical seeded inputs."""
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


def _pack_both(w4, W_cpu, G, sym):
    """GPU pack and oracle pack of the same fp32 weights; asserts bit-exact."""
    p, s, z = w4.w4_pack_rtn(W_cpu.cuda(), G, sym)
    op, os_, oz = O.pack_rtn(W_cpu.numpy(), G, sym)
    assert np.array_equal(to_np(p), op), "packed codes differ"
    assert np.array_equal(to_np(s).view(np.uint32), os_.view(np.uint32)), "scales differ"
    if not sym:
        assert np.array_equal(to_np(z), oz), "zero points differ"
    else:
        assert z is None
    return (p, s, z), (op, os_, oz)


def _sample_rows(N, seed, n=1024):
    if N <= 4096:
        return None
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([rng.choice(N, n, replace=False), [0, N - 1]]))
    return rows


def _run_linear(w4, lin, M=None):
    inp = WL.make_inputs(lin, M)
    (p, s, z), (op, os_, oz) = _pack_both(w4, inp.W, lin.group_size, lin.symmetric)
    b = inp.bias.cuda() if inp.bias is not None else None
    y = w4.w4a16_linear(inp.x.cuda(), p, s, z, b, lin.N, lin.K, lin.group_size)
    torch.cuda.synchronize()
    rows = _sample_rows(lin.N, lin.seed)
    yref = O.w4a16_linear(inp.x, op, os_, oz,
                          None if inp.bias is None else inp.bias.numpy(),
                          lin.K, lin.group_size, rows=rows)
    yg = y if rows is None else y[:, torch.as_tensor(rows, device=y.device)]
    return assert_close(yg, yref, lin.name)


# ---------------------------------------------------------------- quantizer
@pytest.mark.parametrize("N,K,G,sym,wout", [
    (256, 512, 32, True, 0.0), (300, 100, 32, False, 0.0), (64, 3580, 128, True, 0.0),
    (1000, 3840, 32, False, 0.01), (129, 1000, 96, True, 0.0), (33, 18944, 18944, True, 0.0),
    (37888, 3584, 128, True, 0.0),
])
def test_pack_rtn_bit_exact(w4, N, K, G, sym, wout):
    lin = WL.Linear("pack", 1, N, K, G, sym, seed=N + K + G, w_outlier_frac=wout)
    inp = WL.make_inputs(lin)
    _pack_both(w4, inp.W, G, sym)


def test_pack_rtn_zero_groups(w4):
    W = torch.zeros(8, 96)
    W[3, 40] = 0.25
    for sym in (True, False):
        _pack_both(w4, W, 32, sym)


# ---------------------------------------------------------------- W4A16 decode
@pytest.mark.parametrize("lin", WL.tiny() + WL.decode_7b() + WL.padding_w4a16(),
                         ids=lambda l: l.name)
def test_decode_workloads(w4, lin):
    _run_linear(w4, lin)


@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_decode_12b_asym(w4, M):
    for lin in WL.decode_12b(M):
        _run_linear(w4, lin)


@pytest.mark.parametrize("M,N,K,G,sym", [
    (1, 1, 32, 32, True), (1, 7, 96, 32, False), (3, 200, 100, 32, True),
    (5, 129, 512, 64, False), (8, 256, 4096, 128, True), (9, 300, 1000, 96, True),
    (16, 384, 8192, 128, False), (2, 128, 16384, 256, True), (1, 64, 3584, 3584, True),
    (15, 640, 768, 32, False), (16, 1000, 256, 32, True), (1, 130, 40960, 128, False),
])
def test_decode_edge_shapes_random_codes(w4, M, N, K, G, sym):
    """Arbitrary codes (including 0, i.e. q = -8), ragged N and K, odd group
    sizes, split-K shapes, with bias."""
    seed = M * 7 + N * 3 + K + G
    packed, scales, zeros = WL.make_random_format(N, K, G, sym, seed)
    x = WL.make_activations(K, M, seed + 1)
    b = torch.randn(N, generator=torch.Generator().manual_seed(seed + 2)) * 0.1
    y = w4.w4a16_linear(x.cuda(), packed.cuda(), scales.cuda(),
                        None if zeros is None else zeros.cuda(), b.cuda(), N, K, G)
    torch.cuda.synchronize()
    yref = O.w4a16_linear(x, packed.numpy(), scales.numpy(),
                          None if zeros is None else zeros.numpy(), b.numpy(), K, G)
    assert_close(y, yref, f"M{M} N{N} K{K} G{G} sym{sym}")
    # deterministic: a second call gives the same bits
    y2 = w4.w4a16_linear(x.cuda(), packed.cuda(), scales.cuda(),
                         None if zeros is None else zeros.cuda(), b.cuda(), N, K, G)
    assert torch.equal(y, y2)


def test_decode_split_k_workspace_errors(w4):
    """A split-K shape refuses a missing or short workspace."""
    N, K, G = 128, 16384, 128
    need = w4.w4a16_workspace_bytes(1, N, K, G)
    assert need > 0
    packed, scales, _ = WL.make_random_format(N, K, G, True, 5)
    x = WL.make_activations(K, 1, 6).cuda()
    short = torch.zeros(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_linear(x, packed.cuda(), scales.cuda(), None, None, N, K, G, workspace=short)
    assert e.value.code == -6


def test_no_device_error_left(w4):
    assert w4.w4_get_device_error() == 0


# ---------------------------------------------------------------- W4A8
@pytest.mark.parametrize("M,K,G,frac", [(1, 3584, 3584, 0.005), (1, 3580, 3584, 0.005),
                                        (16, 1000, 1024, 0.0), (3, 18944, 18944, 0.005),
                                        (2, 40000, 40000, 0.005), (3, 8000, 8448, 0.0),
                                        (4, 100, 128, 0.0), (2, 1001, 1024, 0.01)])
def test_act_quant_bit_exact(w4, M, K, G, frac):
    x = WL.make_activations(K, M, seed=M + K, outlier_frac=frac)
    x[0, :3] = 0                      # keep a few exact zeros in play
    qx, sx = w4.w4a8_quantize_act(x.cuda(), G)
    oq, osx = O.w4a8_quantize_act(x, O.padded_k(K, G))
    assert np.array_equal(to_np(sx).view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(to_np(qx), oq)


@pytest.mark.parametrize("vmax", [1.0, 3.140625, 100.0, 0.0078125, 1e-38])
def test_act_quant_every_bf16_value(w4, vmax):
    """Every bf16 value v with |v| <= vmax, both signs, in rows of 16384
    columns that each also hold vmax (so s_x = fp32(vmax / 127) in every
    row): q_x bit-exact against the oracle's IEEE division, including the
    values whose quotient lies next to a half-integer."""
    top = int(np.array([vmax], np.float32).view(np.uint32)[0] >> 16)
    bits = np.arange(0, top + 1, dtype=np.uint32)
    vals = np.concatenate([bits, bits | 0x8000]).astype(np.uint32) << 16
    vals = vals.view(np.float32)
    K = 16384
    per = K - 1
    rows = -(-len(vals) // per)
    x = np.zeros((rows, K), np.float32)
    x[:, 0] = vmax
    flat = np.zeros(rows * per, np.float32)
    flat[:len(vals)] = vals
    x[:, 1:] = flat.reshape(rows, per)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    qx, sx = w4.w4a8_quantize_act(xt.cuda(), K)
    oq, osx = O.w4a8_quantize_act(xt, K)
    assert np.array_equal(to_np(sx).view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(to_np(qx), oq)


def test_act_quant_ties(w4):
    """s_x = 1 exactly: x = k + 1/2 are ties of the INT8 grid (half to even)."""
    x = torch.zeros(2, 256)
    x[0, 0] = 127.0
    x[0, 1:9] = torch.tensor([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, -126.5])
    x[1] = torch.linspace(-3, 3, 256)
    x = x.to(torch.bfloat16)
    qx, sx = w4.w4a8_quantize_act(x.cuda(), 256)
    oq, osx = O.w4a8_quantize_act(x, 256)
    assert list(oq[0, 1:9]) == [0, 2, 2, 0, -2, -2, 126, -126]
    assert np.array_equal(to_np(qx), oq) and np.array_equal(to_np(sx), osx)


def test_act_quant_zero_token(w4):
    x = torch.zeros(2, 64, dtype=torch.bfloat16)
    x[1, 5] = 1.0
    qx, sx = w4.w4a8_quantize_act(x.cuda(), 64)
    oq, osx = O.w4a8_quantize_act(x, 64)
    assert np.array_equal(to_np(qx), oq) and np.array_equal(to_np(sx), osx)


def _run_w4a8(w4, lin, M=None):
    inp = WL.make_inputs(lin, M)
    (p, s, _), (op, os_, _) = _pack_both(w4, inp.W, lin.group_size, True)
    qx, sx = w4.w4a8_quantize_act(inp.x.cuda(), lin.group_size)
    oq, osx = O.w4a8_quantize_act(inp.x, O.padded_k(lin.K, lin.group_size))
    assert np.array_equal(to_np(qx), oq)
    b = inp.bias.cuda() if inp.bias is not None else None
    y, acc = w4.w4a8_linear(qx, sx, p, s, b, lin.N, lin.K, lin.group_size, want_acc=True)
    torch.cuda.synchronize()
    oacc, oy = O.w4a8_linear(oq, osx, op, os_, None if inp.bias is None else inp.bias.numpy())
    assert np.all(np.abs(oacc) < 2 ** 31)
    assert np.array_equal(to_np(acc).astype(np.int64), oacc), f"{lin.name}: int32 acc differs"
    assert_close(y, oy, lin.name)


@pytest.mark.parametrize("lin", WL.w4a8_7b(), ids=lambda l: l.name)
def test_w4a8_workloads(w4, lin):
    _run_w4a8(w4, lin)


@pytest.mark.parametrize("M,N,K", [(2, 100, 64), (5, 300, 1000), (16, 129, 4096), (4, 2000, 2048)])
def test_w4a8_edge_shapes(w4, M, N, K):
    G = O.padded_k(K, 32)
    lin = WL.Linear("w4a8_edge", M, N, K, G, True, seed=M + N + K, bias=True,
                    x_outlier_frac=0.01, kind="w4a8")
    _run_w4a8(w4, lin)


def test_w4a8_int32_worst_case(w4):
    """All codes 0 (q = -8) and all q_x = 127 at K = 18944: the accumulator
    must be exactly -8 * 127 * K (page 'Jetson Orin AGX INT4 推理优化实践',
    INT32 accumulator 是否安全)."""
    N, K = 256, 18944
    packed = torch.zeros(N, K // 2, dtype=torch.uint8, device="cuda")
    qx = torch.full((1, K), 127, dtype=torch.int8, device="cuda")
    sx = torch.ones(1, device="cuda")
    ws = torch.ones(N, device="cuda")
    y, acc = w4.w4a8_linear(qx, sx, packed, ws, None, N, K, K, want_acc=True)
    assert torch.all(acc == -8 * 127 * K)
    oacc, _ = O.w4a8_linear(to_np(qx), np.ones(1, np.float32), to_np(packed),
                            np.ones(N, np.float32), None)
    assert np.array_equal(to_np(acc).astype(np.int64), oacc)


def test_workspace_shared_by_shapes(w4, monkeypatch):
    """One zero-filled workspace serves split-K calls of different shapes.
    The arrival counters live in a fixed prefix, so the partial sums of a
    call with few row blocks (N = 512: 4 blocks of 128 rows) never land
    where a call with many row blocks (N = 12288: 96 blocks) keeps its
    counters; the calls alternate twice on the same buffer."""
    monkeypatch.setenv("W4_GEMV_ROWS", "128")
    monkeypatch.setenv("W4_GEMV_SPLIT", "4")
    shapes = [(1, 512, 8192, 128, True), (8, 12288, 2048, 32, False)] * 2
    need = max(w4.w4a16_workspace_bytes(M, N, K, G) for M, N, K, G, _ in shapes)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for i, (M, N, K, G, sym) in enumerate(shapes):
        packed, scales, zeros = WL.make_random_format(N, K, G, sym, 50 + i)
        x = WL.make_activations(K, M, 60 + i)
        zc = None if zeros is None else zeros.cuda()
        y = w4.w4a16_linear(x.cuda(), packed.cuda(), scales.cuda(), zc, None, N, K, G,
                            workspace=ws)
        torch.cuda.synchronize()
        rows = np.arange(N) if N <= 1024 else np.unique(np.concatenate(
            [np.arange(0, N, 97), np.arange(N - 1024, N, 5)]))
        yref = O.w4a16_linear(x, packed.numpy()[rows], scales.numpy()[rows],
                              None if zeros is None else zeros.numpy()[rows], None, K, G)
        assert_close(y[:, torch.as_tensor(rows, device=y.device)], yref, f"call {i} N{N}")
    assert w4.w4_get_device_error() == 0


@pytest.mark.parametrize("xtma", ["0", "1"])
@pytest.mark.parametrize("M,N,K,G,sym", [(1, 4608, 3584, 128, True), (8, 640, 3840, 32, False),
                                         (3, 1000, 18944, 128, True)])
def test_decode_activation_staging_paths(w4, monkeypatch, xtma, M, N, K, G, sym):
    """Activations read from global memory by the consumer threads
    (W4_GEMV_XTMA=0, the default of the fp16 loop) or first copied into
    shared memory by a bulk TMA copy (=1, the default of the bf16 loop):
    same tolerance, same bits for both."""
    monkeypatch.setenv("W4_GEMV_XTMA", xtma)
    seed = M + N + K + G
    packed, scales, zeros = WL.make_random_format(N, K, G, sym, seed)
    x = WL.make_activations(K, M, seed + 1)
    zc = None if zeros is None else zeros.cuda()
    y = w4.w4a16_linear(x.cuda(), packed.cuda(), scales.cuda(), zc, None, N, K, G)
    torch.cuda.synchronize()
    yref = O.w4a16_linear(x, packed.numpy(), scales.numpy(),
                          None if zeros is None else zeros.numpy(), None, K, G)
    assert_close(y, yref, f"xtma{xtma} M{M} N{N} K{K}")
    monkeypatch.setenv("W4_GEMV_XTMA", "1" if xtma == "0" else "0")
    y2 = w4.w4a16_linear(x.cuda(), packed.cuda(), scales.cuda(), zc, None, N, K, G)
    assert torch.equal(y, y2), "the two staging paths differ"


@pytest.mark.parametrize("f16", ["0", "1"])
@pytest.mark.parametrize("csplit", ["0", "1"])
@pytest.mark.parametrize("M,N,K,G,sym,split", [
    (1, 1024, 8192, 128, True, "4"),       # 7B-down-like, one token
    (2, 520, 7680, 64, False, "3"),        # asymmetric, ragged rows
    (8, 640, 15360, 128, True, "8"),       # eight splits: the largest cluster
    (16, 384, 8192, 128, False, "2"),      # two token tiles
])
def test_decode_inner_loops_and_split_handoffs(w4, monkeypatch, f16, csplit, M, N, K, G, sym,
                                               split):
    """Both inner loops (fp16 with the 1024 + c words, W4_GEMV_F16=1, for 1-2
    tokens; bf16 with c - z words, =0) and both hand-offs of a K split (the
    partial sums through a global ticket, W4_GEMV_CSPLIT=0, or through
    distributed shared memory inside a cluster, =1; the fp16 loop has only
    the first) against the oracle; the two hand-offs add the same fp32
    partials in the same split order, so they agree bit for bit."""
    if f16 == "1" and M > 2:
        pytest.skip("the fp16 loop takes 1-2 tokens")
    if f16 == "1" and csplit == "1":
        pytest.skip("the fp16 loop's plans hand splits off through the workspace only")
    monkeypatch.setenv("W4_GEMV_F16", f16)
    monkeypatch.setenv("W4_GEMV_SPLIT", split)
    seed = M + N + K + G + int(split)
    packed, scales, zeros = WL.make_random_format(N, K, G, sym, seed)
    x = WL.make_activations(K, M, seed + 1)
    b = torch.randn(N, generator=torch.Generator().manual_seed(seed + 2)) * 0.1
    args = (x.cuda(), packed.cuda(), scales.cuda(), None if zeros is None else zeros.cuda(),
            b.cuda(), N, K, G)
    assert w4.w4a16_workspace_bytes(M, N, K, G) > 0          # the split plan was taken
    monkeypatch.setenv("W4_GEMV_CSPLIT", csplit)
    y = w4.w4a16_linear(*args)
    torch.cuda.synchronize()
    yref = O.w4a16_linear(x, packed.numpy(), scales.numpy(),
                          None if zeros is None else zeros.numpy(), b.numpy(), K, G)
    assert_close(y, yref, f"f16{f16} csplit{csplit} M{M} N{N} K{K} S{split}")
    monkeypatch.setenv("W4_GEMV_CSPLIT", "1" if csplit == "0" else "0")
    y2 = w4.w4a16_linear(*args)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "the two hand-offs differ"
    assert w4.w4_get_device_error() == 0


@pytest.mark.parametrize("M,N,K,G", [(1, 3584, 18944, 128), (1, 37888, 3584, 128),
                                     (4, 3840, 15360, 32), (16, 4608, 3584, 128)])
def test_host_plan_matches_the_device_calls(w4, M, N, K, G):
    """w4_decode_plan (host planner, any SM count) gives the workspace the
    calls ask for on this device, for both kinds of decode call."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert w4.w4_decode_plan("w4a16", M, N, K, G, sm)["workspace"] == \
        w4.w4a16_workspace_bytes(M, N, K, G)
    assert w4.w4_decode_plan("w4a8", M, N, K, G, sm)["workspace"] == \
        w4.w4a8_workspace_bytes(M, N, K, G)


@pytest.mark.parametrize("M,N,K,G,sym,split", [(1, 3584, 18944, 128, True, "5"),
                                               (2, 4608, 3584, 64, False, "1"),
                                               (1, 1000, 4100, 128, True, "0")])
def test_activation_hold_is_only_timing(w4, monkeypatch, M, N, K, G, sym, split):
    """The fp16 loop's producer holding its ring until the activations are
    staged (W4_GEMV_XFIRST = stages before the hold; -1 none, 0 all held)
    changes when copies are issued, never what is computed: every setting
    gives the same bits, and they match the oracle (K = 4100: a ragged
    slice whose activations are read without vector loads)."""
    if split != "0":
        monkeypatch.setenv("W4_GEMV_SPLIT", split)
    seed = M + N + K
    packed, scales, zeros = WL.make_random_format(N, K, G, sym, seed)
    x = WL.make_activations(K, M, seed + 1)
    args = (x.cuda(), packed.cuda(), scales.cuda(), None if zeros is None else zeros.cuda(),
            None, N, K, G)
    outs = []
    for hold in ("-1", "0", "1", "2", "3"):
        monkeypatch.setenv("W4_GEMV_XFIRST", hold)
        outs.append(w4.w4a16_linear(*args))
    torch.cuda.synchronize()
    yref = O.w4a16_linear(x, packed.numpy(), scales.numpy(),
                          None if zeros is None else zeros.numpy(), None, K, G)
    assert_close(outs[0], yref, f"hold M{M} N{N} K{K}")
    for y in outs[1:]:
        assert torch.equal(y.view(torch.int16), outs[0].view(torch.int16))
    assert w4.w4_get_device_error() == 0
