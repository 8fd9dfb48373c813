"""w4a16_linear_noalloc through the C ABI: the entry point for callers that
cannot allocate device memory (a plugin handed only its input and output
buffers, or a runtime that forbids cudaMalloc after start-up).  It runs the
same decode kernel and plan as w4a16_linear, taking its split-K scratch from
the library's own fixed array, so its output must equal w4a16_linear's bit
for bit and match the fp64 oracle within the layer's tolerance, call after
call: two calls queued back to back on one stream before a single
synchronize share the scratch in stream order.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes on its own."""
import ctypes

import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, check_band, ensure_built, guarded_empty

pytestmark = pytest.mark.gpu

W4_ERR_SCRATCH_LIMIT = -10
W4_NOALLOC_SCRATCH_BYTES = 4 << 20


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, x, packed, scales, zeros, bias, y, N, K, G):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.w4a16_linear_noalloc(_p(x), _p(packed), _p(scales), _p(zeros), _p(bias), _p(y),
                                    x.shape[0], N, K, G, 1 if zeros is None else 0, stream)


@pytest.mark.parametrize("M,N,K,G,sym,split", [
    (1, 3584, 18944, 128, True, True),     # the 7B down projection: K split over CTAs
    (16, 4608, 3584, 128, False, True),    # 16 tokens, asymmetric, K split
    (3, 200, 100, 32, True, False),        # small ragged shape, one pass over K
])
def test_noalloc_matches_workspace_entry_point(w4, monkeypatch, M, N, K, G, sym, split):
    lib = w4.load()
    # the split is pinned (the planner's knob) so that the scratch path runs
    # whatever the cost model prefers; a workspace size > 0 is what makes the
    # plan split K, and so use the scratch
    monkeypatch.setenv("W4_GEMV_SPLIT", "2" if split else "1")
    assert (w4.w4a16_workspace_bytes(M, N, K, G) > 0) == split
    seed = M + N + K
    packed, scales, zeros = WL.make_random_format(N, K, G, sym, seed)
    bias = torch.randn(N, generator=torch.Generator().manual_seed(seed)) * 0.1
    x = WL.make_activations(K, M, seed + 1)
    ref = O.w4a16_linear(x, packed.numpy(), scales.numpy(),
                         None if zeros is None else zeros.numpy(), bias.numpy(), K, G)
    packed, scales, bias, x = packed.cuda(), scales.cuda(), bias.cuda(), x.cuda()
    zeros = None if zeros is None else zeros.cuda()
    y_ws = w4.w4a16_linear(x, packed, scales, zeros, bias, N, K, G)
    assert_close(y_ws, ref, "w4a16_linear")
    # two calls queued back to back, one synchronize: the second call's
    # counter clear and scratch use follow the first call in stream order
    outs = []
    for call in range(2):
        y, band = guarded_empty((M, N), torch.bfloat16)
        y.fill_(float("nan"))
        rc = _noalloc(lib, x, packed, scales, zeros, bias, y, N, K, G)
        assert rc == 0, lib.w4_error_string(rc)
        outs.append((y, band))
    torch.cuda.synchronize()
    for call, (y, band) in enumerate(outs):
        check_band(band, f"noalloc call {call}")
        assert_close(y, ref, f"noalloc call {call} vs oracle")
        assert torch.equal(y.view(torch.int16), y_ws.view(torch.int16)), \
            f"noalloc call {call} differs from w4a16_linear"
    assert w4.w4_get_device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(w4, monkeypatch):
    """16 tokens x 16384 outputs x K=32768 with the plan pinned to 8 K
    slices needs 8 x 16 x 16384 fp32 partials (8 MiB), more than the 4 MiB
    built in."""
    lib = w4.load()
    monkeypatch.setenv("W4_GEMV_SPLIT", "8")
    M, N, K, G = 16, 16384, 32768, 128
    assert w4.w4a16_workspace_bytes(M, N, K, G) > W4_NOALLOC_SCRATCH_BYTES
    x = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    packed = torch.zeros(N, K // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(N, K // G, dtype=torch.float32, device="cuda")
    y = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    rc = _noalloc(lib, x, packed, scales, None, None, y, N, K, G)
    assert rc == W4_ERR_SCRATCH_LIMIT
    assert b"scratch" in lib.w4_error_string(rc)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y) == 0          # nothing was enqueued
