"""The bounded-wait failure path, run on purpose without faulting the GPU.

Every wait in the library's kernels gives up after a limit of SM clock
cycles (w4_set_wait_limit; about one second by default): the kernel raises
W4_ERR_DEVICE_TIMEOUT in the device flag, every thread of the CTA leaves its
loops, the producer lets the copies it already issued land, and the call
returns with unspecified outputs.  A one-cycle limit makes a wait run out on
a call whose copy pipeline must wait: the 7B down projection streams eight
16 KB stages per CTA through a four-deep ring, so each producer waits for its
consumers to free a slot; a grouped call's producer waits for the consumers
to list the groups.  The tests check that such a call returns, that the flag
reports the timeout, and that the next call with the default limit is right
(so the split-K counters were left at zero and the context is usable)."""
import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, ensure_built

pytestmark = pytest.mark.gpu

W4_ERR_DEVICE_TIMEOUT = -9


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def test_decode_wait_runs_out_and_next_call_is_right(w4):
    N, K, G = 3584, 18944, 128
    assert w4.w4a16_workspace_bytes(1, N, K, G) > 0          # split-K plan
    packed, scales, _ = WL.make_random_format(N, K, G, True, 3)
    x = WL.make_activations(K, 1, 4)
    ref = O.w4a16_linear(x, packed.numpy(), scales.numpy(), None, None, K, G)
    packed, scales, xd = packed.cuda(), scales.cuda(), x.cuda()
    assert w4.w4_get_device_error() == 0
    w4.w4_set_wait_limit(1)
    try:
        w4.w4a16_linear(xd, packed, scales, None, None, N, K, G)
        err = w4.w4_get_device_error()
    finally:
        w4.w4_set_wait_limit(0)
    assert err == W4_ERR_DEVICE_TIMEOUT
    for _ in range(2):
        y = w4.w4a16_linear(xd, packed, scales, None, None, N, K, G)
        assert_close(y, ref, "call after the timeout")
        assert w4.w4_get_device_error() == 0


def test_grouped_wait_runs_out_and_next_call_is_right(w4):
    E, N, K, G = 8, 256, 1024, 32
    counts = [3, 0, 5, 1, 0, 2, 7, 1]
    T = sum(counts)
    packed, scales, _ = WL.make_random_format(E * N, K, G, True, 5)
    x = WL.make_activations(K, T, 6)
    goff = torch.zeros(E + 1, dtype=torch.int32)
    goff[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int32), 0)
    ref = O.w4a16_grouped_linear(x, goff.numpy(), packed.numpy(), scales.numpy(), None, None,
                                 E, N, K, G)
    args = (x.cuda(), goff.cuda(), packed.cuda(), scales.cuda(), None, None, E, N, K, G, 8)
    w4.w4_set_wait_limit(1)
    try:
        w4.w4a16_grouped_linear(*args)
        err = w4.w4_get_device_error()
    finally:
        w4.w4_set_wait_limit(0)
    assert err == W4_ERR_DEVICE_TIMEOUT
    y = w4.w4a16_grouped_linear(*args)
    assert_close(y, ref, "grouped call after the timeout")
    assert w4.w4_get_device_error() == 0


def test_default_limit_restored(w4):
    """With the default limit an ordinary call raises nothing."""
    lin = WL.tiny()[0]
    packed, scales, _ = WL.make_random_format(lin.N, lin.K, lin.group_size, True, 9)
    x = WL.make_activations(lin.K, 1, 10)
    w4.w4a16_linear(x.cuda(), packed.cuda(), scales.cuda(), None, None, lin.N, lin.K,
                    lin.group_size)
    assert w4.w4_get_device_error() == 0
