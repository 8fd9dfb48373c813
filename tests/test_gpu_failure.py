"""The bounded-wait failure path, run on purpose without faulting the GPU.

Every wait in the library's kernels gives up after a limit of SM clock
cycles (w4_set_wait_limit; about one second by default): the kernel raises
W4_ERR_DEVICE_TIMEOUT in the device flag, every thread of the CTA leaves its
loops, the producer lets the copies it already issued land, and the call
returns with unspecified outputs.  A wait whose data arrives completes in the
hardware's own suspend of the waiting thread, so the tests make a wait that
can never complete (w4_set_fault_injection, grouped decode kernel):

* mode 1: the consumers never publish the group list, so the copy producer
  times out before issuing anything;
* mode 2: the consumers never free a ring slot, so the producer times out
  with copies in flight (K = 16384: every unit has at least eight stages for
  a three-deep ring) and drains them before its CTA exits.

Each test checks that the call returns, that the flag reports the timeout,
and that the next calls with the switch off and the default limit are right:
the grouped call and a split-K decode call (so the device and the split-K
counters are in order)."""
import contextlib
import os

import pytest
import torch

import oracle as O
import workloads as WL
from helpers import assert_close, ensure_built

pytestmark = pytest.mark.gpu

W4_ERR_DEVICE_TIMEOUT = -9
SHORT_LIMIT = 20000            # SM cycles, ~10 us


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _grouped_case():
    E, N, K, G = 4, 128, 16384, 128
    counts = [3, 0, 6, 2]
    T = sum(counts)
    packed, scales, _ = WL.make_random_format(E * N, K, G, True, 5)
    x = WL.make_activations(K, T, 6)
    goff = torch.zeros(E + 1, dtype=torch.int32)
    goff[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int32), 0)
    ref = O.w4a16_grouped_linear(x, goff.numpy(), packed.numpy(), scales.numpy(), None, None,
                                 E, N, K, G)
    # one-token tiles: the activation slice of a whole 16384-column row
    # then fits the shared memory of a grouped plan (which never splits K)
    args = (x.cuda(), goff.cuda(), packed.cuda(), scales.cuda(), None, None, E, N, K, G, 1)
    return args, ref


@contextlib.contextmanager
def _split4():
    """The planner's knob pins four K slices (grouped plans never split, so
    it is set only around the plain decode calls)."""
    old = os.environ.get("W4_GEMV_SPLIT")
    os.environ["W4_GEMV_SPLIT"] = "4"
    try:
        yield
    finally:
        if old is None:
            os.environ.pop("W4_GEMV_SPLIT", None)
        else:
            os.environ["W4_GEMV_SPLIT"] = old


def _split_k_case():
    N, K, G = 3584, 18944, 128
    packed, scales, _ = WL.make_random_format(N, K, G, True, 3)
    x = WL.make_activations(K, 1, 4)
    ref = O.w4a16_linear(x, packed.numpy(), scales.numpy(), None, None, K, G)
    return (x.cuda(), packed.cuda(), scales.cuda(), None, None, N, K, G), ref


@pytest.mark.parametrize("mode", [1, 2])
def test_wait_runs_out_and_next_calls_are_right(w4, mode):
    gargs, gref = _grouped_case()
    dargs, dref = _split_k_case()
    with _split4():
        assert w4.w4a16_workspace_bytes(1, dargs[5], dargs[6], dargs[7]) > 0   # split-K plan
    assert w4.w4_get_device_error() == 0
    w4.w4_set_wait_limit(SHORT_LIMIT)
    w4.w4_set_fault_injection(mode)
    try:
        w4.w4a16_grouped_linear(*gargs)
        err = w4.w4_get_device_error()
    finally:
        w4.w4_set_fault_injection(0)
        w4.w4_set_wait_limit(0)
    assert err == W4_ERR_DEVICE_TIMEOUT
    for _ in range(2):
        assert_close(w4.w4a16_grouped_linear(*gargs), gref, "grouped call after the timeout")
        with _split4():
            assert_close(w4.w4a16_linear(*dargs), dref, "split-K call after the timeout")
    assert w4.w4_get_device_error() == 0


def test_switch_is_ignored_elsewhere_and_rejects_bad_modes(w4):
    """Only the grouped kernel reads the switch: a plain decode call with it
    on is right and raises nothing."""
    dargs, dref = _split_k_case()
    w4.w4_set_fault_injection(2)
    try:
        with _split4():
            y = w4.w4a16_linear(*dargs)
        err = w4.w4_get_device_error()
    finally:
        w4.w4_set_fault_injection(0)
    assert err == 0
    assert_close(y, dref, "plain decode with the switch on")
    with pytest.raises(w4.W4Error):
        w4.w4_set_fault_injection(4)
