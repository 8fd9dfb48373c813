"""The C ABI library builds, loads and exports every symbol include/w4.h
declares; host-side argument checks reject bad calls before any CUDA work
(no GPU needed: none of these calls reaches a kernel)."""
import ctypes
import os
import re

import pytest

from helpers import ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "w4.h")


def _declared():
    src = open(HEADER).read()
    return re.findall(r"^W4_API\s+[\w\s\*]+?\b(w4\w*)\s*\(", src, flags=re.M)


def _codes():
    src = open(HEADER).read()
    return {k: int(v) for k, v in re.findall(r"#define\s+(W4_\w+)\s+(-?\d+)", src)}


@pytest.fixture(scope="module")
def lib():
    w4 = ensure_built()
    return w4.load()


def test_header_declares_the_boundary():
    names = set(_declared())
    assert {"w4_pack_rtn", "w4a16_linear", "w4a8_quantize_act", "w4a8_linear",
            "w4a16_workspace_bytes", "w4a8_workspace_bytes", "w4_get_device_error",
            "w4_error_string"} <= names


def test_every_declared_symbol_is_exported(lib):
    import int4_weight_only_gb300 as w4
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in w4.EXPORTED, f"binding lacks {name}"


def test_error_strings(lib):
    codes = _codes()
    for k, v in codes.items():
        if k.startswith("W4_ERR_") or k == "W4_OK":
            s = lib.w4_error_string(v)
            assert s and s != b"unknown error code", k
    assert lib.w4_error_string(12345) == b"unknown error code"


def test_host_argument_checks(lib):
    c = _codes()
    P = ctypes.c_void_p
    ok16 = P(0x10000)          # fake, 16-byte aligned; never dereferenced
    odd = P(0x10001)
    # w4_pack_rtn
    assert lib.w4_pack_rtn(None, 4, 64, 32, 1, ok16, ok16, None, None) == c["W4_ERR_NULL_PTR"]
    assert lib.w4_pack_rtn(ok16, 4, 64, 48, 1, ok16, ok16, None, None) == c["W4_ERR_UNSUPPORTED_GROUP"]
    assert lib.w4_pack_rtn(ok16, 4, 64, 0, 1, ok16, ok16, None, None) == c["W4_ERR_UNSUPPORTED_GROUP"]
    assert lib.w4_pack_rtn(ok16, 0, 64, 32, 1, ok16, ok16, None, None) == c["W4_ERR_INVALID_ARG"]
    assert lib.w4_pack_rtn(ok16, 4, 64, 32, 1, ok16, ok16, ok16, None) == c["W4_ERR_INVALID_ARG"]
    assert lib.w4_pack_rtn(ok16, 4, 64, 32, 0, ok16, ok16, None, None) == c["W4_ERR_NULL_PTR"]
    assert lib.w4_pack_rtn(ok16, 4, 64, 32, 1, odd, ok16, None, None) == c["W4_ERR_MISALIGNED"]
    # w4a16_linear
    args = [ok16, ok16, ok16, None, None, ok16, 1, 64, 64, 32, 1, None, 0, None]
    bad = list(args); bad[0] = None
    assert lib.w4a16_linear(*bad) == c["W4_ERR_NULL_PTR"]
    bad = list(args); bad[0] = odd
    assert lib.w4a16_linear(*bad) == c["W4_ERR_MISALIGNED"]
    bad = list(args); bad[9] = 100
    assert lib.w4a16_linear(*bad) == c["W4_ERR_UNSUPPORTED_GROUP"]
    bad = list(args); bad[10] = 0            # asymmetric without zeros
    assert lib.w4a16_linear(*bad) == c["W4_ERR_NULL_PTR"]
    bad = list(args); bad[6] = -1
    assert lib.w4a16_linear(*bad) == c["W4_ERR_INVALID_ARG"]
    bad = list(args); bad[6] = 0             # M = 0: nothing to do
    assert lib.w4a16_linear(*bad) == c["W4_OK"]
    # w4a8_linear: per row or group-wise groups, the int32 bound, alignment
    a8 = [ok16, ok16, ok16, ok16, None, ok16, None, 1, 64, 64, 64, None, 0, None]
    bad = list(a8); bad[9] = 192; bad[10] = 96     # group-wise takes 32/64/128/256k
    assert lib.w4a8_linear(*bad) == c["W4_ERR_UNSUPPORTED_GROUP"]
    bad = list(a8); bad[10] = 32; bad[6] = ok16    # group-wise has no int32 acc_out
    assert lib.w4a8_linear(*bad) == c["W4_ERR_INVALID_ARG"]
    big = c["W4_W4A8_MAX_KP"] + 32 - (c["W4_W4A8_MAX_KP"] % 32)
    bad = list(a8); bad[9] = big; bad[10] = big
    assert lib.w4a8_linear(*bad) == c["W4_ERR_K_TOO_LARGE"]
    bad = list(a8); bad[0] = odd
    assert lib.w4a8_linear(*bad) == c["W4_ERR_MISALIGNED"]
    bad = list(a8); bad[7] = 0
    assert lib.w4a8_linear(*bad) == c["W4_OK"]
    # w4a8_quantize_act
    assert lib.w4a8_quantize_act(ok16, 1, 64, 64, odd, ok16, None) == c["W4_ERR_MISALIGNED"]
    assert lib.w4a8_quantize_act(None, 1, 64, 64, ok16, ok16, None) == c["W4_ERR_NULL_PTR"]


def test_host_argument_checks_later_entry_points(lib):
    """The entry points of the fused, grouped, smoothing, GPTQ and bf16
    parameter paths reject bad arguments on the host."""
    c = _codes()
    P = ctypes.c_void_p
    ok16 = P(0x10000)
    odd = P(0x10001)
    F = ctypes.c_float
    # w4a16_linear_swiglu: F % 8 != 0, M > 16
    sw = [ok16, ok16, ok16, None, None, ok16, 1, 64, 64, 32, 1, None, 0, None]
    bad = list(sw); bad[7] = 12
    assert lib.w4a16_linear_swiglu(*bad) == c["W4_ERR_INVALID_ARG"]
    bad = list(sw); bad[6] = 17
    assert lib.w4a16_linear_swiglu(*bad) == c["W4_ERR_UNSUPPORTED_SHAPE"]
    # w4a16_grouped_linear: tile 0 and 17, E = 0, misaligned x
    gr = [ok16, ok16, ok16, ok16, None, None, ok16, 8, 4, 64, 64, 32, 1, 4, None]
    for i, v in ((13, 0), (13, 257), (8, 0)):
        bad = list(gr); bad[i] = v
        assert lib.w4a16_grouped_linear(*bad) == c["W4_ERR_INVALID_ARG"]
    bad = list(gr); bad[0] = odd
    assert lib.w4a16_grouped_linear(*bad) == c["W4_ERR_MISALIGNED"]
    # w4a8_quantize_act_smooth: no factors, misaligned factors
    assert lib.w4a8_quantize_act_smooth(ok16, None, 1, 64, 64, ok16, ok16, None) == c["W4_ERR_NULL_PTR"]
    assert lib.w4a8_quantize_act_smooth(ok16, P(0x10004), 1, 64, 64, ok16, ok16, None) == \
        c["W4_ERR_MISALIGNED"]
    # w4_smooth: alpha outside [0, 1]
    assert lib.w4_smooth(ok16, 4, ok16, 4, 64, F(1.5), ok16, ok16, None) == c["W4_ERR_INVALID_ARG"]
    assert lib.w4_smooth(ok16, 4, ok16, 4, 64, F(-0.1), ok16, ok16, None) == c["W4_ERR_INVALID_ARG"]
    # w4_gptq: no tokens, bad group, no workspace
    gq = [ok16, 4, ok16, 8, 64, 32, 1, F(0.01), ok16, ok16, None, ok16, ok16, 1 << 30, None]
    bad = list(gq); bad[1] = 0
    assert lib.w4_gptq(*bad) == c["W4_ERR_INVALID_ARG"]
    bad = list(gq); bad[5] = 48
    assert lib.w4_gptq(*bad) == c["W4_ERR_UNSUPPORTED_GROUP"]
    bad = list(gq); bad[12] = None
    assert lib.w4_gptq(*bad) == c["W4_ERR_WORKSPACE"]
    assert lib.w4_gptq_workspace_bytes(8, 64, 48) == 0
    assert lib.w4_gptq_workspace_bytes(8, 64, 32) > 2 * 64 * 64 * 4
    # bf16 parameters: symmetric with offsets, asymmetric without, misaligned scales
    assert lib.w4_pack_rtn_bf16(ok16, 4, 64, 32, 1, ok16, ok16, ok16, None) == c["W4_ERR_INVALID_ARG"]
    assert lib.w4_pack_rtn_bf16(ok16, 4, 64, 32, 0, ok16, ok16, None, None) == c["W4_ERR_NULL_PTR"]
    bp = [ok16, ok16, ok16, None, None, ok16, 1, 64, 64, 32, None, 0, None]
    bad = list(bp); bad[2] = P(0x10002)
    assert lib.w4a16_linear_bf16p(*bad) == c["W4_ERR_MISALIGNED"]
    bad = list(bp); bad[6] = 0
    assert lib.w4a16_linear_bf16p(*bad) == c["W4_OK"]


def test_host_argument_checks_shard_entry_points(lib):
    """w4a16_linear_partial and w4a16_partial_finish reject bad arguments on
    the host; M = 0 enqueues nothing."""
    c = _codes()
    P = ctypes.c_void_p
    ok16 = P(0x10000)
    odd = P(0x10001)
    pa = [ok16, ok16, ok16, None, ok16, 1, 64, 64, 32, 1, None, 0, None]
    bad = list(pa); bad[4] = None
    assert lib.w4a16_linear_partial(*bad) == c["W4_ERR_NULL_PTR"]
    bad = list(pa); bad[4] = P(0x10002)            # fp32 output, 4-byte aligned
    assert lib.w4a16_linear_partial(*bad) == c["W4_ERR_MISALIGNED"]
    bad = list(pa); bad[0] = odd
    assert lib.w4a16_linear_partial(*bad) == c["W4_ERR_MISALIGNED"]
    bad = list(pa); bad[8] = 40
    assert lib.w4a16_linear_partial(*bad) == c["W4_ERR_UNSUPPORTED_GROUP"]
    bad = list(pa); bad[9] = 0                     # asymmetric without zeros
    assert lib.w4a16_linear_partial(*bad) == c["W4_ERR_NULL_PTR"]
    bad = list(pa); bad[5] = 0
    assert lib.w4a16_linear_partial(*bad) == c["W4_OK"]
    assert lib.w4a16_partial_finish(None, None, ok16, 1, 8, None) == c["W4_ERR_NULL_PTR"]
    assert lib.w4a16_partial_finish(ok16, None, odd, 1, 8, None) == c["W4_ERR_MISALIGNED"]
    assert lib.w4a16_partial_finish(ok16, None, ok16, 1, 0, None) == c["W4_ERR_INVALID_ARG"]
    assert lib.w4a16_partial_finish(ok16, None, ok16, 0, 8, None) == c["W4_OK"]


def test_w4a8_bound_constant_matches_int32():
    """W4_W4A8_MAX_KP is the largest Kp with Kp * 15 * 127 < 2^31 (codes in
    [0, 15] times q_x in [-127, 127])."""
    kmax = _codes()["W4_W4A8_MAX_KP"]
    assert kmax * 15 * 127 <= 2 ** 31 - 1 < (kmax + 1) * 15 * 127
