"""The decode planner, on the host alone (w4_decode_plan; no GPU needed).

Every plan the library can pick must be launchable and consistent: its
shared memory fits the SM (two CTAs share 228 KB), its K splits cover the
padded K with no empty split, its units and grid follow from the row blocks,
its workspace is what the split hand-off needs, and the inner loop and the
cluster hand-off are chosen only where the kernels support them.  The
tuning variables pin what they name.  The plans tuned on the GB300 for the
7B decode shapes are pinned too, so that a change of the cost model shows
up here before it shows up as a slower bench."""
import itertools
import os
import re

import pytest

from helpers import ROOT, ensure_built


def _header_int(name):
    """An integer #define of include/w4.h (a number or a shift of numbers)."""
    src = open(os.path.join(ROOT, "include", "w4.h")).read()
    expr = re.search(r"#define\s+" + name + r"\s+\(?([0-9<\s]+)\)?", src).group(1)
    a, _, b = expr.partition("<<")
    return int(a) << int(b) if b else int(a)


W4_WORKSPACE_COUNTER_BYTES = _header_int("W4_WORKSPACE_COUNTER_BYTES")
MAX_COUNTERS = W4_WORKSPACE_COUNTER_BYTES // 4
SMEM_PER_CTA = 232448          # 227 KB
SMEM_HALF = 115712             # two CTAs on one SM's 228 KB, 1 KB reserved each
KNOBS = ("W4_GEMV_ROWS", "W4_GEMV_SPLIT", "W4_GEMV_CPS", "W4_GEMV_F16", "W4_GEMV_CSPLIT")


@pytest.fixture(scope="module")
def w4():
    return ensure_built()


@pytest.fixture(autouse=True)
def _clean_env(monkeypatch):
    for k in KNOBS:
        monkeypatch.delenv(k, raising=False)


def _padded(K, G):
    return -(-K // G) * G


def _check_plan(p, kind, M, N, K, G, sm):
    ab = 2 if kind == "w4a16" else 1
    Kp = _padded(K, G)
    R, S, spl, nst = p["rows"], p["splits"], p["stages_per_split"], p["stages"]
    where = f"{kind} M={M} N={N} K={K} G={G} sm={sm}: {p}"
    assert R in (16, 32, 64, 128), where
    assert p["stage_cols"] == 32768 // R, where
    assert nst == -(-Kp // p["stage_cols"]), where
    # the splits cover every stage, none is empty
    assert 1 <= S <= nst and spl == -(-nst // S) and (S - 1) * spl < nst, where
    NB = -(-N // R)
    assert p["units"] == NB * S, where
    cps = p["ctas_per_sm"]
    assert cps in (1, 2), where
    if cps == 2:
        assert M <= (8 if kind == "w4a16" else 4), where
    assert p["grid"] == min(p["units"], cps * sm), where
    # shared memory: the weight ring (at least two 16 KB stages) and the
    # activation slice of every token, within the SM's share
    assert p["smem"] <= (SMEM_HALF if cps == 2 else SMEM_PER_CTA), where
    assert p["smem"] >= 2 * 16384 + M * spl * p["stage_cols"] * ab, where
    if S == 1:
        assert p["workspace"] == 0, where
    else:
        assert p["workspace"] == W4_WORKSPACE_COUNTER_BYTES + S * M * N * 4, where
        # one arrival counter per row block, clear of the 34 the fused
        # SwiGLU + INT8 call keeps at the end of the counter prefix
        assert NB <= MAX_COUNTERS - 34, where
    if p["fp16_loop"]:
        assert kind == "w4a16" and G % 64 == 0 and M <= 2, where
    if p["cluster_split"]:
        assert kind == "w4a16" and not p["fp16_loop"] and 3 <= M <= 8, where
        assert 2 <= S <= 8 and p["units"] <= p["grid"], where


SHAPES = [(16, 32), (200, 100), (256, 512), (3584, 3584), (4608, 3584), (37888, 3584),
          (3584, 18944), (15360, 3840), (3840, 15360), (1000, 65536), (131072, 256)]


@pytest.mark.parametrize("kind", ["w4a16", "w4a8"])
@pytest.mark.parametrize("sm", [152, 148, 20])
def test_every_plan_is_consistent(w4, kind, sm):
    n = 0
    # (every group size here is one the group-wise W4A8 kernel takes)
    for (N, K), G, M in itertools.product(SHAPES, (32, 64, 128, 256), (1, 2, 3, 4, 8, 9, 16)):
        p = w4.w4_decode_plan(kind, M, N, K, G, sm)
        _check_plan(p, kind, M, N, K, G, sm)
        n += 1
    assert n > 200


def test_inner_loop_and_handoff_rules(w4):
    """fp16 loop for 1-2 tokens with groups of 64 or more; bf16 from 3
    tokens and for G = 32; the cluster hand-off only for 3-8 tokens."""
    assert w4.w4_decode_plan("w4a16", 1, 4608, 3584, 128, 152)["fp16_loop"] == 1
    assert w4.w4_decode_plan("w4a16", 2, 4608, 3584, 64, 152)["fp16_loop"] == 1
    assert w4.w4_decode_plan("w4a16", 1, 4608, 3584, 32, 152)["fp16_loop"] == 0
    assert w4.w4_decode_plan("w4a16", 3, 4608, 3584, 128, 152)["fp16_loop"] == 0
    assert w4.w4_decode_plan("w4a8", 1, 4608, 3584, 128, 152)["fp16_loop"] == 0
    for M in (1, 2, 16):
        for N, K in SHAPES:
            assert w4.w4_decode_plan("w4a16", M, N, K, 128, 152)["cluster_split"] == 0


def test_tuning_variables_pin_the_plan(w4, monkeypatch):
    monkeypatch.setenv("W4_GEMV_ROWS", "32")
    assert w4.w4_decode_plan("w4a16", 1, 3584, 18944, 128, 152)["rows"] == 32
    monkeypatch.setenv("W4_GEMV_SPLIT", "2")
    p = w4.w4_decode_plan("w4a16", 1, 3584, 18944, 128, 152)
    assert (p["rows"], p["splits"]) == (32, 2)
    _check_plan(p, "w4a16", 1, 3584, 18944, 128, 152)
    monkeypatch.delenv("W4_GEMV_ROWS")
    monkeypatch.setenv("W4_GEMV_SPLIT", "1")
    assert w4.w4_decode_plan("w4a16", 1, 3584, 18944, 128, 152)["workspace"] == 0
    monkeypatch.delenv("W4_GEMV_SPLIT")
    monkeypatch.setenv("W4_GEMV_CPS", "1")
    assert w4.w4_decode_plan("w4a16", 1, 4608, 3584, 128, 152)["ctas_per_sm"] == 1
    monkeypatch.delenv("W4_GEMV_CPS")
    monkeypatch.setenv("W4_GEMV_F16", "0")
    assert w4.w4_decode_plan("w4a16", 1, 4608, 3584, 128, 152)["fp16_loop"] == 0
    monkeypatch.setenv("W4_GEMV_F16", "1")        # not where the group size forbids it
    assert w4.w4_decode_plan("w4a16", 1, 4608, 3584, 32, 152)["fp16_loop"] == 0
    monkeypatch.delenv("W4_GEMV_F16")
    monkeypatch.setenv("W4_GEMV_CSPLIT", "0")
    for N, K in SHAPES:
        assert w4.w4_decode_plan("w4a16", 4, N, K, 32, 152)["cluster_split"] == 0


def test_tuned_7b_plans(w4):
    """The plans measured fastest on the GB300 (152 SMs) for the 7B decode
    step at one token: qkv and o in 16-row blocks over the whole K, gate_up
    in 128-row blocks, down (K = 18944) in 64-row blocks split 5 ways."""
    got = {name: w4.w4_decode_plan("w4a16", 1, N, K, 128, 152)
           for name, N, K in (("qkv", 4608, 3584), ("o", 3584, 3584),
                              ("gate_up", 37888, 3584), ("down", 3584, 18944))}
    assert {k: (v["rows"], v["splits"], v["grid"]) for k, v in got.items()} == {
        "qkv": (16, 1, 288), "o": (16, 1, 224), "gate_up": (128, 1, 296), "down": (64, 5, 280)}
    assert all(v["fp16_loop"] == 1 and v["ctas_per_sm"] == 2 for v in got.values())


def test_argument_errors(w4):
    lib = w4.load()
    import ctypes
    out = (ctypes.c_longlong * 12)()
    assert lib.w4_decode_plan(0, 1, 64, 256, 128, 152, None) == -2           # NULL_PTR
    for args in ((2, 1, 64, 256, 128, 152), (0, 0, 64, 256, 128, 152),
                 (0, 17, 64, 256, 128, 152), (0, 1, 0, 256, 128, 152),
                 (0, 1, 64, 256, 128, 0)):
        assert lib.w4_decode_plan(*args, ctypes.addressof(out)) == -1, args  # INVALID_ARG
    assert lib.w4_decode_plan(0, 1, 64, 256, 48, 152, ctypes.addressof(out)) == -4
    assert lib.w4_decode_plan(1, 1, 64, 2048, 96, 152, ctypes.addressof(out)) == -4
    assert lib.w4_decode_plan(1, 1, 64, 1127296, 1127296, 152, ctypes.addressof(out)) == -5
    with pytest.raises(w4.W4Error):
        w4.w4_decode_plan("w4a16", 17, 64, 256, 128, 152)
