"""Shared helpers for the test suite (tolerances, conversions, building,
guard bands around the outputs of every GPU call)."""
import functools
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# bf16 outputs vs the fp64 oracle: relative Frobenius error and max |diff|
# relative to max |y| (the bar the workloads are specified with).
REL_FRO_TOL = 5e-3
MAX_ABS_TOL = 1e-2

# Guard bands: every output buffer the tests let the binding allocate is
# carved out of a larger buffer whose GUARD_BYTES before and after it hold a
# sentinel byte; after the call the bands must be unchanged.  compute-
# sanitizer is not available, so this is how an out-of-bounds store shows.
GUARD_BYTES = 4096
SENTINEL = 0xA5


class GuardViolation(AssertionError):
    pass


def guarded_empty(shape, dtype, device="cuda"):
    """(tensor, band) : a contiguous tensor of `shape` inside a buffer with
    GUARD_BYTES of SENTINEL on both sides (16-byte aligned, like a fresh
    allocation)."""
    esz = torch.empty((), dtype=dtype).element_size()
    n = int(np.prod(shape)) if len(shape) else 1
    raw = torch.full((GUARD_BYTES * 2 + n * esz,), SENTINEL, dtype=torch.uint8, device=device)
    t = raw[GUARD_BYTES:GUARD_BYTES + n * esz].view(dtype).view(*shape)
    return t, raw


def check_band(raw, what):
    torch.cuda.synchronize()
    lo = raw[:GUARD_BYTES]
    hi = raw[raw.numel() - GUARD_BYTES:]
    bad_lo = int((lo != SENTINEL).sum())
    bad_hi = int((hi != SENTINEL).sum())
    if bad_lo or bad_hi:
        raise GuardViolation(f"{what}: {bad_lo} bytes before and {bad_hi} bytes after the "
                             f"output were overwritten")


class GuardedW4:
    """The binding module with its output-producing entry points wrapped:
    when the caller does not pass an output, it is allocated inside guard
    bands, and the bands are checked (after a synchronize) once the call
    returns.  Everything else passes through unchanged."""

    def __init__(self, mod):
        self._mod = mod

    def __getattr__(self, name):
        return getattr(self._mod, name)

    def _run(self, fn, what, outs, *args, **kw):
        bands = []
        for key, shape, dtype in outs:
            if kw.get(key) is None and shape is not None:
                t, raw = guarded_empty(shape, dtype)
                kw[key] = t
                bands.append((raw, f"{what} {key}"))
        res = fn(*args, **kw)
        for raw, w in bands:
            check_band(raw, w)
        return res

    def w4a16_linear(self, x, packed, scales, zeros, bias, N, K, group_size, **kw):
        return self._run(self._mod.w4a16_linear, "w4a16_linear",
                         [("y", (x.shape[0], N), torch.bfloat16)],
                         x, packed, scales, zeros, bias, N, K, group_size, **kw)

    def w4a16_linear_noalloc(self, x, packed, scales, zeros, bias, N, K, group_size, **kw):
        return self._run(self._mod.w4a16_linear_noalloc, "w4a16_linear_noalloc",
                         [("y", (x.shape[0], N), torch.bfloat16)],
                         x, packed, scales, zeros, bias, N, K, group_size, **kw)

    def w4a16_linear_partial(self, x, packed, scales, zeros, N, K, group_size, **kw):
        return self._run(self._mod.w4a16_linear_partial, "w4a16_linear_partial",
                         [("y32", (x.shape[0], N), torch.float32)],
                         x, packed, scales, zeros, N, K, group_size, **kw)

    def w4a16_partial_finish(self, ysum, bias, **kw):
        return self._run(self._mod.w4a16_partial_finish, "w4a16_partial_finish",
                         [("y", tuple(ysum.shape), torch.bfloat16)], ysum, bias, **kw)

    def w4a16_linear_bf16p(self, x, packed, scales_b, offsets_b, bias, N, K, group_size, **kw):
        return self._run(self._mod.w4a16_linear_bf16p, "w4a16_linear_bf16p",
                         [("y", (x.shape[0], N), torch.bfloat16)],
                         x, packed, scales_b, offsets_b, bias, N, K, group_size, **kw)

    def w4a16_linear_swiglu(self, x, packed, scales, zeros, bias, F, K, group_size, **kw):
        return self._run(self._mod.w4a16_linear_swiglu, "w4a16_linear_swiglu",
                         [("y", (x.shape[0], F), torch.bfloat16)],
                         x, packed, scales, zeros, bias, F, K, group_size, **kw)

    def w4a16_linear_swiglu_q8(self, x, packed, scales, zeros, bias, F, K, group_size,
                               q_group_size, **kw):
        Fp = self._mod.padded_k(F, q_group_size) if q_group_size > 0 else None
        return self._run(self._mod.w4a16_linear_swiglu_q8, "w4a16_linear_swiglu_q8",
                         [("y", (x.shape[0], F), torch.bfloat16),
                          ("qx", None if Fp is None else (x.shape[0], Fp), torch.int8),
                          ("sx", (x.shape[0],), torch.float32)],
                         x, packed, scales, zeros, bias, F, K, group_size, q_group_size, **kw)

    def w4a16_grouped_linear(self, x, goff, packed, scales, zeros, bias, E, N, K, group_size,
                             tile_tokens, **kw):
        return self._run(self._mod.w4a16_grouped_linear, "w4a16_grouped_linear",
                         [("y", (x.shape[0], N), torch.bfloat16)],
                         x, goff, packed, scales, zeros, bias, E, N, K, group_size,
                         tile_tokens, **kw)

    def w4a8_quantize_act(self, x, group_size, **kw):
        Kp = self._mod.padded_k(x.shape[1], group_size) if group_size > 0 else None
        return self._run(self._mod.w4a8_quantize_act, "w4a8_quantize_act",
                         [("qx", None if Kp is None else (x.shape[0], Kp), torch.int8),
                          ("sx", (x.shape[0],), torch.float32)],
                         x, group_size, **kw)

    def w4a8_quantize_act_smooth(self, x, inv_s, group_size, **kw):
        Kp = self._mod.padded_k(x.shape[1], group_size) if group_size > 0 else None
        return self._run(self._mod.w4a8_quantize_act_smooth, "w4a8_quantize_act_smooth",
                         [("qx", None if Kp is None else (x.shape[0], Kp), torch.int8),
                          ("sx", (x.shape[0],), torch.float32)],
                         x, inv_s, group_size, **kw)

    def w4a8_linear(self, qx, sx, packed, w_scales, bias, N, K, group_size, **kw):
        outs = [("y", (qx.shape[0], N), torch.bfloat16)]
        if kw.get("want_acc"):
            outs.append(("acc_out", (qx.shape[0], N), torch.int32))
        return self._run(self._mod.w4a8_linear, "w4a8_linear", outs,
                         qx, sx, packed, w_scales, bias, N, K, group_size, **kw)


def ensure_built():
    from int4_weight_only_gb300 import build as b
    b.build()
    import int4_weight_only_gb300 as w4
    w4.load()
    return GuardedW4(w4)


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().to("cpu")
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy()


def assert_close(y_gpu: torch.Tensor, y_ref: np.ndarray, what: str = ""):
    y = to_np(y_gpu).astype(np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    d = y - y_ref
    ref_norm = np.linalg.norm(y_ref)
    rel = np.linalg.norm(d) / ref_norm if ref_norm > 0 else np.linalg.norm(d)
    mx = np.abs(d).max() if d.size else 0.0
    ymax = np.abs(y_ref).max() if d.size else 0.0
    assert rel <= REL_FRO_TOL, f"{what}: rel Frobenius error {rel:.3e} > {REL_FRO_TOL}"
    assert mx <= MAX_ABS_TOL * max(ymax, 1e-30), \
        f"{what}: max|diff| {mx:.3e} > {MAX_ABS_TOL} * max|y| ({ymax:.3e})"
    return rel, mx / max(ymax, 1e-30)
