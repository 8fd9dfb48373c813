"""Shared helpers for the test suite (tolerances, conversions, building)."""
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


def ensure_built():
    from int4_weight_only_gb300 import build as b
    b.build()
    import int4_weight_only_gb300 as w4
    w4.load()
    return w4


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
