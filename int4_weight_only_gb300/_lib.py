"""ctypes binding of libw4.so (see include/w4.h for the contract)."""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libw4.so")

_c_int, _c_size, _vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/w4.h
_SIGS = {
    "w4_pack_rtn": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp]),
    "w4a16_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "w4a16_linear_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                      _c_int, _c_int, _vp]),
    "w4a16_linear": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                              _c_int, _vp, _c_size, _vp]),
    "w4a16_linear_partial": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                      _c_int, _vp, _c_size, _vp]),
    "w4a16_partial_finish": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _vp]),
    "w4_pack_rtn_bf16": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp]),
    "w4a16_linear_bf16p": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                    _vp, _c_size, _vp]),
    "w4a16_linear_swiglu": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                     _c_int, _c_int, _vp, _c_size, _vp]),
    "w4a16_linear_swiglu_q8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int,
                                        _c_int, _c_int, _c_int, _c_int, _vp, _c_size, _vp]),
    "w4a16_grouped_linear": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                      _c_int, _c_int, _c_int, _c_int, _vp]),
    "w4a8_quantize_act": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp, _vp, _vp]),
    "w4a8_quantize_act_smooth": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp]),
    "w4_smooth": (_c_int, [_vp, _c_int, _vp, _c_int, _c_int, ctypes.c_float, _vp, _vp, _vp]),
    "w4_gptq_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "w4_gptq": (_c_int, [_vp, _c_int, _vp, _c_int, _c_int, _c_int, _c_int, ctypes.c_float, _vp,
                         _vp, _vp, _vp, _vp, _c_size, _vp]),
    "w4a8_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "w4_decode_plan": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp]),
    "w4a8_linear": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                             _vp, _c_size, _vp]),
    "w4_get_device_error": (_c_int, [_vp]),
    "w4_set_wait_limit": (_c_int, [ctypes.c_longlong, _vp]),
    "w4_set_fault_injection": (_c_int, [_c_int, _vp]),
    "w4_error_string": (ctypes.c_char_p, [_c_int]),
}
EXPORTED = tuple(_SIGS)

_lib = None
_lock = threading.Lock()


class W4Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({w4_error_string(code)})")


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libw4.so (built by __graft_entry__.build()); raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"libw4.so is not built ({_LIB_PATH}); "
                                   "run int4_weight_only_gb300.build.build()")
            lib = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(lib, name)
                f.restype, f.argtypes = res, args
            _lib = lib
    return _lib


def w4_error_string(code: int) -> str:
    return load().w4_error_string(int(code)).decode()


def padded_k(K: int, group_size: int) -> int:
    return -(-K // group_size) * group_size


def _ptr(t: Optional[torch.Tensor]):
    # plain ints: the argtypes (c_void_p) convert them without a wrapper object
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t: torch.Tensor, stream=None):
    """cudaStream_t of `stream`, or of the current torch stream of t's device."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(t.get_device())
    return torch.cuda.current_stream(t.device).cuda_stream


def _need(t, dtype, shape, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.shape != shape:
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check(fn: str, rc: int):
    if rc != 0:
        raise W4Error(fn, rc)


# ------------------------------------------------------------- workspace
_ws = {}


def _workspace(device: torch.device, nbytes: int) -> Optional[torch.Tensor]:
    """A per-device zero-filled scratch buffer (grown on demand); the kernels
    leave its counters at zero after each call."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    buf = _ws.get(idx)
    if nbytes == 0:
        return buf
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws[idx] = buf
    return buf


W4_ERR_WORKSPACE = -6


def _call_with_workspace(fn, name, args_before, args_after, device, workspace, need_bytes):
    """Call fn(*args_before, ws_ptr, ws_bytes, *args_after).  Without a caller
    workspace the cached one goes in as it is; only when the library answers
    that it is too small is the size queried and the buffer grown (so the
    common call costs no size query)."""
    ws = workspace if workspace is not None else _ws.get(
        device.index if device.index is not None else torch.cuda.current_device())
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    rc = fn(*args_before, _ptr(ws), wsb, *args_after)
    if rc == W4_ERR_WORKSPACE and workspace is None:
        ws = _workspace(device, need_bytes())
        rc = fn(*args_before, _ptr(ws), ws.numel() * ws.element_size(), *args_after)
    _check(name, rc)


# ------------------------------------------------------------- entry points
def w4_pack_rtn(W: torch.Tensor, group_size: int, symmetric: bool,
                packed=None, scales=None, zeros=None, stream=None
                ) -> Tuple[torch.Tensor, torch.Tensor, Optional[torch.Tensor]]:
    """RTN INT4 quantize + pack W [N, K] fp32 -> (packed [N, Kp/2] u8,
    scales [N, Ng] f32, zeros [N, Ng] u8 or None)."""
    N, K = W.shape
    _need(W, torch.float32, (N, K), "W")
    Kp = padded_k(K, group_size)
    Ng = Kp // group_size if group_size > 0 else 0
    dev = W.device
    if packed is None:
        packed = torch.empty(N, Kp // 2, dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(N, Ng, dtype=torch.float32, device=dev)
    if not symmetric and zeros is None:
        zeros = torch.empty(N, Ng, dtype=torch.uint8, device=dev)
    _need(packed, torch.uint8, (N, Kp // 2), "packed")
    _need(scales, torch.float32, (N, Ng), "scales")
    if zeros is not None:
        _need(zeros, torch.uint8, (N, Ng), "zeros")
    rc = load().w4_pack_rtn(_ptr(W), N, K, int(group_size), 1 if symmetric else 0,
                            _ptr(packed), _ptr(scales), _ptr(zeros), _stream(W, stream))
    _check("w4_pack_rtn", rc)
    return packed, scales, zeros


def w4a16_workspace_bytes(M: int, N: int, K: int, group_size: int) -> int:
    return int(load().w4a16_workspace_bytes(M, N, K, group_size))


def w4a8_workspace_bytes(M: int, N: int, K: int, group_size: int) -> int:
    return int(load().w4a8_workspace_bytes(M, N, K, group_size))


DECODE_PLAN_FIELDS = ("rows", "splits", "stages_per_split", "stages", "stage_cols", "units",
                      "grid", "ctas_per_sm", "smem", "workspace", "fp16_loop", "cluster_split")


def w4_decode_plan(kind: str, M: int, N: int, K: int, group_size: int,
                   sm_count: int) -> dict:
    """The decode launch plan of one layer ("w4a16" or "w4a8"), from the host
    planner alone (no device needed), as a dict of DECODE_PLAN_FIELDS."""
    out = (ctypes.c_longlong * len(DECODE_PLAN_FIELDS))()
    k = {"w4a16": 0, "w4a8": 1}[kind]
    _check("w4_decode_plan", load().w4_decode_plan(k, M, N, K, group_size, sm_count,
                                                   ctypes.addressof(out)))
    return dict(zip(DECODE_PLAN_FIELDS, (int(v) for v in out)))


def w4a16_linear(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                 zeros: Optional[torch.Tensor], bias: Optional[torch.Tensor], N: int, K: int,
                 group_size: int, y=None, workspace=None, stream=None) -> torch.Tensor:
    """y [M, N] bf16 = x [M, K] bf16 . W_hat^T (+ bias)."""
    M = x.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    Kp = padded_k(K, group_size)
    Ng = Kp // group_size
    _need(packed, torch.uint8, (N, Kp // 2), "packed")
    _need(scales, torch.float32, (N, Ng), "scales")
    if zeros is not None:
        _need(zeros, torch.uint8, (N, Ng), "zeros")
    if bias is not None:
        _need(bias, torch.float32, (N,), "bias")
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, (M, N), "y")
    if M == 0:
        return y                # no tokens: nothing to launch
    lib = load()
    _call_with_workspace(
        lib.w4a16_linear, "w4a16_linear",
        (_ptr(x), _ptr(packed), _ptr(scales), _ptr(zeros), _ptr(bias), _ptr(y), M, N, K,
         int(group_size), 1 if zeros is None else 0),
        (_stream(x, stream),), x.device, workspace,
        lambda: lib.w4a16_workspace_bytes(M, N, K, group_size))
    return y


def w4a16_linear_partial(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                         zeros: Optional[torch.Tensor], N: int, K: int, group_size: int,
                         y32=None, workspace=None, stream=None) -> torch.Tensor:
    """y32 [M, N] fp32 = x [M, K] bf16 . W_hat^T without bias: a row-parallel
    shard's partial sum (K is the shard's slice width)."""
    M = x.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    Kp = padded_k(K, group_size)
    Ng = Kp // group_size
    _need(packed, torch.uint8, (N, Kp // 2), "packed")
    _need(scales, torch.float32, (N, Ng), "scales")
    if zeros is not None:
        _need(zeros, torch.uint8, (N, Ng), "zeros")
    if y32 is None:
        y32 = torch.empty(M, N, dtype=torch.float32, device=x.device)
    _need(y32, torch.float32, (M, N), "y32")
    if M == 0:
        return y32
    lib = load()
    _call_with_workspace(
        lib.w4a16_linear_partial, "w4a16_linear_partial",
        (_ptr(x), _ptr(packed), _ptr(scales), _ptr(zeros), _ptr(y32), M, N, K,
         int(group_size), 1 if zeros is None else 0),
        (_stream(x, stream),), x.device, workspace,
        lambda: lib.w4a16_workspace_bytes(M, N, K, group_size))
    return y32


def w4a16_partial_finish(ysum: torch.Tensor, bias: Optional[torch.Tensor], y=None,
                         stream=None) -> torch.Tensor:
    """y [M, N] bf16 = ysum [M, N] fp32 (+ bias [N] fp32), one rounding."""
    M, N = ysum.shape
    _need(ysum, torch.float32, (M, N), "ysum")
    if bias is not None:
        _need(bias, torch.float32, (N,), "bias")
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=ysum.device)
    _need(y, torch.bfloat16, (M, N), "y")
    if M == 0:
        return y
    _check("w4a16_partial_finish", load().w4a16_partial_finish(
        _ptr(ysum), _ptr(bias), _ptr(y), M, N, _stream(ysum, stream)))
    return y


def w4_pack_rtn_bf16(W: torch.Tensor, group_size: int, symmetric: bool, stream=None):
    """RTN pack with bf16 parameters -> (packed [N, Kp/2] u8, scales [N, Ng]
    bf16, offsets (8 - z) s [N, Ng] bf16 or None when symmetric)."""
    N, K = W.shape
    _need(W, torch.float32, (N, K), "W")
    Kp = padded_k(K, group_size)
    Ng = Kp // group_size if group_size > 0 else 0
    dev = W.device
    packed = torch.empty(N, Kp // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(N, Ng, dtype=torch.bfloat16, device=dev)
    offs = None if symmetric else torch.empty(N, Ng, dtype=torch.bfloat16, device=dev)
    _check("w4_pack_rtn_bf16", load().w4_pack_rtn_bf16(
        _ptr(W), N, K, int(group_size), 1 if symmetric else 0, _ptr(packed), _ptr(scales),
        _ptr(offs), _stream(W, stream)))
    return packed, scales, offs


def w4a16_linear_bf16p(x: torch.Tensor, packed: torch.Tensor, scales_b: torch.Tensor,
                       offsets_b: Optional[torch.Tensor], bias: Optional[torch.Tensor], N: int,
                       K: int, group_size: int, y=None, workspace=None,
                       stream=None) -> torch.Tensor:
    """w4a16_linear with bf16 scales (and bf16 (8 - z) s offsets)."""
    M = x.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    Kp = padded_k(K, group_size)
    Ng = Kp // group_size
    _need(packed, torch.uint8, (N, Kp // 2), "packed")
    _need(scales_b, torch.bfloat16, (N, Ng), "scales_b")
    if offsets_b is not None:
        _need(offsets_b, torch.bfloat16, (N, Ng), "offsets_b")
    if bias is not None:
        _need(bias, torch.float32, (N,), "bias")
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, (M, N), "y")
    if M == 0:
        return y
    lib = load()
    _call_with_workspace(
        lib.w4a16_linear_bf16p, "w4a16_linear_bf16p",
        (_ptr(x), _ptr(packed), _ptr(scales_b), _ptr(offsets_b), _ptr(bias), _ptr(y), M, N, K,
         int(group_size)),
        (_stream(x, stream),), x.device, workspace,
        lambda: lib.w4a16_workspace_bytes(M, N, K, group_size))
    return y


def pair_gate_up(gate: torch.Tensor, up: torch.Tensor) -> torch.Tensor:
    """Rows of gate and up [F, ...] in the order w4a16_linear_swiglu reads:
    16-row tiles of 8 gate rows followed by the same 8 up rows ([2F, ...]).
    Works for weight matrices (before w4_pack_rtn) and bias vectors."""
    F = gate.shape[0]
    if up.shape != gate.shape or F % 8:
        raise ValueError("gate and up must have the same shape with a multiple of 8 rows")
    rest = tuple(gate.shape[1:])
    return torch.stack([gate.reshape(F // 8, 8, *rest), up.reshape(F // 8, 8, *rest)],
                       dim=1).reshape(2 * F, *rest).contiguous()


def w4a16_linear_swiglu(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                        zeros: Optional[torch.Tensor], bias: Optional[torch.Tensor], F: int,
                        K: int, group_size: int, y=None, workspace=None,
                        stream=None) -> torch.Tensor:
    """y [M, F] bf16 = SiLU(x W_gate^T + b_gate) * (x W_up^T + b_up); packed /
    scales / zeros / bias hold the 2F paired rows (see pair_gate_up)."""
    M = x.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    Kp = padded_k(K, group_size)
    Ng = Kp // group_size
    _need(packed, torch.uint8, (2 * F, Kp // 2), "packed")
    _need(scales, torch.float32, (2 * F, Ng), "scales")
    if zeros is not None:
        _need(zeros, torch.uint8, (2 * F, Ng), "zeros")
    if bias is not None:
        _need(bias, torch.float32, (2 * F,), "bias")
    if y is None:
        y = torch.empty(M, F, dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, (M, F), "y")
    if M == 0:
        return y                # no tokens: nothing to launch
    lib = load()
    _call_with_workspace(
        lib.w4a16_linear_swiglu, "w4a16_linear_swiglu",
        (_ptr(x), _ptr(packed), _ptr(scales), _ptr(zeros), _ptr(bias), _ptr(y), M, F, K,
         int(group_size), 1 if zeros is None else 0),
        (_stream(x, stream),), x.device, workspace,
        lambda: lib.w4a16_workspace_bytes(M, 2 * F, K, group_size))
    return y


def w4a16_linear_swiglu_q8(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                           zeros: Optional[torch.Tensor], bias: Optional[torch.Tensor], F: int,
                           K: int, group_size: int, q_group_size: int, y=None, qx=None, sx=None,
                           workspace=None, stream=None):
    """w4a16_linear_swiglu that also returns the INT8 activations of the
    W4A8 layer after it: (y [M, F] bf16, qx [M, Fp] int8, sx [M] fp32),
    Fp = F padded to q_group_size; qx, sx = w4a8_quantize_act(y)."""
    M = x.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    Kp = padded_k(K, group_size)
    Ng = Kp // group_size
    Fp = padded_k(F, q_group_size)
    _need(packed, torch.uint8, (2 * F, Kp // 2), "packed")
    _need(scales, torch.float32, (2 * F, Ng), "scales")
    if zeros is not None:
        _need(zeros, torch.uint8, (2 * F, Ng), "zeros")
    if bias is not None:
        _need(bias, torch.float32, (2 * F,), "bias")
    dev = x.device
    if y is None:
        y = torch.empty(M, F, dtype=torch.bfloat16, device=dev)
    if qx is None:
        qx = torch.empty(M, Fp, dtype=torch.int8, device=dev)
    if sx is None:
        sx = torch.empty(M, dtype=torch.float32, device=dev)
    _need(y, torch.bfloat16, (M, F), "y")
    _need(qx, torch.int8, (M, Fp), "qx")
    _need(sx, torch.float32, (M,), "sx")
    if M == 0:
        return y, qx, sx
    lib = load()
    _call_with_workspace(
        lib.w4a16_linear_swiglu_q8, "w4a16_linear_swiglu_q8",
        (_ptr(x), _ptr(packed), _ptr(scales), _ptr(zeros), _ptr(bias), _ptr(y), _ptr(qx),
         _ptr(sx), M, F, K, int(group_size), 1 if zeros is None else 0, int(q_group_size)),
        (_stream(x, stream),), dev, workspace,
        lambda: max(lib.w4a16_workspace_bytes(M, 2 * F, K, group_size), 64 << 10))
    return y, qx, sx


def w4a16_grouped_linear(x: torch.Tensor, goff: torch.Tensor, packed: torch.Tensor,
                         scales: torch.Tensor, zeros: Optional[torch.Tensor],
                         bias: Optional[torch.Tensor], E: int, N: int, K: int, group_size: int,
                         tile_tokens: int, y=None, stream=None) -> torch.Tensor:
    """Grouped W4A16 linear: rows goff[e] .. goff[e+1]-1 of x [T, K] (sorted
    by group) times group e's matrix -> the same rows of y [T, N].  packed /
    scales / zeros / bias hold the E groups stacked ([E*N, ...] or [E, N, ...]);
    goff is an int32 CUDA tensor [E+1]; groups are taken in passes of at
    most tile_tokens tokens: 1..16 on the decode kernel, 17..256 on the
    tensor-core kernel (tiles of 64 or 256 tokens, K % 8 == 0)."""
    T = x.shape[0]
    _need(x, torch.bfloat16, (T, K), "x")
    Kp = padded_k(K, group_size)
    Ng = Kp // group_size
    _need(goff, torch.int32, (E + 1,), "goff")
    packed = packed.reshape(E * N, -1)
    scales = scales.reshape(E * N, -1)
    _need(packed, torch.uint8, (E * N, Kp // 2), "packed")
    _need(scales, torch.float32, (E * N, Ng), "scales")
    if zeros is not None:
        zeros = zeros.reshape(E * N, -1)
        _need(zeros, torch.uint8, (E * N, Ng), "zeros")
    if bias is not None:
        bias = bias.reshape(E * N)
        _need(bias, torch.float32, (E * N,), "bias")
    if y is None:
        y = torch.empty(T, N, dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, (T, N), "y")
    if T == 0:
        return y
    lib = load()
    _check("w4a16_grouped_linear", lib.w4a16_grouped_linear(
        _ptr(x), _ptr(goff), _ptr(packed), _ptr(scales), _ptr(zeros), _ptr(bias), _ptr(y),
        T, E, N, K, int(group_size), 1 if zeros is None else 0, int(tile_tokens),
        _stream(x, stream)))
    return y


def w4a16_linear_noalloc(x: torch.Tensor, packed: torch.Tensor, scales: torch.Tensor,
                         zeros: Optional[torch.Tensor], bias: Optional[torch.Tensor], N: int,
                         K: int, group_size: int, y=None, stream=None) -> torch.Tensor:
    """w4a16_linear (M <= 16) with the library's built-in split-K scratch;
    for callers that cannot allocate device memory.  Calls must not overlap
    on the GPU."""
    M = x.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    Kp = padded_k(K, group_size)
    Ng = Kp // group_size
    _need(packed, torch.uint8, (N, Kp // 2), "packed")
    _need(scales, torch.float32, (N, Ng), "scales")
    if zeros is not None:
        _need(zeros, torch.uint8, (N, Ng), "zeros")
    if bias is not None:
        _need(bias, torch.float32, (N,), "bias")
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    _need(y, torch.bfloat16, (M, N), "y")
    rc = load().w4a16_linear_noalloc(_ptr(x), _ptr(packed), _ptr(scales), _ptr(zeros),
                                     _ptr(bias), _ptr(y), M, N, K, int(group_size),
                                     1 if zeros is None else 0, _stream(x, stream))
    _check("w4a16_linear_noalloc", rc)
    return y


def w4a8_quantize_act(x: torch.Tensor, group_size: int, qx=None, sx=None, stream=None):
    """Per-token INT8 activations: (qx [M, Kp] int8, sx [M] fp32)."""
    M, K = x.shape
    _need(x, torch.bfloat16, (M, K), "x")
    Kp = padded_k(K, group_size)
    if qx is None:
        qx = torch.empty(M, Kp, dtype=torch.int8, device=x.device)
    if sx is None:
        sx = torch.empty(M, dtype=torch.float32, device=x.device)
    _need(qx, torch.int8, (M, Kp), "qx")
    _need(sx, torch.float32, (M,), "sx")
    rc = load().w4a8_quantize_act(_ptr(x), M, K, int(group_size), _ptr(qx), _ptr(sx),
                                  _stream(x, stream))
    _check("w4a8_quantize_act", rc)
    return qx, sx


def w4a8_quantize_act_smooth(x: torch.Tensor, inv_s: torch.Tensor, group_size: int, qx=None,
                             sx=None, stream=None):
    """w4a8_quantize_act on x * inv_s (SmoothQuant) -> (qx [M, Kp] int8, sx [M] fp32)."""
    M, K = x.shape
    _need(x, torch.bfloat16, (M, K), "x")
    _need(inv_s, torch.float32, (K,), "inv_s")
    Kp = padded_k(K, group_size)
    if qx is None:
        qx = torch.empty(M, Kp, dtype=torch.int8, device=x.device)
    if sx is None:
        sx = torch.empty(M, dtype=torch.float32, device=x.device)
    _need(qx, torch.int8, (M, Kp), "qx")
    _need(sx, torch.float32, (M,), "sx")
    _check("w4a8_quantize_act_smooth", load().w4a8_quantize_act_smooth(
        _ptr(x), _ptr(inv_s), M, K, int(group_size), _ptr(qx), _ptr(sx), _stream(x, stream)))
    return qx, sx


def w4_smooth(X: torch.Tensor, W: torch.Tensor, alpha: float = 0.5, stream=None):
    """SmoothQuant calibration: returns (s, inv_s) [K] fp32 and multiplies
    the columns of W [N, K] fp32 (in place) by s."""
    T, K = X.shape
    N = W.shape[0]
    _need(X, torch.bfloat16, (T, K), "X")
    _need(W, torch.float32, (N, K), "W")
    s = torch.empty(K, dtype=torch.float32, device=W.device)
    inv_s = torch.empty(K, dtype=torch.float32, device=W.device)
    _check("w4_smooth", load().w4_smooth(_ptr(X), T, _ptr(W), N, K, float(alpha), _ptr(s),
                                         _ptr(inv_s), _stream(W, stream)))
    return s, inv_s


def w4_gptq(X: torch.Tensor, W: torch.Tensor, group_size: int, symmetric: bool,
            damp: float = 0.01, stream=None):
    """GPTQ of W [N, K] fp32 with calibration X [T, K] bf16 -> (packed
    [N, Kp/2] u8, scales [N, Ng] f32, zeros [N, Ng] u8 or None, loss [N] f32)."""
    T, K = X.shape
    N = W.shape[0]
    _need(X, torch.bfloat16, (T, K), "X")
    _need(W, torch.float32, (N, K), "W")
    Kp = padded_k(K, group_size)
    Ng = Kp // group_size
    dev = W.device
    packed = torch.empty(N, Kp // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(N, Ng, dtype=torch.float32, device=dev)
    zeros = None if symmetric else torch.empty(N, Ng, dtype=torch.uint8, device=dev)
    loss = torch.empty(N, dtype=torch.float32, device=dev)
    lib = load()
    nbytes = lib.w4_gptq_workspace_bytes(N, K, int(group_size))
    wsv = None                  # no size: the call reports why (group, shape)
    if nbytes:
        ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev)
        off = (-ws.data_ptr()) % 256
        wsv = ws[off:off + nbytes]
    _check("w4_gptq", lib.w4_gptq(_ptr(X), T, _ptr(W), N, K, int(group_size),
                                  1 if symmetric else 0, float(damp), _ptr(packed), _ptr(scales),
                                  _ptr(zeros), _ptr(loss), _ptr(wsv), nbytes, _stream(W, stream)))
    return packed, scales, zeros, loss


def w4a8_linear(qx: torch.Tensor, sx: torch.Tensor, packed: torch.Tensor,
                w_scales: torch.Tensor, bias: Optional[torch.Tensor], N: int, K: int,
                group_size: int, y=None, acc_out=None, want_acc: bool = False,
                workspace=None, stream=None):
    """(y [M, N] bf16, acc [M, N] int32 or None).  group_size == Kp: one
    weight scale per row (w_scales [N] or [N, 1]); smaller: group-wise
    (w_scales [N, Kp / group_size], no acc)."""
    M, Kp = qx.shape
    _need(qx, torch.int8, (M, padded_k(K, group_size)), "qx")
    _need(sx, torch.float32, (M,), "sx")
    _need(packed, torch.uint8, (N, Kp // 2), "packed")
    Ng = Kp // group_size
    w_scales = w_scales.reshape(N, Ng)
    _need(w_scales, torch.float32, (N, Ng), "w_scales")
    if bias is not None:
        _need(bias, torch.float32, (N,), "bias")
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=qx.device)
    _need(y, torch.bfloat16, (M, N), "y")
    if acc_out is None and want_acc:
        acc_out = torch.empty(M, N, dtype=torch.int32, device=qx.device)
    if acc_out is not None:
        _need(acc_out, torch.int32, (M, N), "acc_out")
    lib = load()
    _call_with_workspace(
        lib.w4a8_linear, "w4a8_linear",
        (_ptr(qx), _ptr(sx), _ptr(packed), _ptr(w_scales), _ptr(bias), _ptr(y), _ptr(acc_out),
         M, N, K, int(group_size)),
        (_stream(qx, stream),), qx.device, workspace,
        lambda: lib.w4a8_workspace_bytes(M, N, K, group_size))
    return y, acc_out


def w4_get_device_error(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load().w4_get_device_error(ctypes.c_void_p(s.cuda_stream)))


def w4_set_wait_limit(cycles: int, stream=None) -> None:
    """Limit (SM clock cycles) of the kernels' bounded waits on the current
    device; 0 restores the default (about one second)."""
    s = stream if stream is not None else torch.cuda.current_stream()
    _check("w4_set_wait_limit", load().w4_set_wait_limit(int(cycles), ctypes.c_void_p(s.cuda_stream)))


def w4_set_fault_injection(mode: int, stream=None) -> None:
    """Failure-test switch of the grouped decode kernel (0 off, 1 the group
    list is never published, 2 ring slots are never freed)."""
    s = stream if stream is not None else torch.cuda.current_stream()
    _check("w4_set_fault_injection",
           load().w4_set_fault_injection(int(mode), ctypes.c_void_p(s.cuda_stream)))
