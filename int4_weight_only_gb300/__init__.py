"""Python binding of libw4 (the INT4 weight-only linear layer for GB300).

The functions here carry the names of the C entry points in ``include/w4.h``
and only marshal arguments: they check dtypes and shapes of torch CUDA
tensors, allocate outputs with torch when the caller passes none, and call
the library through ctypes on the current torch stream.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.
"""
from ._lib import (W4Error, lib_path, load, w4_pack_rtn, w4a16_workspace_bytes,
                   w4a16_linear, w4a16_linear_noalloc, w4a16_linear_swiglu, w4a16_linear_swiglu_q8,
                   pair_gate_up,
                   w4a16_linear_partial, w4a16_partial_finish,
                   w4_pack_rtn_bf16, w4a16_linear_bf16p,
                   w4a16_grouped_linear, w4a8_quantize_act, w4a8_workspace_bytes, w4a8_linear,
                   w4_decode_plan, DECODE_PLAN_FIELDS,
                   w4a8_quantize_act_smooth, w4_smooth, w4_gptq,
                   w4_get_device_error, w4_set_wait_limit, w4_set_fault_injection,
                   w4_error_string, padded_k,
                   EXPORTED)

__all__ = ["W4Error", "lib_path", "load", "w4_pack_rtn", "w4a16_workspace_bytes",
           "w4a16_linear", "w4a16_linear_noalloc", "w4a16_linear_swiglu", "w4a16_linear_swiglu_q8",
           "pair_gate_up",
           "w4a16_linear_partial", "w4a16_partial_finish",
           "w4_pack_rtn_bf16", "w4a16_linear_bf16p",
           "w4a16_grouped_linear", "w4a8_quantize_act", "w4a8_workspace_bytes", "w4a8_linear",
           "w4_decode_plan", "DECODE_PLAN_FIELDS",
           "w4a8_quantize_act_smooth", "w4_smooth", "w4_gptq",
           "w4_get_device_error", "w4_set_wait_limit", "w4_set_fault_injection", "w4_error_string", "padded_k",
           "EXPORTED"]
