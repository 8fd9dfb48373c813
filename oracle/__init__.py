"""CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does.
"""
from .w4_oracle import (padded_k, rtn_params, rtn_codes, rtn_quantize, pack_nibbles, unpack_nibbles,
                        pack_rtn, dequantize_f64, bf16_to_f64, w4a16_linear,
                        swiglu_rows, pair_rows, silu_f64, w4a16_linear_swiglu,
                        w4a16_grouped_linear,
                        w4a8_quantize_act, w4a8_linear, int32_worst_case,
                        smooth_factors, w4a8_linear_grouped,
                        gptq_hessian, gptq_quantize, round_bf16, pack_rtn_bf16,
                        dequantize_bf16_params, w4a16_linear_bf16_params)

__all__ = ["padded_k", "rtn_params", "rtn_codes", "rtn_quantize", "pack_nibbles", "unpack_nibbles",
           "pack_rtn", "dequantize_f64", "bf16_to_f64", "w4a16_linear",
           "swiglu_rows", "pair_rows", "silu_f64", "w4a16_linear_swiglu",
           "w4a16_grouped_linear",
           "w4a8_quantize_act", "w4a8_linear", "int32_worst_case",
           "smooth_factors", "w4a8_linear_grouped",
           "gptq_hessian", "gptq_quantize", "round_bf16", "pack_rtn_bf16",
           "dequantize_bf16_params", "w4a16_linear_bf16_params"]
