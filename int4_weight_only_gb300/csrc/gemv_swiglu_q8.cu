// gemv_swiglu_q8.cu - launches of the fused gate|up + SiLU decode kernels
// whose last CTA to finish also writes the INT8 activations of the W4A8
// down projection (Q8 instances; kernels in gemv_impl.cuh).  Their own
// translation unit, so that the other instances keep their code generation.
#include "gemv_impl.cuh"

namespace w4 {

int launch_w4a16_swiglu_q8(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                           cudaStream_t st) {
    if (a.S > 1) return launch_w4a16_variant<true, true, false, false, false, true>(packed, a, p, st);
    return launch_w4a16_variant<false, true, false, false, false, true>(packed, a, p, st);
}

}  // namespace w4
