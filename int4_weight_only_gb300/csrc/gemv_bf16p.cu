// gemv_bf16p.cu - launches of the decode kernels for the bf16 parameter
// layout (bf16 scales and, asymmetric, bf16 (8 - z) s offsets); the kernels
// are in gemv_impl.cuh.  A separate translation unit: these instances
// compile in parallel with the others and leave their code untouched.
#include "gemv_impl.cuh"

namespace w4 {

int launch_w4a16_gemv_bf16p(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                            cudaStream_t st) {
    if (a.S > 1) return launch_w4a16_variant<true, false, false, true>(packed, a, p, st);
    return launch_w4a16_variant<false, false, false, true>(packed, a, p, st);
}

}  // namespace w4
