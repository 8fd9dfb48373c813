// gemv_swiglu.cu - launches of the decode kernels with the SwiGLU epilogue
// (gate/up row pairs in, SiLU(gate) * up out); the kernels are in
// gemv_impl.cuh.  A separate translation unit: these instances compile in
// parallel with the others and leave their code untouched.
#include "gemv_impl.cuh"

namespace w4 {

int launch_w4a16_swiglu(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                        cudaStream_t st) {
    if (a.S > 1) return launch_w4a16_variant<true, true>(packed, a, p, st);
    return launch_w4a16_variant<false, true>(packed, a, p, st);
}

}  // namespace w4
