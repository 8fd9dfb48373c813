// gemv_split.cu - launches of the W4A16 decode kernels for K-split plans
// (a separate translation unit so that the two halves compile in parallel);
// the kernels are in gemv_impl.cuh.
#include "gemv_impl.cuh"

namespace w4 {

int launch_w4a16_gemv_split(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                            cudaStream_t st) {
    return launch_w4a16_variant<true>(packed, a, p, st);
}

}  // namespace w4
