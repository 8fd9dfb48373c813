// gemv_grouped.cu - launches of the grouped decode kernels (one matrix per
// group of tokens, e.g. the experts of a mixture-of-experts layer); the
// kernels are in gemv_impl.cuh.  A separate translation unit: these
// instances compile in parallel with the others and leave their code
// untouched.
#include "gemv_impl.cuh"

namespace w4 {

int launch_w4a16_grouped(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                         cudaStream_t st) {
    return launch_w4a16_variant<false, false, true>(packed, a, p, st);
}

}  // namespace w4
