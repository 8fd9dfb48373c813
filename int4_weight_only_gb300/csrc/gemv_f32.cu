// gemv_f32.cu - launches of the W4A16 decode kernels that write fp32 outputs
// without the bias: the partial sums of a row-parallel shard of a layer,
// which the shards add (all-reduce) before w4a16_partial_finish.  Their own
// translation unit, so that the plain instances keep their code generation.
#include "gemv_impl.cuh"

namespace w4 {

int launch_w4a16_gemv_f32(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                          cudaStream_t st) {
    if (a.S > 1) return launch_w4a16_variant<true, false, false, false, true>(packed, a, p, st);
    return launch_w4a16_variant<false, false, false, false, true>(packed, a, p, st);
}

}  // namespace w4
