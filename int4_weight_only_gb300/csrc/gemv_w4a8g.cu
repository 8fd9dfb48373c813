// gemv_w4a8g.cu - launches of the group-wise W4A8 decode kernels (one fp32
// weight scale per group of G input columns); the kernels are in
// gemv_impl.cuh.  A separate translation unit: these instances compile in
// parallel with the others and leave their code untouched.
#include "gemv_impl.cuh"

namespace w4 {

namespace {
template <int CPGW>
int launch_w4a8g_m(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p, cudaStream_t st) {
    if (a.M <= 1) return launch(k_w4a8g_gemv_m4<1, CPGW>, packed, a, p, st);
    if (a.M <= 2) return launch(k_w4a8g_gemv_m4<2, CPGW>, packed, a, p, st);
    if (a.M <= 4) return launch(k_w4a8g_gemv_m4<4, CPGW>, packed, a, p, st);
    if (a.M <= 8) return launch(k_w4a8g_gemv_m16<8, CPGW>, packed, a, p, st);
    return launch(k_w4a8g_gemv_m16<16, CPGW>, packed, a, p, st);
}
}  // namespace

bool w4a8_group_supported(int G) {
    return G == 32 || G == 64 || G == 128 || (G > 0 && G % 256 == 0);
}

int launch_w4a8g_gemv(const uint8_t* packed, const GemvArgs& a, const GemvPlan& p,
                      cudaStream_t st) {
    switch (a.G) {
        case 32: return launch_w4a8g_m<1>(packed, a, p, st);
        case 64: return launch_w4a8g_m<2>(packed, a, p, st);
        case 128: return launch_w4a8g_m<4>(packed, a, p, st);
        default: return launch_w4a8g_m<8>(packed, a, p, st);
    }
}

}  // namespace w4
