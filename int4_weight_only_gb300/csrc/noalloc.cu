// noalloc.cu - w4a16_linear_noalloc: the decode path of w4a16_linear
// (M <= 16) with its split-K scratch taken from a fixed array that lives in
// the library itself, so the caller never provides or allocates a workspace.
//
// Some callers cannot allocate device memory at all: hosts that hand a
// plugin only its input and output buffers, and runtimes that forbid
// cudaMalloc after start-up because it can synchronize the device and can
// fail under a fixed memory budget.  This entry point serves them.
//
// The scratch below is a file-scope device array of W4_NOALLOC_SCRATCH_BYTES
// that every GPU loading the library keeps until process exit.  Every call
// uses the same array, so calls that overlap on the GPU (other streams,
// other host threads) race on it and must be serialized by the caller.
#include "w4_internal.h"

#include <mutex>

// Split-K scratch of w4a16_linear_noalloc (arrival counters, then partial
// sums); zero-initialized when the module loads, shared by every call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[W4_NOALLOC_SCRATCH_BYTES];

namespace w4 {
namespace {

constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDev] = {nullptr};

// Device address of the scratch array on the current device.  Resolved once
// per device (with that device current) on the first call; in host code the
// array's name is only a host-side stand-in and must never reach a kernel.
int scratch_address(void** out) {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDev) return W4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[d]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return W4_ERR_CUDA;
        g_scratch_ptr[d] = p;
    }
    *out = g_scratch_ptr[d];
    return W4_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace w4

using namespace w4;

extern "C" int w4a16_linear_noalloc(const uint16_t* x, const uint8_t* packed,
                                    const float* scales, const uint8_t* zeros,
                                    const float* bias, uint16_t* y, int M, int N, int K,
                                    int group_size, int symmetric, void* stream) {
    if (!x || !packed || !scales || !y) return W4_ERR_NULL_PTR;
    if (symmetric && zeros) return W4_ERR_INVALID_ARG;
    if (!symmetric && !zeros) return W4_ERR_NULL_PTR;
    if (M < 0 || N <= 0 || K <= 0) return W4_ERR_INVALID_ARG;
    if (group_size <= 0 || (group_size % 32) != 0) return W4_ERR_UNSUPPORTED_GROUP;
    const long long Kp = ((long long)K + group_size - 1) / group_size * group_size;
    if (Kp > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!al16(x) || !al16(packed)) return W4_ERR_MISALIGNED;
    if (!al4(scales) || (bias && !al4(bias)) || (reinterpret_cast<uintptr_t>(y) & 1))
        return W4_ERR_MISALIGNED;
    if (M == 0) return W4_OK;
    if (M > 16) return W4_ERR_UNSUPPORTED_SHAPE;

    GemvPlan p;
    if (!plan_gemv(M, N, (int)Kp, group_size, 2, current_sm_count(), &p)) return W4_ERR_UNSUPPORTED_SHAPE;
    if (p.ws_bytes > (size_t)W4_NOALLOC_SCRATCH_BYTES) return W4_ERR_SCRATCH_LIMIT;

    GemvArgs a{};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (p.S > 1) {
        void* base = nullptr;
        int rc = scratch_address(&base);
        if (rc) return rc;
        const size_t ticket_bytes = ((size_t)p.NB * 4 + 255) / 256 * 256;   // counters in use
        // the clear must stay inside the counter prefix, below the partial sums
        if (ticket_bytes > kCounterBytes) return W4_ERR_UNSUPPORTED_SHAPE;
        // The arrival counters must start at zero; the array keeps whatever
        // the previous call left, so clear them in stream order first.
        if (cudaMemsetAsync(base, 0, ticket_bytes, st) != cudaSuccess) return W4_ERR_CUDA;
        a.tickets = static_cast<int*>(base);
        a.partial = static_cast<unsigned char*>(base) + kCounterBytes;
    }
    a.x = x; a.scales = scales; a.zeros = zeros; a.bias = bias; a.y = y;
    a.xtma = (K % 8) == 0 && gemv_tma_activations(p);
    a.err = device_error_flag();
    if (!a.err) return W4_ERR_CUDA;
    a.M = M; a.N = N; a.K = K; a.Kp = (int)Kp; a.G = group_size;
    a.Ng = (int)(Kp / group_size);
    a.R = p.R; a.SKE = p.SKE; a.nst = p.nst; a.S = p.S; a.spl = p.spl; a.units = p.units;
    a.XS = p.XS; a.red = p.red;
    return launch_w4a16_gemv(packed, a, p, st);
}
