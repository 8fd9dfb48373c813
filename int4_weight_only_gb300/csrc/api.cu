// api.cu - the extern "C" entry points of libw4 (declared in include/w4.h):
// argument checks on the host, kernel selection, tensor-map encoding, and
// the device error flag.  No entry point allocates or frees device memory.
#include "w4_device.cuh"
#include "w4_internal.h"

#include <cstdlib>

#include <algorithm>
#include <cstddef>
#include <cstring>
#include <cudaTypedefs.h>
#include <mutex>

namespace w4 {

// error flag (set by bounded waits that give up and by data checks) and the
// wait limit, one block per device
__device__ DeviceStatus g_status = {0, 0, 0};

namespace {

constexpr int kMaxDevices = 64;

int device_index() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

int current_sm_count() {
    static int cache[kMaxDevices] = {0};
    const int d = device_index();
    if (d < 0) return 0;
    if (d < kMaxDevices && cache[d] > 0) return cache[d];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
    if (d < kMaxDevices) cache[d] = n;
    return n;
}

int* device_error_flag() {
    static int* cache[kMaxDevices] = {nullptr};
    const int d = device_index();
    if (d < 0) return nullptr;
    if (d < kMaxDevices && cache[d]) return cache[d];
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    if (d < kMaxDevices) cache[d] = static_cast<int*>(p);
    return static_cast<int*>(p);
}

// Recently encoded tensor maps, direct-mapped by a hash of every encoding
// input: a decode call on the same weights reuses its map instead of another
// driver call (a map depends on nothing but these inputs).
namespace {
struct TmapKey {
    int dtype, swizzle;
    const void* base;
    uint64_t dim0, dim1, stride;
    uint32_t box0, box1;
    bool operator==(const TmapKey& o) const {
        return dtype == o.dtype && swizzle == o.swizzle && base == o.base && dim0 == o.dim0 &&
               dim1 == o.dim1 && stride == o.stride && box0 == o.box0 && box1 == o.box1;
    }
};
struct TmapEntry {
    bool used = false;
    TmapKey key{};
    CUtensorMap map;
};
constexpr int kTmapSlots = 256;
TmapEntry g_tmaps[kTmapSlots];
std::mutex g_tmap_mu;

size_t tmap_hash(const TmapKey& k) {
    uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
    for (uint64_t v : {(uint64_t)k.dtype, (uint64_t)k.swizzle, k.dim0, k.dim1, k.stride,
                       (uint64_t)k.box0, (uint64_t)k.box1})
        h = (h ^ v) * 0x100000001B3ull;
    return (size_t)(h >> 17) % kTmapSlots;
}
}  // namespace

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t dim0, uint64_t dim1, uint64_t row_stride_bytes,
                    uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle) {
    const TmapKey key{(int)dtype, (int)swizzle, base, dim0, dim1, row_stride_bytes, box0, box1};
    const size_t slot = tmap_hash(key);
    {
        std::lock_guard<std::mutex> lk(g_tmap_mu);
        if (g_tmaps[slot].used && g_tmaps[slot].key == key) {
            *map = g_tmaps[slot].map;
            return true;
        }
    }
    auto fn = get_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {dim0, dim1};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box0, box1};
    cuuint32_t estr[2] = {1, 1};
    std::memset(map, 0, sizeof(*map));
    if (fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    g_tmaps[slot].used = true;
    g_tmaps[slot].key = key;
    g_tmaps[slot].map = *map;
    return true;
}

namespace {

int check_group(int K, int G) {
    if (G <= 0 || (G % 32) != 0) return W4_ERR_UNSUPPORTED_GROUP;
    if (K <= 0) return W4_ERR_INVALID_ARG;
    return W4_OK;
}

long long padded_k(int K, int G) { return ((long long)K + G - 1) / G * G; }

// Workspace layout: [counters: kCounterBytes][partials].
int split_workspace(const GemvPlan& p, void* ws, size_t ws_bytes, int** tickets, void** part) {
    *tickets = nullptr;
    *part = nullptr;
    if (p.S <= 1) return W4_OK;
    if (!ws) return W4_ERR_WORKSPACE;
    if (ws_bytes < p.ws_bytes) return W4_ERR_WORKSPACE;
    if (!aligned16(ws)) return W4_ERR_MISALIGNED;
    *tickets = static_cast<int*>(ws);
    *part = static_cast<uint8_t*>(ws) + kCounterBytes;
    return W4_OK;
}

}  // namespace
}  // namespace w4

using namespace w4;

extern "C" {

int w4_pack_rtn(const float* W, int N, int K, int group_size, int symmetric,
                uint8_t* packed, float* scales, uint8_t* zeros, void* stream) {
    if (!W || !packed || !scales) return W4_ERR_NULL_PTR;
    if (symmetric && zeros) return W4_ERR_INVALID_ARG;
    if (!symmetric && !zeros) return W4_ERR_NULL_PTR;
    if (N <= 0) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    if (padded_k(K, group_size) > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(packed)) return W4_ERR_MISALIGNED;
    if (!aligned4(W) || !aligned4(scales)) return W4_ERR_MISALIGNED;
    return launch_pack_rtn(W, N, K, group_size, symmetric ? 1 : 0, packed, scales, zeros,
                           nullptr, nullptr, static_cast<cudaStream_t>(stream));
}

int w4_pack_rtn_bf16(const float* W, int N, int K, int group_size, int symmetric,
                     uint8_t* packed, uint16_t* scales_b, uint16_t* offsets_b, void* stream) {
    if (!W || !packed || !scales_b) return W4_ERR_NULL_PTR;
    if (symmetric && offsets_b) return W4_ERR_INVALID_ARG;
    if (!symmetric && !offsets_b) return W4_ERR_NULL_PTR;
    if (N <= 0) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    if (padded_k(K, group_size) > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(packed)) return W4_ERR_MISALIGNED;
    if (!aligned4(W) || (reinterpret_cast<uintptr_t>(scales_b) & 1) ||
        (reinterpret_cast<uintptr_t>(offsets_b) & 1))
        return W4_ERR_MISALIGNED;
    return launch_pack_rtn(W, N, K, group_size, symmetric ? 1 : 0, packed, nullptr, nullptr,
                           scales_b, offsets_b, static_cast<cudaStream_t>(stream));
}

size_t w4a16_workspace_bytes(int M, int N, int K, int group_size) {
    if (M <= 0 || N <= 0 || check_group(K, group_size)) return 0;
    const long long Kp = padded_k(K, group_size);
    if (M <= 16) {
        GemvPlan p;
        if (!plan_gemv(M, N, (int)Kp, group_size, 2, current_sm_count(), &p)) return 0;
        return p.ws_bytes;
    }
    GemmPlan g;
    if (!plan_gemm(M, N, K, group_size, current_sm_count(), &g)) return 0;
    return g.ws_bytes;
}

int w4a16_linear(const uint16_t* x, const uint8_t* packed, const float* scales,
                 const uint8_t* zeros, const float* bias, uint16_t* y, int M, int N, int K,
                 int group_size, int symmetric, void* workspace, size_t workspace_bytes,
                 void* stream) {
    if (!x || !packed || !scales || !y) return W4_ERR_NULL_PTR;
    if (symmetric && zeros) return W4_ERR_INVALID_ARG;
    if (!symmetric && !zeros) return W4_ERR_NULL_PTR;
    if (M < 0 || N <= 0) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    const long long Kp = padded_k(K, group_size);
    if (Kp > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(packed)) return W4_ERR_MISALIGNED;
    if (!aligned4(scales) || (bias && !aligned4(bias)) || (reinterpret_cast<uintptr_t>(y) & 1))
        return W4_ERR_MISALIGNED;
    if (M == 0) return W4_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M > 16) {
        if (K % 8 != 0) return W4_ERR_UNSUPPORTED_SHAPE;
        GemmPlan g;
        if (!plan_gemm(M, N, K, group_size, current_sm_count(), &g)) return W4_ERR_UNSUPPORTED_SHAPE;
        if (g.S > 1) {
            if (!workspace || workspace_bytes < g.ws_bytes) return W4_ERR_WORKSPACE;
            if (!aligned16(workspace)) return W4_ERR_MISALIGNED;
        }
        int* err = device_error_flag();
        if (!err) return W4_ERR_CUDA;
        return launch_w4a16_gemm(x, packed, scales, zeros, bias, y, M, N, K, (int)Kp,
                                 group_size, g, workspace, err, st);
    }

    GemvPlan p;
    if (!plan_gemv(M, N, (int)Kp, group_size, 2, current_sm_count(), &p)) return W4_ERR_UNSUPPORTED_SHAPE;
    GemvArgs a{};
    rc = split_workspace(p, workspace, workspace_bytes, &a.tickets, &a.partial);
    if (rc) return rc;
    a.x = x; a.scales = scales; a.zeros = zeros; a.bias = bias; a.y = y;
    a.xtma = (K % 8) == 0 && gemv_tma_activations(p);
    a.err = device_error_flag();
    if (!a.err) return W4_ERR_CUDA;
    a.M = M; a.N = N; a.K = K; a.Kp = (int)Kp; a.G = group_size; a.Ng = (int)(Kp / group_size);
    a.R = p.R; a.SKE = p.SKE; a.nst = p.nst; a.S = p.S; a.spl = p.spl; a.units = p.units;
    a.XS = p.XS; a.red = p.red;
    return launch_w4a16_gemv(packed, a, p, st);
}

int w4a16_linear_partial(const uint16_t* x, const uint8_t* packed, const float* scales,
                         const uint8_t* zeros, float* y32, int M, int N, int K, int group_size,
                         int symmetric, void* workspace, size_t workspace_bytes, void* stream) {
    if (!x || !packed || !scales || !y32) return W4_ERR_NULL_PTR;
    if (symmetric && zeros) return W4_ERR_INVALID_ARG;
    if (!symmetric && !zeros) return W4_ERR_NULL_PTR;
    if (M < 0 || N <= 0) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    const long long Kp = padded_k(K, group_size);
    if (Kp > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(packed)) return W4_ERR_MISALIGNED;
    if (!aligned4(scales) || !aligned4(y32)) return W4_ERR_MISALIGNED;
    if (M == 0) return W4_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M > 16) {
        if (K % 8 != 0) return W4_ERR_UNSUPPORTED_SHAPE;
        GemmPlan g;
        if (!plan_gemm(M, N, K, group_size, current_sm_count(), &g)) return W4_ERR_UNSUPPORTED_SHAPE;
        if (g.S > 1) {
            if (!workspace || workspace_bytes < g.ws_bytes) return W4_ERR_WORKSPACE;
            if (!aligned16(workspace)) return W4_ERR_MISALIGNED;
        }
        int* err = device_error_flag();
        if (!err) return W4_ERR_CUDA;
        return launch_w4a16_gemm(x, packed, scales, zeros, nullptr, nullptr, M, N, K, (int)Kp,
                                 group_size, g, workspace, err, st, nullptr, nullptr, y32);
    }
    GemvPlan p;
    if (!plan_gemv(M, N, (int)Kp, group_size, 2, current_sm_count(), &p)) return W4_ERR_UNSUPPORTED_SHAPE;
    GemvArgs a{};
    rc = split_workspace(p, workspace, workspace_bytes, &a.tickets, &a.partial);
    if (rc) return rc;
    a.x = x; a.scales = scales; a.zeros = zeros; a.bias = nullptr; a.y = nullptr; a.y32 = y32;
    a.xtma = (K % 8) == 0 && gemv_tma_activations(p);
    a.err = device_error_flag();
    if (!a.err) return W4_ERR_CUDA;
    a.M = M; a.N = N; a.K = K; a.Kp = (int)Kp; a.G = group_size; a.Ng = (int)(Kp / group_size);
    a.R = p.R; a.SKE = p.SKE; a.nst = p.nst; a.S = p.S; a.spl = p.spl; a.units = p.units;
    a.XS = p.XS; a.red = p.red;
    return launch_w4a16_gemv_f32(packed, a, p, st);
}

int w4a16_partial_finish(const float* ysum, const float* bias, uint16_t* y, int M, int N,
                         void* stream) {
    if (!ysum || !y) return W4_ERR_NULL_PTR;
    if (M < 0 || N <= 0) return W4_ERR_INVALID_ARG;
    if (!aligned4(ysum) || (bias && !aligned4(bias)) || (reinterpret_cast<uintptr_t>(y) & 1))
        return W4_ERR_MISALIGNED;
    return launch_partial_finish(ysum, bias, y, M, N, static_cast<cudaStream_t>(stream));
}

int w4a16_linear_bf16p(const uint16_t* x, const uint8_t* packed, const uint16_t* scales_b,
                       const uint16_t* offsets_b, const float* bias, uint16_t* y, int M, int N,
                       int K, int group_size, void* workspace, size_t workspace_bytes,
                       void* stream) {
    if (!x || !packed || !scales_b || !y) return W4_ERR_NULL_PTR;
    if (M < 0 || N <= 0) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    const long long Kp = padded_k(K, group_size);
    if (Kp > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(packed) || !aligned16(scales_b) ||
        (offsets_b && !aligned16(offsets_b)))
        return W4_ERR_MISALIGNED;
    if ((bias && !aligned4(bias)) || (reinterpret_cast<uintptr_t>(y) & 1)) return W4_ERR_MISALIGNED;
    if (M == 0) return W4_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M > 16) {
        if (K % 8 != 0) return W4_ERR_UNSUPPORTED_SHAPE;
        GemmPlan g;
        if (!plan_gemm(M, N, K, group_size, current_sm_count(), &g)) return W4_ERR_UNSUPPORTED_SHAPE;
        if (g.S > 1) {
            if (!workspace || workspace_bytes < g.ws_bytes) return W4_ERR_WORKSPACE;
            if (!aligned16(workspace)) return W4_ERR_MISALIGNED;
        }
        int* err = device_error_flag();
        if (!err) return W4_ERR_CUDA;
        return launch_w4a16_gemm(x, packed, nullptr, nullptr, bias, y, M, N, K, (int)Kp,
                                 group_size, g, workspace, err, st, scales_b, offsets_b);
    }
    GemvPlan p;
    if (!plan_gemv(M, N, (int)Kp, group_size, 2, current_sm_count(), &p)) return W4_ERR_UNSUPPORTED_SHAPE;
    GemvArgs a{};
    rc = split_workspace(p, workspace, workspace_bytes, &a.tickets, &a.partial);
    if (rc) return rc;
    a.x = x; a.scales_b = scales_b; a.offs_b = offsets_b; a.bias = bias; a.y = y;
    a.xtma = (K % 8) == 0 && gemv_tma_activations(p);
    a.err = device_error_flag();
    if (!a.err) return W4_ERR_CUDA;
    a.M = M; a.N = N; a.K = K; a.Kp = (int)Kp; a.G = group_size; a.Ng = (int)(Kp / group_size);
    a.R = p.R; a.SKE = p.SKE; a.nst = p.nst; a.S = p.S; a.spl = p.spl; a.units = p.units;
    a.XS = p.XS; a.red = p.red;
    return launch_w4a16_gemv_bf16p(packed, a, p, st);
}

int w4a16_linear_swiglu(const uint16_t* x, const uint8_t* packed, const float* scales,
                        const uint8_t* zeros, const float* bias, uint16_t* y, int M, int F,
                        int K, int group_size, int symmetric, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if (!x || !packed || !scales || !y) return W4_ERR_NULL_PTR;
    if (symmetric && zeros) return W4_ERR_INVALID_ARG;
    if (!symmetric && !zeros) return W4_ERR_NULL_PTR;
    if (M < 0 || F <= 0 || (F % 8) != 0 || F > 0x3fffffff) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    const long long Kp = padded_k(K, group_size);
    if (Kp > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(packed)) return W4_ERR_MISALIGNED;
    if (!aligned4(scales) || (bias && !aligned4(bias)) || (reinterpret_cast<uintptr_t>(y) & 1))
        return W4_ERR_MISALIGNED;
    if (M > 16) return W4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return W4_OK;
    const int N = 2 * F;                        // gate/up row pairs
    GemvPlan p;
    if (!plan_gemv(M, N, (int)Kp, group_size, 2, current_sm_count(), &p)) return W4_ERR_UNSUPPORTED_SHAPE;
    GemvArgs a{};
    rc = split_workspace(p, workspace, workspace_bytes, &a.tickets, &a.partial);
    if (rc) return rc;
    a.x = x; a.scales = scales; a.zeros = zeros; a.bias = bias; a.y = y;
    a.xtma = (K % 8) == 0 && gemv_tma_activations(p);
    a.err = device_error_flag();
    if (!a.err) return W4_ERR_CUDA;
    a.M = M; a.N = N; a.K = K; a.Kp = (int)Kp; a.G = group_size; a.Ng = (int)(Kp / group_size);
    a.R = p.R; a.SKE = p.SKE; a.nst = p.nst; a.S = p.S; a.spl = p.spl; a.units = p.units;
    a.XS = p.XS; a.red = p.red;
    return launch_w4a16_swiglu(packed, a, p, static_cast<cudaStream_t>(stream));
}

int w4a16_linear_swiglu_q8(const uint16_t* x, const uint8_t* packed, const float* scales,
                           const uint8_t* zeros, const float* bias, uint16_t* y, int8_t* qx,
                           float* sx, int M, int F, int K, int group_size, int symmetric,
                           int q_group_size, void* workspace, size_t workspace_bytes,
                           void* stream) {
    if (!x || !packed || !scales || !y || !qx || !sx) return W4_ERR_NULL_PTR;
    if (symmetric && zeros) return W4_ERR_INVALID_ARG;
    if (!symmetric && !zeros) return W4_ERR_NULL_PTR;
    if (M < 0 || F <= 0 || (F % 8) != 0 || F > 0x3fffffff) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    if (q_group_size <= 0 || (q_group_size % 32) != 0) return W4_ERR_UNSUPPORTED_GROUP;
    const long long Kp = padded_k(K, group_size);
    const long long Fp = padded_k(F, q_group_size);
    if (Kp > 0x7fffffffLL || Fp > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(packed) || !aligned16(y) || !aligned16(qx))
        return W4_ERR_MISALIGNED;
    if (!aligned4(scales) || (bias && !aligned4(bias)) || !aligned4(sx)) return W4_ERR_MISALIGNED;
    if (M > 16) return W4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return W4_OK;
    const int N = 2 * F;                        // gate/up row pairs
    GemvPlan p;
    if (!plan_gemv(M, N, (int)Kp, group_size, 2, current_sm_count(), &p)) return W4_ERR_UNSUPPORTED_SHAPE;
    // the completion ticket sits in the counter prefix: a workspace is
    // needed even when the plan does not split K
    if (!workspace || workspace_bytes < std::max(p.ws_bytes, kCounterBytes)) return W4_ERR_WORKSPACE;
    if (!aligned16(workspace)) return W4_ERR_MISALIGNED;
    GemvArgs a{};
    rc = split_workspace(p, workspace, workspace_bytes, &a.tickets, &a.partial);
    if (rc) return rc;
    // the last 34 counters of the prefix: two buffers of 16 per-token maxima,
    // the call generation, the arrival counter
    a.done = static_cast<int*>(workspace) + (kMaxCounters - 1);
    a.ymax = reinterpret_cast<unsigned*>(static_cast<int*>(workspace) + (kMaxCounters - 34));
    // the grid-wide hand-off (cooperative launch); W4_GEMV_COOP=0 keeps the
    // last-CTA path, for tests of both
    const char* ecoop = std::getenv("W4_GEMV_COOP");
    a.coop = (ecoop && std::atoi(ecoop) == 0) ? 0 : 1;
    a.qx = qx; a.sx_out = sx; a.Fp = (int)Fp;
    a.x = x; a.scales = scales; a.zeros = zeros; a.bias = bias; a.y = y;
    a.xtma = (K % 8) == 0 && gemv_tma_activations(p);
    a.err = device_error_flag();
    if (!a.err) return W4_ERR_CUDA;
    a.M = M; a.N = N; a.K = K; a.Kp = (int)Kp; a.G = group_size; a.Ng = (int)(Kp / group_size);
    a.R = p.R; a.SKE = p.SKE; a.nst = p.nst; a.S = p.S; a.spl = p.spl; a.units = p.units;
    a.XS = p.XS; a.red = p.red;
    return launch_w4a16_swiglu_q8(packed, a, p, static_cast<cudaStream_t>(stream));
}

int w4a16_grouped_linear(const uint16_t* x, const int32_t* goff, const uint8_t* packed,
                         const float* scales, const uint8_t* zeros, const float* bias,
                         uint16_t* y, int T, int E, int N, int K, int group_size, int symmetric,
                         int tile_tokens, void* stream) {
    if (!x || !goff || !packed || !scales || !y) return W4_ERR_NULL_PTR;
    if (symmetric && zeros) return W4_ERR_INVALID_ARG;
    if (!symmetric && !zeros) return W4_ERR_NULL_PTR;
    if (T < 0 || E <= 0 || E > 32767 || N <= 0 || tile_tokens < 1 || tile_tokens > 256)
        return W4_ERR_INVALID_ARG;
    if (tile_tokens <= 16 && T / tile_tokens >= 65536) return W4_ERR_UNSUPPORTED_SHAPE;   // 16-bit tile index
    if ((long long)E * N > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    const long long Kp = padded_k(K, group_size);
    if (Kp > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(packed)) return W4_ERR_MISALIGNED;
    if (!aligned4(goff) || !aligned4(scales) || (bias && !aligned4(bias)) ||
        (reinterpret_cast<uintptr_t>(y) & 1))
        return W4_ERR_MISALIGNED;
    if (T == 0) return W4_OK;
    if (tile_tokens > 16) {
        // groups of many tokens: tensor-core tiles of 64 or 256 tokens, each
        // group's weights dequantized once per tile
        if (K % 8 != 0) return W4_ERR_UNSUPPORTED_SHAPE;
        int* err = device_error_flag();
        if (!err) return W4_ERR_CUDA;
        return launch_w4a16_grouped_gemm(x, goff, packed, scales, zeros, bias, y, T, E, N, K,
                                         (int)Kp, group_size, tile_tokens, err,
                                         static_cast<cudaStream_t>(stream));
    }
    // at most E + T / tile items (each has a token); plan for their rows
    const long long items = std::min<long long>(T, (long long)E + (T + tile_tokens - 1) / tile_tokens);
    const long long n_eff = std::min(items * N, 0x7fffffffLL);
    const int cap = (int)((long long)E + (T + tile_tokens - 1) / tile_tokens);
    GemvPlan p;
    if (!plan_gemv(tile_tokens, (int)n_eff, (int)Kp, group_size, 2, current_sm_count(), &p, cap))
        return W4_ERR_UNSUPPORTED_SHAPE;
    GemvArgs a{};
    a.x = x; a.scales = scales; a.zeros = zeros; a.bias = bias; a.y = y;
    a.err = device_error_flag();
    if (!a.err) return W4_ERR_CUDA;
    a.M = T; a.N = N; a.K = K; a.Kp = (int)Kp; a.G = group_size; a.Ng = (int)(Kp / group_size);
    a.R = p.R; a.SKE = p.SKE; a.nst = p.nst; a.S = 1; a.spl = p.spl; a.units = p.units;
    a.XS = p.XS; a.red = p.red;
    a.goff = goff; a.E = E; a.gmax = tile_tokens; a.NBg = (N + p.R - 1) / p.R;
    a.list_off = (int)p.list_off;
    a.list_cap = cap;
    return launch_w4a16_grouped(packed, a, p, static_cast<cudaStream_t>(stream));
}

size_t w4_gptq_workspace_bytes(int N, int K, int group_size) {
    if (N <= 0 || check_group(K, group_size)) return 0;
    const long long Kp = padded_k(K, group_size);
    if (Kp > 65536) return 0;
    return gptq_workspace_bytes(N, (int)Kp, gptq_block_cols(group_size));
}

int w4_gptq(const uint16_t* X, int T, const float* W, int N, int K, int group_size,
            int symmetric, float damp, uint8_t* packed, float* scales, uint8_t* zeros,
            float* loss, void* workspace, size_t workspace_bytes, void* stream) {
    if (!X || !W || !packed || !scales || !loss) return W4_ERR_NULL_PTR;
    if (symmetric && zeros) return W4_ERR_INVALID_ARG;
    if (!symmetric && !zeros) return W4_ERR_NULL_PTR;
    if (T < 1 || N <= 0 || !(damp >= 0.f)) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    const long long Kp = padded_k(K, group_size);
    if (Kp > 65536) return W4_ERR_UNSUPPORTED_SHAPE;      // two Kp x Kp fp32 matrices
    if (!workspace || workspace_bytes < w4_gptq_workspace_bytes(N, K, group_size))
        return W4_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) || !aligned4(W) || !aligned4(scales) ||
        !aligned4(loss) || (reinterpret_cast<uintptr_t>(X) & 1))
        return W4_ERR_MISALIGNED;
    int* err = device_error_flag();
    if (!err) return W4_ERR_CUDA;
    return launch_gptq(X, T, W, N, K, (int)Kp, group_size, symmetric, damp, packed, scales, zeros,
                       loss, workspace, err, static_cast<cudaStream_t>(stream));
}

int w4a8_quantize_act(const uint16_t* x, int M, int K, int group_size, int8_t* qx,
                      float* sx, void* stream) {
    if (!x || !qx || !sx) return W4_ERR_NULL_PTR;
    if (M < 0) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    const long long Kp = padded_k(K, group_size);
    if (Kp > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(qx) || !aligned4(sx) || (reinterpret_cast<uintptr_t>(x) & 1))
        return W4_ERR_MISALIGNED;
    if (M == 0) return W4_OK;
    return launch_act_quant(x, nullptr, M, K, (int)Kp, qx, sx, static_cast<cudaStream_t>(stream));
}

int w4a8_quantize_act_smooth(const uint16_t* x, const float* inv_s, int M, int K,
                             int group_size, int8_t* qx, float* sx, void* stream) {
    if (!x || !inv_s || !qx || !sx) return W4_ERR_NULL_PTR;
    if (M < 0) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    const long long Kp = padded_k(K, group_size);
    if (Kp > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(qx) || !aligned16(inv_s) || !aligned4(sx) ||
        (reinterpret_cast<uintptr_t>(x) & 1))
        return W4_ERR_MISALIGNED;
    if (M == 0) return W4_OK;
    return launch_act_quant(x, inv_s, M, K, (int)Kp, qx, sx, static_cast<cudaStream_t>(stream));
}

int w4_smooth(const uint16_t* X, int T, float* W, int N, int K, float alpha, float* s,
              float* inv_s, void* stream) {
    if (!W || !s || !inv_s || (T > 0 && !X)) return W4_ERR_NULL_PTR;
    if (T < 0 || N <= 0 || K <= 0 || !(alpha >= 0.f && alpha <= 1.f)) return W4_ERR_INVALID_ARG;
    if ((long long)N * K > 0x7fffffffLL * 256LL || (long long)T * K > 0x7fffffffffffLL)
        return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned4(W) || !aligned4(s) || !aligned4(inv_s) ||
        (reinterpret_cast<uintptr_t>(X) & 1))
        return W4_ERR_MISALIGNED;
    return launch_smooth(X, T, W, N, K, alpha, s, inv_s, static_cast<cudaStream_t>(stream));
}

size_t w4a8_workspace_bytes(int M, int N, int K, int group_size) {
    if (M <= 0 || M > 16 || N <= 0 || check_group(K, group_size)) return 0;
    GemvPlan p;
    if (!plan_gemv(M, N, (int)padded_k(K, group_size), group_size, 1, current_sm_count(), &p)) return 0;
    return p.ws_bytes;
}

int w4_decode_plan(int kind, int M, int N, int K, int group_size, int sm_count,
                   long long* out) {
    if (!out) return W4_ERR_NULL_PTR;
    if ((kind != 0 && kind != 1) || M < 1 || M > 16 || N <= 0 || sm_count < 1)
        return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    const long long Kp = padded_k(K, group_size);
    if (Kp > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    if (kind == 1) {
        if (Kp != group_size && !w4a8_group_supported(group_size)) return W4_ERR_UNSUPPORTED_GROUP;
        if (Kp > W4_W4A8_MAX_KP) return W4_ERR_K_TOO_LARGE;
    }
    GemvPlan p;
    if (!plan_gemv(M, N, (int)Kp, group_size, kind == 0 ? 2 : 1, sm_count, &p))
        return W4_ERR_UNSUPPORTED_SHAPE;
    const long long v[W4_DECODE_PLAN_FIELDS] = {
        p.R, p.S, p.spl, p.nst, p.SKE, p.units, p.grid, p.cps, (long long)p.smem,
        (long long)p.ws_bytes, p.f16 ? 1 : 0, p.csplit ? 1 : 0};
    for (int i = 0; i < W4_DECODE_PLAN_FIELDS; ++i) out[i] = v[i];
    return W4_OK;
}

int w4a8_linear(const int8_t* qx, const float* sx, const uint8_t* packed,
                const float* w_scales, const float* bias, uint16_t* y, int32_t* acc_out,
                int M, int N, int K, int group_size, void* workspace, size_t workspace_bytes,
                void* stream) {
    if (!qx || !sx || !packed || !w_scales || !y) return W4_ERR_NULL_PTR;
    if (M < 0 || N <= 0) return W4_ERR_INVALID_ARG;
    int rc = check_group(K, group_size);
    if (rc) return rc;
    const long long Kp = padded_k(K, group_size);
    // one group per row (the integer path with exact int32 accumulators), or
    // group-wise scales (fp32 sums of the groups' integer partials)
    const bool grouped = Kp != group_size;
    if (grouped && !w4a8_group_supported(group_size)) return W4_ERR_UNSUPPORTED_GROUP;
    if (grouped && acc_out) return W4_ERR_INVALID_ARG;
    if (Kp > W4_W4A8_MAX_KP) return W4_ERR_K_TOO_LARGE;
    if (!aligned16(qx) || !aligned16(packed)) return W4_ERR_MISALIGNED;
    if (!aligned4(sx) || !aligned4(w_scales) || (bias && !aligned4(bias)) ||
        (acc_out && !aligned4(acc_out)) || (reinterpret_cast<uintptr_t>(y) & 1))
        return W4_ERR_MISALIGNED;
    if (M == 0) return W4_OK;
    if (M > 16) return W4_ERR_UNSUPPORTED_SHAPE;
    GemvPlan p;
    if (!plan_gemv(M, N, (int)Kp, group_size, 1, current_sm_count(), &p)) return W4_ERR_UNSUPPORTED_SHAPE;
    GemvArgs a{};
    rc = split_workspace(p, workspace, workspace_bytes, &a.tickets, &a.partial);
    if (rc) return rc;
    a.x = qx; a.sx = sx; a.scales = w_scales; a.bias = bias; a.y = y; a.acc_out = acc_out;
    a.err = device_error_flag();
    if (!a.err) return W4_ERR_CUDA;
    a.M = M; a.N = N; a.K = K; a.Kp = (int)Kp; a.G = group_size;
    a.Ng = (int)(Kp / group_size);
    a.R = p.R; a.SKE = p.SKE; a.nst = p.nst; a.S = p.S; a.spl = p.spl; a.units = p.units;
    a.XS = p.XS; a.red = p.red;
    if (grouped) return launch_w4a8g_gemv(packed, a, p, static_cast<cudaStream_t>(stream));
    return launch_w4a8_gemv(packed, a, p, static_cast<cudaStream_t>(stream));
}

int w4_get_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W4_ERR_CUDA;
    int* flag = device_error_flag();
    if (!flag) return W4_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return W4_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(flag, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return W4_ERR_CUDA;
    return v;
}

int w4_set_wait_limit(long long cycles, void* stream) {
    int* flag = device_error_flag();
    if (!flag) return W4_ERR_CUDA;
    const long long v = cycles > 0 ? cycles : 0;
    char* block = reinterpret_cast<char*>(flag);
    if (cudaMemcpyAsync(block + offsetof(DeviceStatus, wait_limit), &v, sizeof(v),
                        cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W4_ERR_CUDA;
    return W4_OK;
}

int w4_set_fault_injection(int mode, void* stream) {
    if (mode < 0 || mode > (kInjectNoList | kInjectNoRelease)) return W4_ERR_INVALID_ARG;
    int* flag = device_error_flag();
    if (!flag) return W4_ERR_CUDA;
    char* block = reinterpret_cast<char*>(flag);
    if (cudaMemcpyAsync(block + offsetof(DeviceStatus, inject), &mode, sizeof(mode),
                        cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return W4_ERR_CUDA;
    return W4_OK;
}

const char* w4_error_string(int code) {
    switch (code) {
        case W4_OK: return "ok";
        case W4_ERR_INVALID_ARG: return "invalid argument (size or flag out of range)";
        case W4_ERR_NULL_PTR: return "a required pointer is NULL";
        case W4_ERR_MISALIGNED: return "pointer misaligned (packed, x and qx need 16 bytes)";
        case W4_ERR_UNSUPPORTED_GROUP:
            return "group_size must be a positive multiple of 32 (W4A8: one group per row)";
        case W4_ERR_K_TOO_LARGE: return "padded K exceeds the int32 accumulator bound";
        case W4_ERR_WORKSPACE: return "workspace missing or smaller than required";
        case W4_ERR_CUDA: return "CUDA runtime error";
        case W4_ERR_UNSUPPORTED_SHAPE: return "shape not supported by the kernels";
        case W4_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait timed out";
        case W4_ERR_SCRATCH_LIMIT:
            return "shape needs more split-K scratch than W4_NOALLOC_SCRATCH_BYTES";
        case W4_ERR_NOT_SPD:
            return "GPTQ met a non-positive Cholesky pivot (damped Hessian not positive definite)";
        case W4_ERR_GROUP_TOKENS:
            return "a group's token offsets were invalid (outside [0, T] or decreasing)";
        default: return "unknown error code";
    }
}

}  // extern "C"
