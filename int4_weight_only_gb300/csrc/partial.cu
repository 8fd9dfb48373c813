// partial.cu - the last step of a row-parallel (K-split) linear layer: the
// fp32 partial sums of the shards, already added across shards, plus the
// bias, rounded once to bf16.
//
// A layer y = x W_hat^T + b whose input columns are split into group-aligned
// slices computes on each shard the fp32 partial x_s W_hat_s^T
// (w4a16_linear_partial); the partials are summed across shards by one
// all-reduce, and this kernel adds b and rounds.  Elementwise and HBM-bound:
// 4 + 2 bytes per output (+ 4 per column of bias).
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

// four outputs per thread when N % 4 == 0 (16-byte loads), else one
template <int V>
__global__ void __launch_bounds__(256)
k_partial_finish(const float* __restrict__ ysum, const float* __restrict__ bias,
                 uint16_t* __restrict__ y, long long total, int N) {
    const long long i0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * V;
    if (i0 >= total) return;
    if constexpr (V == 4) {
        const float4 v = *reinterpret_cast<const float4*>(ysum + i0);
        const int n = (int)(i0 % N);
        float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
        if (bias) b = *reinterpret_cast<const float4*>(bias + n);
        const uint32_t lo = (uint32_t)f32_to_bf16_bits(v.x + b.x) |
                            ((uint32_t)f32_to_bf16_bits(v.y + b.y) << 16);
        const uint32_t hi = (uint32_t)f32_to_bf16_bits(v.z + b.z) |
                            ((uint32_t)f32_to_bf16_bits(v.w + b.w) << 16);
        *reinterpret_cast<uint2*>(y + i0) = make_uint2(lo, hi);
    } else {
        const int n = (int)(i0 % N);
        y[i0] = f32_to_bf16_bits(ysum[i0] + (bias ? bias[n] : 0.f));
    }
}

}  // namespace

int launch_partial_finish(const float* ysum, const float* bias, uint16_t* y, int M, int N,
                          cudaStream_t st) {
    const long long total = (long long)M * N;
    if (total == 0) return W4_OK;
    const bool vec = (N % 4) == 0 && (reinterpret_cast<uintptr_t>(ysum) & 15) == 0 &&
                     (!bias || (reinterpret_cast<uintptr_t>(bias) & 15) == 0) &&
                     (reinterpret_cast<uintptr_t>(y) & 7) == 0;
    const int V = vec ? 4 : 1;
    const long long threads = (total + V - 1) / V;
    const unsigned grid = (unsigned)((threads + 255) / 256);
    if (vec) k_partial_finish<4><<<grid, 256, 0, st>>>(ysum, bias, y, total, N);
    else k_partial_finish<1><<<grid, 256, 0, st>>>(ysum, bias, y, total, N);
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

}  // namespace w4
