// quant.cu - RTN INT4 quantize + pack of the weights, and dynamic INT8
// quantization of the activations.
//
// Weights ("Lab 5: Gemma4 端到端推理优化", section "INT4 线性量化"): per
// (output channel, group of group_size input columns), symmetric
// s = max|r| / 7 with codes round(r/s) + 8 clipped to [0, 15], or asymmetric
// s = (r_max - r_min) / 15, z = round(-r_min / s), code = round(r/s + z)
// clipped to [0, 15].  Two codes per byte, earlier column in the low nibble;
// the padded columns K..Kp-1 take part as zeros.
//
// Activations ("Jetson Orin AGX INT4 推理优化实践", section
// "从 FP 线性层到 INT4 DP4A 的数学推导"): s_x = max|x| / 127,
// q_x = clip(round(x / s_x), -127, 127) per token.
//
// Every division is an explicit IEEE round-to-nearest fp32 division and
// rint() rounds half to even, so the codes are reproducible bit for bit by
// any scalar fp32 evaluation of the same formulas.
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One warp per (row n, group g).
__global__ void __launch_bounds__(256)
k_pack_rtn(const float* __restrict__ W, int N, int K, int G, int Ng, int symmetric,
           uint8_t* __restrict__ packed, float* __restrict__ scales,
           uint8_t* __restrict__ zeros) {
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= (long long)N * Ng) return;
    const int n = (int)(wid / Ng), g = (int)(wid - (long long)n * Ng);
    const int k0 = g * G;
    const float* row = W + (size_t)n * K;
    const int Kp2 = Ng * G / 2;

    float mx = 0.f, mn = 0.f;   // pads are zeros, so 0 is always a member
    for (int k = k0 + lane; k < k0 + G; k += 32) {
        const float r = k < K ? __ldg(row + k) : 0.f;
        if (symmetric) {
            mx = fmaxf(mx, fabsf(r));
        } else {
            mx = fmaxf(mx, r);
            mn = fminf(mn, r);
        }
    }
    mx = warp_max(mx);
    float s, z = 0.f;
    if (symmetric) {
        s = __fdiv_rn(mx, 7.0f);
    } else {
        mn = warp_min(mn);
        s = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
        if (s != 0.f) z = fminf(fmaxf(rintf(__fdiv_rn(-mn, s)), 0.f), 15.f);
    }
    if (lane == 0) {
        scales[(size_t)n * Ng + g] = s;
        if (!symmetric) zeros[(size_t)n * Ng + g] = (uint8_t)z;
    }
    // each lane packs 8 consecutive columns into one 32-bit word
    for (int k = k0 + lane * 8; k < k0 + G; k += 256) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float r = (k + j) < K ? __ldg(row + k + j) : 0.f;
            uint32_t code;
            if (symmetric) {
                code = 8;
                if (s != 0.f) code = (uint32_t)((int)fminf(fmaxf(rintf(__fdiv_rn(r, s)), -8.f), 7.f) + 8);
            } else {
                code = 0;
                if (s != 0.f)
                    code = (uint32_t)fminf(fmaxf(rintf(__fadd_rn(__fdiv_rn(r, s), z)), 0.f), 15.f);
            }
            word |= code << (4 * j);
        }
        *reinterpret_cast<uint32_t*>(packed + (size_t)n * Kp2 + k / 2) = word;
    }
}

// One CTA of 1024 threads per token: the max|x| pass and the quantize pass
// both read x with 16-byte loads where the row allows it (the second pass
// hits L1/L2).
constexpr int kActThreads = 1024;

__global__ void __launch_bounds__(kActThreads)
k_act_quant(const uint16_t* __restrict__ x, int K, int Kp, int8_t* __restrict__ qx,
            float* __restrict__ sx) {
    __shared__ float red[kActThreads / 32];
    const int m = blockIdx.x, tid = threadIdx.x;
    const uint16_t* row = x + (size_t)m * K;
    int8_t* out = qx + (size_t)m * Kp;
    const bool vec = (K & 7) == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    float mx = 0.f;
    if (vec) {
        for (int k = tid * 8; k < K; k += kActThreads * 8) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + k));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[j] << 16)),
                                     fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
        }
    } else {
        for (int k = tid; k < K; k += kActThreads) mx = fmaxf(mx, fabsf(bf16_bits_to_f32(__ldg(row + k))));
    }
    mx = warp_max(mx);
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    if (tid < 32) {
        float v = red[tid];
        v = warp_max(v);
        if (tid == 0) red[0] = v;
    }
    __syncthreads();
    const float s = __fdiv_rn(red[0], 127.0f);
    if (tid == 0) sx[m] = s;
    auto q8 = [&](float v) -> uint32_t {
        if (s == 0.f) return 0u;
        return (uint32_t)(uint8_t)(int8_t)(int)fminf(fmaxf(rintf(__fdiv_rn(v, s)), -127.f), 127.f);
    };
    if (vec) {
        // 8 columns per step; columns K..Kp-1 (a multiple of 8 past K) are zero
        for (int k = tid * 8; k < Kp; k += kActThreads * 8) {
            uint2 o = make_uint2(0u, 0u);
            if (k < K) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + k));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t b[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    b[2 * j] = q8(__uint_as_float(w[j] << 16));
                    b[2 * j + 1] = q8(__uint_as_float(w[j] & 0xFFFF0000u));
                }
                o.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
                o.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
            }
            *reinterpret_cast<uint2*>(out + k) = o;
        }
    } else {
        for (int k = tid; k < Kp; k += kActThreads) {
            int q = 0;
            if (k < K) q = (int)(int8_t)(uint8_t)q8(bf16_bits_to_f32(__ldg(row + k)));
            out[k] = (int8_t)q;
        }
    }
}

}  // namespace

__global__ void k_stream_fence() {}

int launch_pack_rtn(const float* W, int N, int K, int G, int symmetric, uint8_t* packed,
                    float* scales, uint8_t* zeros, cudaStream_t stream) {
    const int Ng = (K + G - 1) / G;
    const long long warps = (long long)N * Ng;
    const long long blocks = (warps * 32 + 255) / 256;
    if (blocks > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    k_pack_rtn<<<(unsigned)blocks, 256, 0, stream>>>(W, N, K, G, Ng, symmetric, packed,
                                                     scales, zeros);
    // An ordinary launch starts only after k_pack_rtn has finished and its
    // stores are visible; a linear-layer kernel enqueued next may overlap
    // this empty kernel (programmatic dependent launch) and read the new
    // weights before its dependency wait.
    k_stream_fence<<<1, 32, 0, stream>>>();
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

int launch_act_quant(const uint16_t* x, int M, int K, int Kp, int8_t* qx, float* sx,
                     cudaStream_t stream) {
    k_act_quant<<<M, kActThreads, 0, stream>>>(x, K, Kp, qx, sx);
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

}  // namespace w4
