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
#include <algorithm>
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
           uint8_t* __restrict__ zeros, uint16_t* __restrict__ scales_b,
           uint16_t* __restrict__ offs_b) {
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
        if (scales_b) {
            // bf16 parameters: bf16(s) and, asymmetric, bf16(fp32((8 - z) s))
            scales_b[(size_t)n * Ng + g] = f32_to_bf16_bits(s);
            if (!symmetric) offs_b[(size_t)n * Ng + g] = f32_to_bf16_bits(__fmul_rn(8.f - z, s));
        } else {
            scales[(size_t)n * Ng + g] = s;
            if (!symmetric) zeros[(size_t)n * Ng + g] = (uint8_t)z;
        }
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

// Eight columns k .. k+7 (four bf16x2 words) as fp32, smoothed when
// inv_s is given: x' = fp32(x * inv_s[k + j]) (the product rounded once).
// Columns >= K hold zero words and are not smoothed.
template <bool SMOOTH>
__device__ __forceinline__ void cols8(const uint4& v, const float* inv_s, int k, int K, float f[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = __uint_as_float(w[j] << 16);
        f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
    if (SMOOTH && k < K) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(inv_s + k));
        const float4 b = __ldg(reinterpret_cast<const float4*>(inv_s + k + 4));
        f[0] *= a.x; f[1] *= a.y; f[2] *= a.z; f[3] *= a.w;
        f[4] *= b.x; f[5] *= b.y; f[6] *= b.z; f[7] *= b.w;
    }
}

// Four columns k .. k+3 (two bf16x2 words, k < K) as fp32, smoothed as above.
template <bool SMOOTH>
__device__ __forceinline__ void cols4(const uint2& v, const float* inv_s, int k, float f[4]) {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xFFFF0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    if (SMOOTH) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(inv_s + k));
        f[0] *= a.x; f[1] *= a.y; f[2] *= a.z; f[3] *= a.w;
    }
}

// Grid (C, M): C CTAs of 512 threads per token.  Every CTA reduces max|x|
// over the whole row (so no CTA waits for another) and quantizes only its
// share, the 8-column words [c W, (c + 1) W) with W = ceil(Kp / 8 / C); CTA 0
// stores s_x.  RV > 0: the row has at most RV * 4096 columns and each thread
// keeps its RV 16-byte words in registers between the two steps (one read of
// x); RV = 0 (longer rows, C = 1): two passes, the second hitting L1/L2.
// SMOOTH: the activations are first divided by the SmoothQuant factors, as
// x * inv_s per column ("【infra之路】12-投机解码、量化与推理引擎对比",
// section 2.4), and the rule applies to x'.
// Launched with programmatic dependent launch: it waits for the kernel before
// it (which may have written x, or may still be reading qx and sx) before
// touching memory, and at once lets the next kernel start its prologue (a
// linear layer prefetches its weights meanwhile and waits for this kernel
// before reading qx).
constexpr int kActThreads = 512;

template <int RV, bool SMOOTH>
__global__ void __launch_bounds__(kActThreads)
k_act_quant(const uint16_t* __restrict__ x, const float* __restrict__ inv_s, int K, int Kp,
            int8_t* __restrict__ qx, float* __restrict__ sx) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float red[kActThreads / 32];
    const int m = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    const uint16_t* row = x + (size_t)m * K;
    int8_t* out = qx + (size_t)m * Kp;
    const bool vec = (K & 7) == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0;
    // otherwise 8-byte loads of four columns where K % 4 == 0 allows them
    const bool vec4 = !vec && (K & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 7) == 0;
    const int nw = Kp >> 3;                                   // 8-column words of the output row
    const int wpc = (nw + gridDim.x - 1) / gridDim.x;
    const int w0 = c * wpc, w1 = min(w0 + wpc, nw);           // this CTA's share
    constexpr int NR = RV > 0 ? RV : 1;
    auto col1 = [&](int k) -> float {                         // one column, k < K
        const float v = bf16_bits_to_f32(__ldg(row + k));
        return SMOOTH ? v * __ldg(inv_s + k) : v;
    };
    uint4 keep[NR];
    float mx = 0.f;
    auto max8 = [&](const uint4& v, int k) {
        float f[8];
        cols8<SMOOTH>(v, inv_s, k, K, f);
#pragma unroll
        for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(f[j]));
    };
    if (vec && RV > 0) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int k = (r * kActThreads + tid) * 8;
            keep[r] = k < K ? __ldg(reinterpret_cast<const uint4*>(row + k)) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) max8(keep[r], (r * kActThreads + tid) * 8);
    } else if (vec) {
        for (int k = tid * 8; k < K; k += kActThreads * 8)
            max8(__ldg(reinterpret_cast<const uint4*>(row + k)), k);
    } else if (vec4) {
#pragma unroll 4
        for (int k = tid * 4; k < K; k += kActThreads * 4) {
            float f[4];
            cols4<SMOOTH>(__ldg(reinterpret_cast<const uint2*>(row + k)), inv_s, k, f);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3]))));
        }
    } else {
#pragma unroll 4
        for (int k = tid; k < K; k += kActThreads) mx = fmaxf(mx, fabsf(col1(k)));
    }
    mx = warp_max(mx);
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    if (tid < 32) {
        float v = tid < kActThreads / 32 ? red[tid] : 0.f;
        v = warp_max(v);
        if (tid == 0) red[0] = v;
    }
    __syncthreads();
    const float s = __fdiv_rn(red[0], 127.0f);
    const float rs = s != 0.f ? __frcp_rn(s) : 0.f;
    if (tid == 0 && c == 0) sx[m] = s;
    if (vec) {
        // word w covers columns 8w .. 8w+7; words at or past K are zero
        int w = tid;
        if (RV > 0) {
#pragma unroll
            for (int r = 0; r < NR; ++r, w += kActThreads)
                if (w >= w0 && w < w1) {
                    float f[8];
                    cols8<SMOOTH>(keep[r], inv_s, 8 * w, K, f);
                    *reinterpret_cast<uint2*>(out + 8 * w) = quant_s8x8(f, s, rs);
                }
        }
        for (; w < w1; w += kActThreads) {
            if (w < w0) continue;
            uint2 o = make_uint2(0u, 0u);
            if (8 * w < K) {
                float f[8];
                cols8<SMOOTH>(__ldg(reinterpret_cast<const uint4*>(row + 8 * w)), inv_s, 8 * w, K, f);
                o = quant_s8x8(f, s, rs);
            }
            *reinterpret_cast<uint2*>(out + 8 * w) = o;
        }
    } else if (vec4) {
        // four columns per step; columns K..Kp-1 are zero
        for (int k = 8 * w0 + tid * 4; k < 8 * w1; k += kActThreads * 4) {
            uint32_t o = 0u;
            if (k < K && s != 0.f) {
                float f[4];
                cols4<SMOOTH>(__ldg(reinterpret_cast<const uint2*>(row + k)), inv_s, k, f);
                o = quant_s8(f[0], s, rs) | (quant_s8(f[1], s, rs) << 8) |
                    (quant_s8(f[2], s, rs) << 16) | (quant_s8(f[3], s, rs) << 24);
            }
            *reinterpret_cast<uint32_t*>(out + k) = o;
        }
    } else {
#pragma unroll 4
        for (int k = 8 * w0 + tid; k < 8 * w1; k += kActThreads) {
            uint32_t q = 0u;
            if (k < K && s != 0.f) q = quant_s8(col1(k), s, rs);
            out[k] = (int8_t)(uint8_t)q;
        }
    }
}

// SmoothQuant calibration, step 1: the largest |value| of every column over
// the rows, as fp32 bit patterns (non-negative floats order as integers) by
// atomicMax into `colmax` (zeroed by the caller).  BF16: the values are bf16
// bits, else fp32.  A block covers 256 columns x 64 rows.
template <bool BF16>
__global__ void k_col_absmax(const void* __restrict__ v, int rows, int cols, unsigned* colmax) {
    const int col = blockIdx.x * 256 + threadIdx.x;
    const int r0 = blockIdx.y * 64;
    if (col >= cols) return;
    unsigned mx = 0u;
    for (int r = r0; r < min(r0 + 64, rows); ++r) {
        const float f = BF16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(v)[(size_t)r * cols + col])
                             : static_cast<const float*>(v)[(size_t)r * cols + col];
        mx = max(mx, __float_as_uint(fabsf(f)));
    }
    atomicMax(colmax + col, mx);
}

// Step 2: s_j = max|X_j|^alpha / max|W_j|^(1 - alpha) (1 where either
// maximum is 0) and inv_s_j = fp32(1 / s_j), in place over the two maxima.
__global__ void k_smooth_factors(float* s_xmax, float* inv_wmax, int cols, float alpha) {
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= cols) return;
    const float xm = s_xmax[j], wm = inv_wmax[j];
    float sj = 1.f;
    if (xm > 0.f && wm > 0.f) sj = powf(xm, alpha) / powf(wm, 1.f - alpha);
    s_xmax[j] = sj;
    inv_wmax[j] = __fdiv_rn(1.f, sj);
}

// Step 3: W[n, j] *= s_j (the weights take the activations' outliers).
__global__ void k_scale_cols(float* W, const float* s, int rows, int cols) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)rows * cols) return;
    W[i] *= __ldg(s + (i % (size_t)cols));
}

}  // namespace

__global__ void k_stream_fence() {}

int launch_pack_rtn(const float* W, int N, int K, int G, int symmetric, uint8_t* packed,
                    float* scales, uint8_t* zeros, uint16_t* scales_b, uint16_t* offs_b,
                    cudaStream_t stream) {
    const int Ng = (K + G - 1) / G;
    const long long warps = (long long)N * Ng;
    const long long blocks = (warps * 32 + 255) / 256;
    if (blocks > 0x7fffffffLL) return W4_ERR_UNSUPPORTED_SHAPE;
    k_pack_rtn<<<(unsigned)blocks, 256, 0, stream>>>(W, N, K, G, Ng, symmetric, packed,
                                                     scales, zeros, scales_b, offs_b);
    // An ordinary launch starts only after k_pack_rtn has finished and its
    // stores are visible; a linear-layer kernel enqueued next may overlap
    // this empty kernel (programmatic dependent launch) and read the new
    // weights before its dependency wait.
    k_stream_fence<<<1, 32, 0, stream>>>();
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

int launch_act_quant(const uint16_t* x, const float* inv_s, int M, int K, int Kp, int8_t* qx,
                     float* sx, cudaStream_t stream) {
    // 16-byte words per thread to hold the row; each CTA quantizes up to
    // 4096 columns
    const int v = (K + kActThreads * 8 - 1) / (kActThreads * 8);
    const int C = v <= 8 ? std::min((Kp + 4095) / 4096, 16) : 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, M);
    cfg.blockDim = dim3(kActThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto go = [&](auto kern) { return cudaLaunchKernelEx(&cfg, kern, x, inv_s, K, Kp, qx, sx); };
    cudaError_t e;
    if (inv_s) {
        if (v <= 1) e = go(k_act_quant<1, true>);
        else if (v <= 2) e = go(k_act_quant<2, true>);
        else if (v <= 4) e = go(k_act_quant<4, true>);
        else if (v <= 8) e = go(k_act_quant<8, true>);
        else e = go(k_act_quant<0, true>);
    } else {
        if (v <= 1) e = go(k_act_quant<1, false>);
        else if (v <= 2) e = go(k_act_quant<2, false>);
        else if (v <= 4) e = go(k_act_quant<4, false>);
        else if (v <= 8) e = go(k_act_quant<8, false>);
        else e = go(k_act_quant<0, false>);
    }
    if (e != cudaSuccess) return W4_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

int launch_smooth(const uint16_t* X, int T, float* W, int N, int K, float alpha, float* s,
                  float* inv_s, cudaStream_t stream) {
    if (cudaMemsetAsync(s, 0, sizeof(float) * (size_t)K, stream) != cudaSuccess ||
        cudaMemsetAsync(inv_s, 0, sizeof(float) * (size_t)K, stream) != cudaSuccess)
        return W4_ERR_CUDA;
    const dim3 gx((K + 255) / 256, (T + 63) / 64), gw((K + 255) / 256, (N + 63) / 64);
    if (T > 0) k_col_absmax<true><<<gx, 256, 0, stream>>>(X, T, K, reinterpret_cast<unsigned*>(s));
    k_col_absmax<false><<<gw, 256, 0, stream>>>(W, N, K, reinterpret_cast<unsigned*>(inv_s));
    k_smooth_factors<<<(K + 255) / 256, 256, 0, stream>>>(s, inv_s, K, alpha);
    const size_t n = (size_t)N * K;
    k_scale_cols<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(W, s, N, K);
    // the next linear may start early under programmatic dependent launch
    // and read its weights before its dependency wait: end with an ordinary
    // launch, as w4_pack_rtn does
    k_stream_fence<<<1, 32, 0, stream>>>();
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

}  // namespace w4
