// gptq.cu - GPTQ quantizer on the GPU ("Lab 5: Gemma4 端到端推理优化",
// section "从 RTN 到 GPTQ"), in FP32 as the page's implementation:
//   H = (2/T) X^T X; dead columns (H_jj = 0): W[:, j] = 0, H_jj = 1;
//   H += lambda I, lambda = damp * mean(diag H); H^-1 = U^T U (U upper);
//   column by column: q_i from w_i by the RTN rule of its group (parameters
//   fixed at the group's first column from its current weights),
//   e_i = (w_i - q_i) / U_ii, W[:, i:] -= e_i U[i, i:],
//   L_pred = 1/2 sum (w_i - q_i)^2 / U_ii^2 per row.
//
// GPU formulation:
//  * U without an explicit inverse: H^-1 = U^T U  <=>  H = R R^T with
//    R = U^-1 upper triangular.  With P the index reversal, P H P = (P R P)
//    (P R P)^T is an ordinary lower Cholesky factorisation, so
//    U = P inv(chol(P H P)) P: one blocked Cholesky and one blocked
//    triangular inverse (32-wide blocks).
//  * The column loop runs in blocks of B <= 128 columns: one warp per row
//    applies the updates inside the block as it goes; at the end of the
//    block the rest of the row receives them at once,
//    W[:, i1:] -= E[:, block] U[block, i1:] (the same update, summed).
// The packed codes, scales and zero points have the layout of w4_pack_rtn.
#include "w4_device.cuh"
#include "w4_internal.h"

#include <algorithm>

namespace w4 {
namespace {

constexpr int TBK = 32;             // Cholesky / triangular-inverse block

__device__ __forceinline__ float wmax(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float wmin(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// The RTN rule of w4_pack_rtn for a group with max|r| (sym) or the range
// [mn, mx] holding 0 (asym): scale s, zero point z (8 when symmetric).
__device__ __forceinline__ void group_params(bool sym, float mx, float mn, float& s, float& z) {
    if (sym) {
        s = __fdiv_rn(mx, 7.0f);
        z = 8.f;
    } else {
        s = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
        z = s != 0.f ? fminf(fmaxf(rintf(__fdiv_rn(-mn, s)), 0.f), 15.f) : 0.f;
    }
}
__device__ __forceinline__ int code_of(bool sym, float r, float s, float z) {
    if (s == 0.f) return sym ? 8 : 0;
    if (sym) return (int)fminf(fmaxf(rintf(__fdiv_rn(r, s)), -8.f), 7.f) + 8;
    return (int)fminf(fmaxf(rintf(__fadd_rn(__fdiv_rn(r, s), z)), 0.f), 15.f);
}

// H = scale * X^T X over columns < K (zero beyond), [Kp, Kp]; a 64 x 64
// tile per CTA of 256 threads (4 x 4 each), tokens in chunks of 16.
__global__ void __launch_bounds__(256)
k_hessian(const uint16_t* __restrict__ X, int T, int K, int Kp, float scale, float* __restrict__ H) {
    __shared__ float xa[16][64], xb[16][64];
    const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    float acc[4][4] = {};
    for (int t0 = 0; t0 < T; t0 += 16) {
        for (int e = tid; e < 16 * 64; e += 256) {
            const int tt = e >> 6, c = e & 63, t = t0 + tt;
            xa[tt][c] = (t < T && i0 + c < K) ? bf16_bits_to_f32(X[(size_t)t * K + i0 + c]) : 0.f;
            xb[tt][c] = (t < T && j0 + c < K) ? bf16_bits_to_f32(X[(size_t)t * K + j0 + c]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int tt = 0; tt < 16; ++tt) {
            float a[4], b[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                a[r] = xa[tt][ty * 4 + r];
                b[r] = xb[tt][tx * 4 + r];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int i = i0 + ty * 4 + r, j = j0 + tx * 4 + c;
            if (i < Kp && j < Kp) H[(size_t)i * Kp + j] = acc[r][c] * scale;
        }
}

// Dead columns and damping, one CTA: H_jj = 0 -> 1 (flagged), then every
// H_jj += damp * mean(diag H).
__global__ void __launch_bounds__(1024)
k_dead_damp(float* __restrict__ H, int Kp, float damp, uint8_t* __restrict__ dead) {
    __shared__ float part[32];
    const int tid = threadIdx.x;
    float sum = 0.f;
    for (int j = tid; j < Kp; j += 1024) {
        float d = H[(size_t)j * Kp + j];
        const bool z = d == 0.f;
        if (z) {
            d = 1.f;
            H[(size_t)j * Kp + j] = 1.f;
        }
        dead[j] = z ? 1 : 0;
        sum += d;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if ((tid & 31) == 0) part[tid >> 5] = sum;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < 32; ++w) tot += part[w];
    const float lam = damp * (tot / (float)Kp);
    for (int j = tid; j < Kp; j += 1024) H[(size_t)j * Kp + j] += lam;
}

// Working copy of the weights, [N, Kp]: zero in dead and padded columns.
__global__ void k_copy_w(const float* __restrict__ W, int N, int K, int Kp,
                         const uint8_t* __restrict__ dead, float* __restrict__ Wc) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)N * Kp) return;
    const int j = (int)(i % (size_t)Kp);
    const size_t n = i / (size_t)Kp;
    Wc[i] = (j < K && !dead[j]) ? W[n * K + j] : 0.f;
}

// dst[a][b] = src[Kp-1-a][Kp-1-b]
__global__ void k_reverse(const float* __restrict__ src, float* __restrict__ dst, int Kp) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t n = (size_t)Kp * Kp;
    if (i >= n) return;
    dst[i] = src[n - 1 - i];
}

// Cholesky, diagonal block kb of A (lower, in place), unblocked in shared
// memory.  A non-positive pivot raises W4_ERR_NOT_SPD and is replaced by 1.
__global__ void k_chol_diag(float* __restrict__ A, int Kp, int kb, int* err) {
    __shared__ float D[TBK][TBK + 1];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const size_t o = (size_t)kb * TBK;
    D[ty][tx] = A[(o + ty) * Kp + o + tx];
    __syncthreads();
    for (int j = 0; j < TBK; ++j) {
        if (ty == j && tx == j) {
            float d = D[j][j];
            if (!(d > 0.f)) {
                atomicCAS(err, 0, W4_ERR_NOT_SPD);
                d = 1.f;
            }
            D[j][j] = sqrtf(d);
        }
        __syncthreads();
        if (tx == j && ty > j) D[ty][j] = D[ty][j] / D[j][j];
        __syncthreads();
        if (ty > j && tx > j && tx <= ty) D[ty][tx] -= D[ty][j] * D[tx][j];
        __syncthreads();
    }
    A[(o + ty) * Kp + o + tx] = tx <= ty ? D[ty][tx] : 0.f;
}

// Cholesky panel: rows r below block kb solve x L_kk^T = A[r, block]; one
// warp per row, 8 rows per CTA.
__global__ void __launch_bounds__(256)
k_chol_panel(float* __restrict__ A, int Kp, int kb) {
    __shared__ float Lk[TBK][TBK + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t o = (size_t)kb * TBK;
    for (int e = tid; e < TBK * TBK; e += 256) Lk[e >> 5][e & 31] = A[(o + (e >> 5)) * Kp + o + (e & 31)];
    __syncthreads();
    const size_t r = o + TBK + (size_t)blockIdx.x * 8 + warp;
    if (r >= (size_t)Kp) return;
    const float a = A[r * Kp + o + lane];
    float x = 0.f, acc = 0.f;
    for (int j = 0; j < TBK; ++j) {
        if (lane == j) x = (a - acc) / Lk[j][j];
        const float xj = __shfl_sync(0xffffffffu, x, j);
        if (lane > j) acc = fmaf(xj, Lk[lane][j], acc);
    }
    A[r * Kp + o + lane] = x;
}

// Cholesky trailing update below and right of block kb (lower triangle
// only): A[r][c] -= sum_l A[r][kb l] A[c][kb l], 64 x 64 tiles.
__global__ void __launch_bounds__(256)
k_chol_update(float* __restrict__ A, int Kp, int kb) {
    if (blockIdx.x > blockIdx.y) return;                 // tiles above the diagonal
    __shared__ float Pr[64][TBK + 1], Pc[64][TBK + 1];
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const size_t o = (size_t)kb * TBK, s0 = o + TBK;
    const size_t r0 = s0 + (size_t)blockIdx.y * 64, c0 = s0 + (size_t)blockIdx.x * 64;
    for (int e = tid; e < 64 * TBK; e += 256) {
        const int rr = e >> 5, l = e & 31;
        Pr[rr][l] = r0 + rr < (size_t)Kp ? A[(r0 + rr) * Kp + o + l] : 0.f;
        Pc[rr][l] = c0 + rr < (size_t)Kp ? A[(c0 + rr) * Kp + o + l] : 0.f;
    }
    __syncthreads();
    float acc[4][4] = {};
#pragma unroll 8
    for (int l = 0; l < TBK; ++l) {
        float a[4], b[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            a[q] = Pr[ty * 4 + q][l];
            b[q] = Pc[tx * 4 + q][l];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const size_t rr = r0 + ty * 4 + r, cc = c0 + tx * 4 + c;
            if (rr < (size_t)Kp && cc <= rr) A[rr * Kp + cc] -= acc[r][c];
        }
}

// Inverse of each 32 x 32 lower diagonal block of L into the same block of
// Li; thread c solves column c by forward substitution.
__global__ void k_trinv_diag(const float* __restrict__ L, float* __restrict__ Li, int Kp) {
    __shared__ float Ls[TBK][TBK + 1], Xs[TBK][TBK + 1];
    const int c = threadIdx.x;
    const size_t o = (size_t)blockIdx.x * TBK;
    for (int r = 0; r < TBK; ++r) Ls[r][c] = L[(o + r) * Kp + o + c];
    __syncthreads();
    for (int r = 0; r < TBK; ++r) {
        float v = 0.f;
        if (r == c) {
            v = 1.f / Ls[c][c];
        } else if (r > c) {
            float s = 0.f;
            for (int k = c; k < r; ++k) s = fmaf(Ls[r][k], Xs[k][c], s);
            v = -s / Ls[r][r];
        }
        Xs[r][c] = v;
    }
    for (int r = 0; r < TBK; ++r) Li[(o + r) * Kp + o + c] = Xs[r][c];
}

// Off-diagonal blocks of the inverse, block column j per CTA, down the rows:
// Li[i, j] = -Li[i, i] sum_{k = j .. i-1} L[i, k] Li[k, j].
__global__ void __launch_bounds__(256)
k_trinv_col(const float* __restrict__ L, float* __restrict__ Li, int Kp) {
    __shared__ float A[TBK][TBK + 1], B[TBK][TBK + 1], S[TBK][TBK + 1];
    const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;
    const int nb = Kp / TBK, j = blockIdx.x;
    const size_t oj = (size_t)j * TBK;
    for (int i = j + 1; i < nb; ++i) {
        const size_t oi = (size_t)i * TBK;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k = j; k < i; ++k) {
            const size_t ok = (size_t)k * TBK;
            for (int e = tid; e < TBK * TBK; e += 256) {
                A[e >> 5][e & 31] = L[(oi + (e >> 5)) * Kp + ok + (e & 31)];
                B[e >> 5][e & 31] = Li[(ok + (e >> 5)) * Kp + oj + (e & 31)];
            }
            __syncthreads();
#pragma unroll 8
            for (int l = 0; l < TBK; ++l) {
                const float a = A[ty][l];
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[c] = fmaf(a, B[l][tx * 4 + c], acc[c]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) S[ty][tx * 4 + c] = acc[c];
        for (int e = tid; e < TBK * TBK; e += 256) A[e >> 5][e & 31] = Li[(oi + (e >> 5)) * Kp + oi + (e & 31)];
        __syncthreads();
        float out[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int l = 0; l < TBK; ++l) {
            const float a = A[ty][l];
#pragma unroll
            for (int c = 0; c < 4; ++c) out[c] = fmaf(a, S[l][tx * 4 + c], out[c]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) Li[(oi + ty) * Kp + oj + tx * 4 + c] = -out[c];
        __syncthreads();      // Li[i, j] is read by this CTA's later rows; A is reloaded
    }
}

// One block of B = 32 NS columns [i0, i0 + B): one warp per row, 8 rows per
// CTA, U[block, block] in shared memory.  Per column: the group's
// parameters at its first column, the code, the normalised error e (kept
// in E for the update of the later columns), the updates of the block's
// later columns, and L_pred.
template <int NS>
__global__ void __launch_bounds__(256)
k_gptq_block(float* __restrict__ Wc, int N, int Kp, const float* __restrict__ U, int i0, int G,
             int sym_i, uint8_t* __restrict__ codes, float* __restrict__ scales,
             uint8_t* __restrict__ zeros, float* __restrict__ E, float* __restrict__ loss) {
    constexpr int B = 32 * NS;
    extern __shared__ float Us[];                         // [B][B]
    const bool sym = sym_i != 0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < B * B; e += 256) Us[e] = U[(size_t)(i0 + e / B) * Kp + i0 + e % B];
    __syncthreads();
    const int r = blockIdx.x * 8 + warp;
    if (r >= N) return;
    const int Ng = Kp / G;
    float* wrow = Wc + (size_t)r * Kp;
    float w[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) w[s] = wrow[i0 + s * 32 + lane];
    float sg = 0.f, zg = 8.f, lsum = 0.f;
    if (G > B) {
        // the group spans blocks: its parameters come from its first block
        const int g = i0 / G;
        if (i0 % G == 0) {
            float mx = 0.f, mn = 0.f;
            for (int k = i0 + lane; k < i0 + G; k += 32) {
                const float v = wrow[k];
                mx = fmaxf(mx, sym ? fabsf(v) : v);
                mn = fminf(mn, v);
            }
            group_params(sym, wmax(mx), wmin(mn), sg, zg);
            if (lane == 0) {
                scales[(size_t)r * Ng + g] = sg;
                if (!sym) zeros[(size_t)r * Ng + g] = (uint8_t)zg;
            }
        } else {
            sg = scales[(size_t)r * Ng + g];
            zg = sym ? 8.f : (float)zeros[(size_t)r * Ng + g];
        }
    }
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        for (int l = 0; l < 32; ++l) {
            const int ii = s * 32 + l, i = i0 + ii;
            if (G <= B && i % G == 0) {
                // parameters from the current weights of columns ii .. ii + G - 1
                float mx = 0.f, mn = 0.f;
#pragma unroll
                for (int q = 0; q < NS; ++q) {
                    const int col = q * 32 + lane;
                    if (col >= ii && col < ii + G) {
                        mx = fmaxf(mx, sym ? fabsf(w[q]) : w[q]);
                        mn = fminf(mn, w[q]);
                    }
                }
                group_params(sym, wmax(mx), wmin(mn), sg, zg);
                if (lane == 0) {
                    scales[(size_t)r * Ng + i / G] = sg;
                    if (!sym) zeros[(size_t)r * Ng + i / G] = (uint8_t)zg;
                }
            }
            const float wi = __shfl_sync(0xffffffffu, w[s], l);
            const int code = code_of(sym, wi, sg, zg);
            const float d = wi - sg * ((float)code - zg);
            const float uii = Us[ii * B + ii];
            const float e = d / uii;
            lsum += 0.5f * (d * d) / (uii * uii);
            if (lane == l) {
                codes[(size_t)r * Kp + i] = (uint8_t)code;
                E[(size_t)r * B + ii] = e;
            }
#pragma unroll
            for (int q = s; q < NS; ++q) {
                const int col = q * 32 + lane;
                if (col > ii) w[q] = fmaf(-e, Us[ii * B + col], w[q]);
            }
        }
    }
    if (lane == 0) loss[r] += lsum;
}

// The block's errors reach the later columns at once:
// Wc[:, i1:] -= E[:, 0:B] U[i0:i1, i1:], 64 x 64 tiles, B in steps of 32.
__global__ void __launch_bounds__(256)
k_gptq_lazy(float* __restrict__ Wc, int N, int Kp, const float* __restrict__ E, int B,
            const float* __restrict__ U, int i0, int i1) {
    __shared__ float Es[64][33], Ub[32][65];
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int n0 = blockIdx.y * 64, c0 = i1 + blockIdx.x * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < B; k0 += 32) {
        for (int e = tid; e < 64 * 32; e += 256) {
            const int rr = e >> 5, l = e & 31;
            Es[rr][l] = n0 + rr < N ? E[(size_t)(n0 + rr) * B + k0 + l] : 0.f;
            const int l2 = e >> 6, cc = e & 63;
            Ub[l2][cc] = c0 + cc < Kp ? U[(size_t)(i0 + k0 + l2) * Kp + c0 + cc] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int l = 0; l < 32; ++l) {
            float a[4], b[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a[q] = Es[ty * 4 + q][l];
                b[q] = Ub[l][tx * 4 + q];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int n = n0 + ty * 4 + r, cc = c0 + tx * 4 + c;
            if (n < N && cc < Kp) Wc[(size_t)n * Kp + cc] -= acc[r][c];
        }
}

// Two codes per byte, low nibble first.
__global__ void k_pack_codes(const uint8_t* __restrict__ codes, size_t nbytes,
                             uint8_t* __restrict__ packed) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nbytes) return;
    packed[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
}

unsigned blocks_for(size_t n, unsigned t) { return (unsigned)((n + t - 1) / t); }

}  // namespace

// Column block of the loop: 128 columns when the groups tile it (G = 32, 64,
// 128) or it tiles the groups (G a multiple of 128); else the group itself
// (G < 128) or the largest of 64, 32 that divides it.  Either way a group's
// first column is where its block starts or inside its block.
int gptq_block_cols(int G) {
    if (128 % G == 0 || G % 128 == 0) return 128;
    if (G < 128) return G;
    return G % 64 == 0 ? 64 : 32;
}

size_t gptq_workspace_bytes(int N, int Kp, int B) {
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    return 2 * up((size_t)Kp * Kp * 4) + up((size_t)N * Kp * 4) + up((size_t)N * B * 4) +
           up((size_t)N * Kp) + up((size_t)Kp);
}

int launch_gptq(const uint16_t* X, int T, const float* W, int N, int K, int Kp, int G,
                int symmetric, float damp, uint8_t* packed, float* scales, uint8_t* zeros,
                float* loss, void* ws, int* err, cudaStream_t st) {
    const int B = gptq_block_cols(G);
    auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
    uint8_t* base = static_cast<uint8_t*>(ws);
    float* H = reinterpret_cast<float*>(base);
    base += up((size_t)Kp * Kp * 4);
    float* A = reinterpret_cast<float*>(base);
    base += up((size_t)Kp * Kp * 4);
    float* Wc = reinterpret_cast<float*>(base);
    base += up((size_t)N * Kp * 4);
    float* E = reinterpret_cast<float*>(base);
    base += up((size_t)N * B * 4);
    uint8_t* codes = base;
    base += up((size_t)N * Kp);
    uint8_t* dead = base;

    const dim3 tiles((Kp + 63) / 64, (Kp + 63) / 64);
    k_hessian<<<tiles, 256, 0, st>>>(X, T, K, Kp, 2.f / (float)T, H);
    k_dead_damp<<<1, 1024, 0, st>>>(H, Kp, damp, dead);
    k_copy_w<<<blocks_for((size_t)N * Kp, 256), 256, 0, st>>>(W, N, K, Kp, dead, Wc);
    const size_t kk = (size_t)Kp * Kp;
    k_reverse<<<blocks_for(kk, 256), 256, 0, st>>>(H, A, Kp);           // A = P H P
    const int nb = Kp / TBK;
    for (int kb = 0; kb < nb; ++kb) {                                  // A = L L^T (lower)
        k_chol_diag<<<1, dim3(TBK, TBK), 0, st>>>(A, Kp, kb, err);
        const int below = Kp - (kb + 1) * TBK;
        if (below > 0) {
            k_chol_panel<<<(below + 7) / 8, 256, 0, st>>>(A, Kp, kb);
            const unsigned nt = (unsigned)((below + 63) / 64);
            k_chol_update<<<dim3(nt, nt), 256, 0, st>>>(A, Kp, kb);
        }
    }
    if (cudaMemsetAsync(H, 0, kk * 4, st) != cudaSuccess) return W4_ERR_CUDA;   // H = L^-1
    k_trinv_diag<<<nb, TBK, 0, st>>>(A, H, Kp);
    k_trinv_col<<<nb, 256, 0, st>>>(A, H, Kp);
    k_reverse<<<blocks_for(kk, 256), 256, 0, st>>>(H, A, Kp);           // A = U = P L^-1 P
    const float* U = A;

    if (cudaMemsetAsync(loss, 0, (size_t)N * 4, st) != cudaSuccess) return W4_ERR_CUDA;
    const size_t smem = (size_t)B * B * 4;
    auto run_block = [&](auto kern) -> int {
        if (smem > 48 * 1024 &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess)
            return W4_ERR_CUDA;
        for (int i0 = 0; i0 < Kp; i0 += B) {
            kern<<<(N + 7) / 8, 256, smem, st>>>(Wc, N, Kp, U, i0, G, symmetric, codes, scales,
                                                 zeros, E, loss);
            const int i1 = i0 + B;
            if (i1 < Kp)
                k_gptq_lazy<<<dim3((Kp - i1 + 63) / 64, (N + 63) / 64), 256, 0, st>>>(
                    Wc, N, Kp, E, B, U, i0, i1);
        }
        return W4_OK;
    };
    int rc;
    switch (B / 32) {
        case 1: rc = run_block(k_gptq_block<1>); break;
        case 2: rc = run_block(k_gptq_block<2>); break;
        case 3: rc = run_block(k_gptq_block<3>); break;
        default: rc = run_block(k_gptq_block<4>); break;
    }
    if (rc) return rc;
    const size_t nbytes = (size_t)N * Kp / 2;
    k_pack_codes<<<blocks_for(nbytes, 256), 256, 0, st>>>(codes, nbytes, packed);
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

}  // namespace w4
