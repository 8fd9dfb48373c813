// gemm_tc.cu - prefill kernel (M > 16) for the INT4 weight-only linear layer
// on the 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA).
//
// "Lab 5: Gemma4 端到端推理优化", section "Prefill和Decode分流": for a large
// number of tokens the layer is a dense GEMM and dequantizing costs little
// next to it; the page dequantizes the whole layer to bf16 in HBM and calls
// cuBLAS.  Here the INT4 tiles are dequantized on chip instead, straight into
// the shared-memory operand of the tensor-core MMA, so bf16 weights never
// touch HBM.
//
// D[128 weight rows x 256 tokens] (fp32, TMEM) += W_hat[128 x 64] * x[256 x 64]^T
// per 64-column stage; W_hat = s (code - z) is rounded once to bf16.
//
// Warp roles (448 threads, one CTA per SM, persistent over output tiles):
//   warp 0     TMA: x tile (256 tokens x 64 columns, bf16, 128-byte swizzle)
//              and packed tile (128 rows x 32 bytes) into a 4-stage ring
//   warp 1     allocates 512 TMEM columns (two 256-column accumulators);
//              one thread issues tcgen05.mma (M=128, N=256, K=16) x 4 per stage
//   warps 2-9  dequantize (one weight row and 32 columns per thread) into
//              the 128-byte-swizzled K-major bf16 A operand (3-stage ring)
//   warps 10-13 epilogue: tcgen05.ld of the accumulator, + bias, bf16 stores
// Every mbarrier wait is bounded; a failed wait raises the CTA abort flag and
// the device error flag, in-flight copies and MMAs are drained before exit.
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {
namespace {

constexpr int BM = 128;                 // weight rows per tile (MMA M)
constexpr int BN = 256;                 // tokens per tile (MMA N)
constexpr int BK = 64;                  // columns per stage
constexpr int NST = 4;                  // TMA stages
constexpr int NSA = 3;                  // dequantized A stages
constexpr int X_BYTES = BN * BK * 2;    // 32 KB
constexpr int P_BYTES = BM * BK / 2;    // 4 KB
constexpr int A_BYTES = BM * BK * 2;    // 16 KB
constexpr int THREADS = 448;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

struct GemmArgs {
    const float* scales;
    const uint8_t* zeros;
    const float* bias;
    uint16_t* y;
    int* err;
    int M, N, K, G, Ng;
    int nks;        // k stages
    int TB;         // token blocks
    int ntiles;
};

struct Ctl {
    uint64_t tfull[NST], tempty[NST];
    uint64_t afull[NSA], aempty[NSA];
    uint64_t accfull[2], accempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = 1024 + (size_t)NST * X_BYTES + (size_t)NSA * A_BYTES +
                              (size_t)NST * P_BYTES + 256;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t s = smem_u32(p);
    return p + (((s + 1023u) & ~1023u) - s);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(THREADS, 1)
k_w4a16_gemm_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmP,
                const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = align1024(smem_raw);
    uint8_t* xs = base;                                     // NST x 32 KB
    uint8_t* as = xs + NST * X_BYTES;                       // NSA x 16 KB
    uint8_t* ps = as + NSA * A_BYTES;                       // NST x 4 KB
    Ctl* ctl = reinterpret_cast<Ctl*>(ps + NST * P_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) { mbar_init(&ctl->tfull[i], 1); mbar_init(&ctl->tempty[i], 1); }
        for (int i = 0; i < NSA; ++i) { mbar_init(&ctl->afull[i], 256); mbar_init(&ctl->aempty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&ctl->accfull[i], 1); mbar_init(&ctl->accempty[i], 128); }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) { tma_prefetch_desc(&tmX); tma_prefetch_desc(&tmP); }
    if (warp == 1) { tmem_alloc(&ctl->tmem_base, TMEM_COLS); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            const uint64_t pol_x = policy_evict_last();
            const uint64_t pol_w = policy_evict_last();
            uint32_t it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.ntiles && ok; u += gridDim.x) {
                const int nb = u / a.TB, tb = u - nb * a.TB;
                for (int ks = 0; ks < a.nks; ++ks, ++it) {
                    const int s = it % NST;
                    if (it >= (uint32_t)NST &&
                        !mbar_wait(&ctl->tempty[s], ((it / NST) & 1) ^ 1, &ctl->abort, a.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ctl->tfull[s], X_BYTES + P_BYTES);
                    tma_load_2d(xs + s * X_BYTES, &tmX, ks * BK, tb * BN, &ctl->tfull[s], pol_x);
                    tma_load_2d(ps + s * P_BYTES, &tmP, ks * (BK / 2), nb * BM, &ctl->tfull[s], pol_w);
                }
            }
            if (!ok || ctl->abort) {
                const uint32_t first = it > (uint32_t)NST ? it - NST : 0;
                for (uint32_t j = first; j < it; ++j)
                    mbar_wait_drain(&ctl->tfull[j % NST], (j / NST) & 1, a.err);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            uint32_t it = 0, ia = 0, tc = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < a.ntiles && ok; u += gridDim.x, ++tc) {
                const uint32_t b = tc & 1;
                if (tc >= 2 && !mbar_wait(&ctl->accempty[b], ((tc / 2) & 1) ^ 1, &ctl->abort, a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + b * BN;
                for (int ks = 0; ks < a.nks; ++ks, ++it, ++ia) {
                    const int s = it % NST, sa = ia % NSA;
                    if (!mbar_wait(&ctl->tfull[s], (it / NST) & 1, &ctl->abort, a.err) ||
                        !mbar_wait(&ctl->afull[sa], (ia / NSA) & 1, &ctl->abort, a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(as + sa * A_BYTES);
                    const uint32_t x_addr = smem_u32(xs + s * X_BYTES);
#pragma unroll
                    for (int i = 0; i < BK / 16; ++i)
                        tc_mma_f16(d, smem_desc_sw128(a_addr + 32 * i),
                                   smem_desc_sw128(x_addr + 32 * i), IDESC,
                                   (ks | i) != 0 ? 1u : 0u);
                    tc_commit(&ctl->tempty[s]);
                    tc_commit(&ctl->aempty[sa]);
                }
                if (!ok) break;
                tc_commit(&ctl->accfull[b]);
            }
            // every MMA issued by this thread completes before the CTA ends
            tc_commit(&ctl->drain);
            mbar_wait_drain(&ctl->drain, 0, a.err);
        }
    } else if (warp < 10) {
        // ------------------------------------------------------------ dequantize
        // 256 threads: weight row r of the tile, columns [32 h, 32 h + 32) of
        // each 64-column stage
        const int dw = warp - 2;
        const int r = (dw & 3) * 32 + lane, h = dw >> 2;
        uint32_t it = 0, ia = 0;
        for (int u = blockIdx.x; u < a.ntiles; u += gridDim.x) {
            const int nb = u / a.TB;
            const int n = min(nb * BM + r, a.N - 1);
            const float* srow = a.scales + (size_t)n * a.Ng;
            const uint8_t* zrow = a.zeros ? a.zeros + (size_t)n * a.Ng : nullptr;
            // scale (and offset -(128 + z) s) of this thread's 32 columns,
            // loaded one stage ahead
            auto group_of = [&](int ks) { return min((ks * BK + 32 * h) / a.G, a.Ng - 1); };
            float sc = __ldg(srow + group_of(0));
            float zz = zrow ? (float)__ldg(zrow + group_of(0)) : 8.f;
            for (int ks = 0; ks < a.nks; ++ks, ++it, ++ia) {
                const int s = it % NST, sa = ia % NSA;
                float nsc = sc, nzz = zz;
                if (ks + 1 < a.nks) {
                    const int g = group_of(ks + 1);
                    nsc = __ldg(srow + g);
                    nzz = zrow ? (float)__ldg(zrow + g) : 8.f;
                }
                const float cc = -(128.f + zz) * sc;
                bool ok = mbar_wait(&ctl->tfull[s], (it / NST) & 1, &ctl->abort, a.err);
                if (ok && ia >= (uint32_t)NSA)
                    ok = mbar_wait(&ctl->aempty[sa], ((ia / NSA) & 1) ^ 1, &ctl->abort, a.err);
                if (ok) {
                    const uint4 q = *reinterpret_cast<const uint4*>(ps + s * P_BYTES + r * 32 + h * 16);
                    const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
                    uint8_t* arow = as + sa * A_BYTES + r * 128;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int j = 4 * h + jj;               // 16-byte chunk of the row
                        const uint32_t w = wv[jj], wh = w >> 4;
                        // bf16x2 (128 + c_2i, 128 + c_2i+1) for i = 0..3
                        const uint32_t e = 0x43004300u, m = 0x000F000Fu;
                        const uint32_t p01 = and_or(prmt(w, wh, 0x5410), m, e);
                        const uint32_t p23 = and_or(prmt(w, wh, 0x6521), m, e);
                        const uint32_t p45 = and_or(prmt(w, wh, 0x7632), m, e);
                        const uint32_t p67 = and_or(prmt(w, wh, 0x0703), m, e);
                        uint4 o;
                        o.x = pack_bf16x2(fmaf(bf16lo(p01), sc, cc), fmaf(bf16hi(p01), sc, cc));
                        o.y = pack_bf16x2(fmaf(bf16lo(p23), sc, cc), fmaf(bf16hi(p23), sc, cc));
                        o.z = pack_bf16x2(fmaf(bf16lo(p45), sc, cc), fmaf(bf16hi(p45), sc, cc));
                        o.w = pack_bf16x2(fmaf(bf16lo(p67), sc, cc), fmaf(bf16hi(p67), sc, cc));
                        *reinterpret_cast<uint4*>(arow + ((j ^ (r & 7)) << 4)) = o;
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&ctl->afull[sa]);
                }
                sc = nsc;
                zz = nzz;
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                            // TMEM lane quarter of this warp
        const int r = q * 32 + lane;
        uint32_t tc = 0;
        for (int u = blockIdx.x; u < a.ntiles; u += gridDim.x, ++tc) {
            const int nb = u / a.TB, tb = u - nb * a.TB;
            const uint32_t b = tc & 1;
            const bool ok = mbar_wait(&ctl->accfull[b], (tc / 2) & 1, &ctl->abort, a.err);
            tc_fence_after();
            const int n = nb * BM + r;
            const float bn = (a.bias && n < a.N) ? __ldg(a.bias + n) : 0.f;
            if (ok) {
                for (int j = 0; j < BN / 32; ++j) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + b * BN + j * 32, v);
                    tc_wait_ld();
                    if (n < a.N) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int t = tb * BN + j * 32 + i;
                            if (t < a.M)
                                a.y[(size_t)t * a.N + n] = f32_to_bf16_bits(__uint_as_float(v[i]) + bn);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&ctl->accempty[b]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace

int launch_w4a16_gemm(const uint16_t* x, const uint8_t* packed, const float* scales,
                      const uint8_t* zeros, const float* bias, uint16_t* y, int M, int N, int K,
                      int Kp, int G, int* err, int sm_count, cudaStream_t stream) {
    CUtensorMap tmX, tmP;
    if (!encode_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, (uint64_t)K, (uint64_t)M,
                        (uint64_t)K * 2, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return W4_ERR_CUDA;
    if (!encode_tmap_2d(&tmP, CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, (uint64_t)(Kp / 2),
                        (uint64_t)N, (uint64_t)(Kp / 2), BK / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
        return W4_ERR_CUDA;
    GemmArgs a{};
    a.scales = scales; a.zeros = zeros; a.bias = bias; a.y = y; a.err = err;
    a.M = M; a.N = N; a.K = K; a.G = G; a.Ng = Kp / G;
    a.nks = (K + BK - 1) / BK;
    a.TB = (M + BN - 1) / BN;
    a.ntiles = ((N + BM - 1) / BM) * a.TB;
    const int grid = a.ntiles < sm_count ? a.ntiles : sm_count;
    if (cudaFuncSetAttribute(k_w4a16_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
        return W4_ERR_CUDA;
    k_w4a16_gemm_tc<<<grid, THREADS, kSmemBytes, stream>>>(tmX, tmP, a);
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

}  // namespace w4
