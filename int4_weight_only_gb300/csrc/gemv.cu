// gemv.cu - decode kernels (M <= 16) for the INT4 weight-only linear layer.
//
// W4A16 ("Lab 5: Gemma4 端到端推理优化", sections "INT4 线性量化" and
// "融合INT4反量化与矩阵乘"): y = x W_hat^T (+b) with W_hat = s (code - z),
// dequantized in registers next to the multiply, one pass over the packed
// weights.  W4A8 ("Jetson Orin AGX INT4 推理优化实践", sections
// "从 FP 线性层到 INT4 DP4A 的数学推导" and "DP4A 做了什么"):
// acc = sum (code - 8) q_x in int32, y = s_W s_x acc + b.
//
// Structure (both kernels): one CTA per SM, 8 consumer warps + 1 producer
// warp.  The producer streams 128-row x 256-column tiles of the packed
// weights (16 KB, 128-byte swizzled) into a 6-deep shared-memory ring with
// TMA; each consumer warp owns 16 rows of the tile and reads its fragments
// with ldmatrix.  A unit of work is (128-row block, K slice); units are dealt
// round-robin to the persistent CTAs, and K slices (split-K) are combined by
// the last CTA to finish a row block, in a fixed order.
//
// W4A16 inner product: each 32-bit ldmatrix word holds 8 codes of one row;
// they become four bf16x2 words (c - z exact) that feed mma.sync m16n8k16
// directly as the A operand (16 weight rows), with the activations as the B
// operand (8 tokens per n-tile).  The order of k inside a 32-column chunk is
// permuted identically on both operands, so no data shuffles are needed.  All
// 16 columns of one MMA come from one 32-column chunk and hence one group:
// the group scale is applied to the fp32 partial sums, not to the weights.
#include "w4_device.cuh"
#include "w4_internal.h"

#include <algorithm>

namespace w4 {
namespace {

constexpr int CW = kGemvConsumerWarps;
constexpr int NCT = CW * 32;
constexpr int NS = kGemvStages;
constexpr int ROWS = kGemvRows;
constexpr int STAGE_K = kGemvStageK;
constexpr int STAGE_BYTES = ROWS * (STAGE_K / 2);      // 16 KB

struct SmemCtl {
    uint64_t full[NS];
    uint64_t empty[NS];
    int abort;
    int last;
    int sumq[16];
};
constexpr int kCtlBytes = (int)((sizeof(SmemCtl) + 127) / 128 * 128);

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t s = smem_u32(p);
    return p + (((s + 1023u) & ~1023u) - s);
}

__device__ __forceinline__ void unit_coords(int u, const GemvArgs& a, int& rb, int& s,
                                            int& ks0, int& ks1) {
    rb = u / a.S;
    s = u - rb * a.S;
    ks0 = s * a.spl;
    ks1 = min(ks0 + a.spl, a.nst);
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t* v) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "r"(addr));
}

__device__ __forceinline__ void lds64(uint32_t addr, uint32_t& a, uint32_t& b) {
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
}

// Producer: one thread streams every stage of every unit of this CTA.
__device__ void gemv_producer(const CUtensorMap* tm, uint8_t* wbuf, SmemCtl* ctl,
                              const GemvArgs& a) {
    const uint64_t pol = policy_evict_first();
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < a.units && ok; u += gridDim.x) {
        int rb, s, ks0, ks1;
        unit_coords(u, a, rb, s, ks0, ks1);
        for (int ks = ks0; ks < ks1; ++ks, ++it) {
            const int slot = it % NS;
            if (it >= (uint32_t)NS &&
                !mbar_wait(&ctl->empty[slot], ((it / NS) & 1) ^ 1, &ctl->abort, a.err)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&ctl->full[slot], STAGE_BYTES);
            tma_load_2d(wbuf + slot * STAGE_BYTES, tm, ks * (STAGE_K / 2), rb * ROWS,
                        &ctl->full[slot], pol);
        }
    }
    if (!ok || ctl->abort) {
        // A wait gave up: let the copies already issued land before exiting.
        const uint32_t first = it > (uint32_t)NS ? it - NS : 0;
        for (uint32_t j = first; j < it; ++j)
            mbar_wait_drain(&ctl->full[j % NS], (j / NS) & 1, a.err);
    }
}

// Activations of one unit into shared memory, bf16, columns [k0, k0+nk).
// Within every 8-column block the order is (0,4,1,5,2,6,3,7), the order in
// which nibbles_to_bf16x2 emits weights; columns >= K are zero.
__device__ void stage_x_bf16(uint8_t* xbuf, const uint16_t* x, int M, int K, int XS,
                             int k0, int nk, int tid) {
    const int nb = nk >> 3;
    const bool vec = (K & 7) == 0;
    for (int idx = tid; idx < M * nb; idx += NCT) {
        const int m = idx / nb, b = idx - m * nb;
        const int k = k0 + b * 8;
        uint32_t q[4];
        const uint16_t* src = x + (size_t)m * K + k;
        if (vec && k + 8 <= K) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
            q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
        } else {
            uint16_t e[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) e[j] = (k + j < K) ? __ldg(src + j) : (uint16_t)0;
#pragma unroll
            for (int j = 0; j < 4; ++j) q[j] = (uint32_t)e[2 * j] | ((uint32_t)e[2 * j + 1] << 16);
        }
        uint4 o;
        o.x = __byte_perm(q[0], q[2], 0x5410);   // (x0, x4)
        o.y = __byte_perm(q[0], q[2], 0x7632);   // (x1, x5)
        o.z = __byte_perm(q[1], q[3], 0x5410);   // (x2, x6)
        o.w = __byte_perm(q[1], q[3], 0x7632);   // (x3, x7)
        *reinterpret_cast<uint4*>(xbuf + (size_t)m * XS + b * 16) = o;
    }
}

// INT8 activations of one unit, order (0,2,4,6 | 1,3,5,7) per 8-column
// block to match the byte lanes of (v & 0x0F0F0F0F) and ((v >> 4) & ...);
// also accumulates sum(q_x) per token into ctl->sumq.
__device__ void stage_x_s8(uint8_t* xbuf, SmemCtl* ctl, const int8_t* qx, int M, int Kp,
                           int XS, int k0, int nk, int tid) {
    const int nb = nk >> 3;
    for (int m = 0; m < M; ++m) {
        int part = 0;
        for (int b = tid; b < nb; b += NCT) {
            const int k = k0 + b * 8;
            uint32_t w0 = 0, w1 = 0;
            if (k < Kp) {
                const uint2 v = __ldg(reinterpret_cast<const uint2*>(qx + (size_t)m * Kp + k));
                w0 = v.x; w1 = v.y;
            }
            part = __dp4a((int)w0, 0x01010101, part);
            part = __dp4a((int)w1, 0x01010101, part);
            uint2 o;
            o.x = __byte_perm(w0, w1, 0x6420);
            o.y = __byte_perm(w0, w1, 0x7531);
            *reinterpret_cast<uint2*>(xbuf + (size_t)m * XS + b * 8) = o;
        }
        part = __reduce_add_sync(0xffffffffu, part);
        if ((tid & 31) == 0) atomicAdd(&ctl->sumq[m], part);
    }
}

template <int NT, int CPG, bool ASYM>
__device__ void w4a16_consumer(uint8_t* wbuf, uint8_t* xbuf, SmemCtl* ctl, const GemvArgs& a) {
    constexpr int SEG = 8 / CPG;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tig = lane & 3, gid = lane >> 2;
    const uint16_t* x = static_cast<const uint16_t*>(a.x);
    const uint32_t wbuf_u = smem_u32(wbuf), xbuf_u = smem_u32(xbuf);
    const int lj = lane >> 3, li = lane & 7;
    const uint32_t l_rowoff = (uint32_t)(warp * 16 + ((lj & 1) << 3) + li) * 128u;
    const int l_chi = lj >> 1;
    uint32_t xrow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
        xrow[nt] = xbuf_u + (uint32_t)(min(nt * 8 + gid, a.M - 1) * a.XS + tig * 16);

    uint32_t it = 0;
    for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
        int rb, s, ks0, ks1;
        unit_coords(u, a, rb, s, ks0, ks1);
        const int row0 = rb * ROWS + warp * 16;
        const int nr = min(row0 + gid, a.N - 1), nr8 = min(row0 + gid + 8, a.N - 1);
        const float* sc_r = a.scales + (size_t)nr * a.Ng;
        const float* sc_r8 = a.scales + (size_t)nr8 * a.Ng;

        named_bar_sync(1, NCT);
        stage_x_bf16(xbuf, x, a.M, a.K, a.XS, ks0 * STAGE_K, (ks1 - ks0) * STAGE_K, tid);
        named_bar_sync(1, NCT);

        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[nt][j] = 0.f;

        for (int ks = ks0; ks < ks1; ++ks, ++it) {
            const int slot = it % NS;
            float sr[SEG], sr8[SEG];
            uint32_t zr[SEG], zr8[SEG];
#pragma unroll
            for (int j = 0; j < SEG; ++j) {
                const int g = min((ks * STAGE_K + j * CPG * 32) / a.G, a.Ng - 1);
                sr[j] = __ldg(sc_r + g);
                sr8[j] = __ldg(sc_r8 + g);
                if (ASYM) {
                    zr[j] = (0x4300u + __ldg(a.zeros + (size_t)nr * a.Ng + g)) * 0x10001u;
                    zr8[j] = (0x4300u + __ldg(a.zeros + (size_t)nr8 * a.Ng + g)) * 0x10001u;
                } else {
                    zr[j] = zr8[j] = 0x43084308u;          // 128 + 8
                }
            }
            if (mbar_wait(&ctl->full[slot], (it / NS) & 1, &ctl->abort, a.err)) {
                const uint32_t wst = wbuf_u + slot * STAGE_BYTES + l_rowoff;
                const uint32_t xoff = (uint32_t)(ks - ks0) * (STAGE_K * 2);
                float tmp[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 4; ++j) tmp[nt][j] = 0.f;
#pragma unroll
                for (int cp = 0; cp < 4; ++cp) {
                    uint32_t r[4];
                    ldmatrix_x4(wst + ((uint32_t)((2 * cp + l_chi) ^ li) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = 2 * cp + h;
                        const int seg = c / CPG;
                        uint32_t P[4], Q[4];
                        nibbles_to_bf16x2(r[2 * h], zr[seg], P);
                        nibbles_to_bf16x2(r[2 * h + 1], zr8[seg], Q);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            uint32_t X[4];
                            lds128(xrow[nt] + xoff + c * 64, X);
                            mma_bf16_16816(tmp[nt], P[0], Q[0], P[1], Q[1], X[0], X[1], tmp[nt]);
                            mma_bf16_16816(tmp[nt], P[2], Q[2], P[3], Q[3], X[2], X[3], tmp[nt]);
                        }
                        if ((c + 1) % CPG == 0) {
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                acc[nt][0] = fmaf(sr[seg], tmp[nt][0], acc[nt][0]);
                                acc[nt][1] = fmaf(sr[seg], tmp[nt][1], acc[nt][1]);
                                acc[nt][2] = fmaf(sr8[seg], tmp[nt][2], acc[nt][2]);
                                acc[nt][3] = fmaf(sr8[seg], tmp[nt][3], acc[nt][3]);
#pragma unroll
                                for (int j = 0; j < 4; ++j) tmp[nt][j] = 0.f;
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->empty[slot]);
        }

        // ---- epilogue: thread holds (token 8nt + 2tig + (j&1), row gid + 8(j>>1))
        if (a.S == 1) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = nt * 8 + 2 * tig + (j & 1);
                    const int n = row0 + gid + 8 * (j >> 1);
                    if (t < a.M && n < a.N) {
                        const float b = a.bias ? __ldg(a.bias + n) : 0.f;
                        a.y[(size_t)t * a.N + n] = f32_to_bf16_bits(acc[nt][j] + b);
                    }
                }
        } else {
            float* part = static_cast<float*>(a.partial);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = nt * 8 + 2 * tig + (j & 1);
                    const int n = row0 + gid + 8 * (j >> 1);
                    if (t < a.M && n < a.N) part[((size_t)s * a.M + t) * a.N + n] = acc[nt][j];
                }
            __threadfence();
            named_bar_sync(1, NCT);
            if (tid == 0) ctl->last = (atomicAdd(&a.tickets[rb], 1) == a.S - 1);
            named_bar_sync(1, NCT);
            if (ctl->last) {
                __threadfence();
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int t = nt * 8 + 2 * tig + (j & 1);
                        const int n = row0 + gid + 8 * (j >> 1);
                        if (t < a.M && n < a.N) {
                            float v = 0.f;
                            for (int q = 0; q < a.S; ++q)
                                v += ld_cg_f32(part + ((size_t)q * a.M + t) * a.N + n);
                            const float b = a.bias ? __ldg(a.bias + n) : 0.f;
                            a.y[(size_t)t * a.N + n] = f32_to_bf16_bits(v + b);
                        }
                    }
                if (tid == 0) a.tickets[rb] = 0;
            }
        }
    }
}

template <int MT>
__device__ void w4a8_consumer(uint8_t* wbuf, uint8_t* xbuf, SmemCtl* ctl, const GemvArgs& a) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tig = lane & 3, gid = lane >> 2;
    const int8_t* qx = static_cast<const int8_t*>(a.x);
    const uint32_t wbuf_u = smem_u32(wbuf), xbuf_u = smem_u32(xbuf);
    const int lj = lane >> 3, li = lane & 7;
    const uint32_t l_rowoff = (uint32_t)(warp * 16 + ((lj & 1) << 3) + li) * 128u;
    const int l_chi = lj >> 1;
    uint32_t xrow[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m)
        xrow[m] = xbuf_u + (uint32_t)(min(m, a.M - 1) * a.XS + tig * 8);

    uint32_t it = 0;
    for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
        int rb, s, ks0, ks1;
        unit_coords(u, a, rb, s, ks0, ks1);
        const int row0 = rb * ROWS + warp * 16;

        named_bar_sync(1, NCT);
        if (tid < 16) ctl->sumq[tid] = 0;
        named_bar_sync(1, NCT);
        stage_x_s8(xbuf, ctl, qx, a.M, a.Kp, a.XS, ks0 * STAGE_K, (ks1 - ks0) * STAGE_K, tid);
        named_bar_sync(1, NCT);

        int acc[MT][2];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = 0;

        for (int ks = ks0; ks < ks1; ++ks, ++it) {
            const int slot = it % NS;
            if (mbar_wait(&ctl->full[slot], (it / NS) & 1, &ctl->abort, a.err)) {
                const uint32_t wst = wbuf_u + slot * STAGE_BYTES + l_rowoff;
                const uint32_t xoff = (uint32_t)(ks - ks0) * STAGE_K;
#pragma unroll
                for (int cp = 0; cp < 4; ++cp) {
                    uint32_t r[4];
                    ldmatrix_x4(wst + ((uint32_t)((2 * cp + l_chi) ^ li) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = 2 * cp + h;
                        const uint32_t lo = r[2 * h] & 0x0F0F0F0Fu, hi = (r[2 * h] >> 4) & 0x0F0F0F0Fu;
                        const uint32_t lo8 = r[2 * h + 1] & 0x0F0F0F0Fu, hi8 = (r[2 * h + 1] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            uint32_t xe, xo;
                            lds64(xrow[m] + xoff + c * 32, xe, xo);
                            acc[m][0] = dp4a_us(lo, xe, acc[m][0]);
                            acc[m][0] = dp4a_us(hi, xo, acc[m][0]);
                            acc[m][1] = dp4a_us(lo8, xe, acc[m][1]);
                            acc[m][1] = dp4a_us(hi8, xo, acc[m][1]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->empty[slot]);
        }

        // reduce over the four lanes that share a row, remove the +8 offset
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int v = acc[m][h];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                acc[m][h] = v - 8 * ctl->sumq[min(m, a.M - 1)];
            }
        int32_t* part = static_cast<int32_t*>(a.partial);
        if (a.S > 1) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int n = row0 + gid + 8 * h;
                    if (m < a.M && (m & 3) == tig && n < a.N)
                        part[((size_t)s * a.M + m) * a.N + n] = acc[m][h];
                }
            __threadfence();
            named_bar_sync(1, NCT);
            if (tid == 0) ctl->last = (atomicAdd(&a.tickets[rb], 1) == a.S - 1);
            named_bar_sync(1, NCT);
            if (!ctl->last) continue;
            __threadfence();
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = row0 + gid + 8 * h;
                if (m < a.M && (m & 3) == tig && n < a.N) {
                    int v = acc[m][h];
                    if (a.S > 1) {
                        v = 0;
                        for (int q = 0; q < a.S; ++q)
                            v += ld_cg_s32(part + ((size_t)q * a.M + m) * a.N + n);
                    }
                    if (a.acc_out) a.acc_out[(size_t)m * a.N + n] = v;
                    const float sc = __ldg(a.scales + n) * __ldg(a.sx + m);
                    const float b = a.bias ? __ldg(a.bias + n) : 0.f;
                    a.y[(size_t)m * a.N + n] = f32_to_bf16_bits(fmaf(sc, (float)v, b));
                }
            }
        if (a.S > 1 && tid == 0) a.tickets[rb] = 0;
    }
}

__device__ __forceinline__ void gemv_init(uint8_t*& wbuf, uint8_t*& xbuf, SmemCtl*& ctl,
                                          const CUtensorMap* tm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = align1024(smem_raw);
    wbuf = base;
    ctl = reinterpret_cast<SmemCtl*>(base + NS * STAGE_BYTES);
    xbuf = base + NS * STAGE_BYTES + kCtlBytes;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&ctl->full[i], 1);
            mbar_init(&ctl->empty[i], CW);
        }
        ctl->abort = 0;
        ctl->last = 0;
        for (int i = 0; i < 16; ++i) ctl->sumq[i] = 0;
        fence_mbar_init();
    }
    if (threadIdx.x == NCT) tma_prefetch_desc(tm);
    __syncthreads();
}

template <int NT, int CPG, bool ASYM>
__global__ void __launch_bounds__(kGemvThreads, 1)
k_w4a16_gemv(const __grid_constant__ CUtensorMap tmW, const GemvArgs a) {
    uint8_t *wbuf, *xbuf;
    SmemCtl* ctl;
    gemv_init(wbuf, xbuf, ctl, &tmW);
    if (threadIdx.x >= NCT) {
        if (threadIdx.x == NCT) gemv_producer(&tmW, wbuf, ctl, a);
    } else {
        w4a16_consumer<NT, CPG, ASYM>(wbuf, xbuf, ctl, a);
    }
}

template <int MT>
__global__ void __launch_bounds__(kGemvThreads, 1)
k_w4a8_gemv(const __grid_constant__ CUtensorMap tmW, const GemvArgs a) {
    uint8_t *wbuf, *xbuf;
    SmemCtl* ctl;
    gemv_init(wbuf, xbuf, ctl, &tmW);
    if (threadIdx.x >= NCT) {
        if (threadIdx.x == NCT) gemv_producer(&tmW, wbuf, ctl, a);
    } else {
        w4a8_consumer<MT>(wbuf, xbuf, ctl, a);
    }
}

template <typename Kern>
int launch(Kern kern, const CUtensorMap& tm, const GemvArgs& a, const GemvPlan& p,
           cudaStream_t stream) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)p.smem) != cudaSuccess)
        return W4_ERR_CUDA;
    kern<<<p.grid, kGemvThreads, p.smem, stream>>>(tm, a);
    return cudaGetLastError() == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

template <int NT, bool ASYM>
int launch_w4a16_cpg(int cpg, const CUtensorMap& tm, const GemvArgs& a, const GemvPlan& p,
                     cudaStream_t st) {
    switch (cpg) {
        case 8: return launch(k_w4a16_gemv<NT, 8, ASYM>, tm, a, p, st);
        case 4: return launch(k_w4a16_gemv<NT, 4, ASYM>, tm, a, p, st);
        case 2: return launch(k_w4a16_gemv<NT, 2, ASYM>, tm, a, p, st);
        default: return launch(k_w4a16_gemv<NT, 1, ASYM>, tm, a, p, st);
    }
}

}  // namespace

bool plan_gemv(int M, int N, int Kp, int act_bytes, int sm_count, GemvPlan* p) {
    if (M < 1 || M > 16 || N < 1 || Kp < 1) return false;
    const int nst = (Kp + STAGE_K - 1) / STAGE_K;
    const int NB = (N + ROWS - 1) / ROWS;
    const size_t cap = 232448;                       // 227 KB opt-in per CTA
    const size_t fixed = 1024 + (size_t)NS * STAGE_BYTES + kCtlBytes;
    const int pad = act_bytes == 2 ? 64 : 16;
    const long per_tok = (long)((cap - fixed) / (size_t)M) - pad;
    const int spl_max = (int)(per_tok / (STAGE_K * act_bytes));
    if (spl_max < 1) return false;
    const int s_min = (nst + spl_max - 1) / spl_max;
    double best = 1e30;
    for (int S = s_min; S <= nst; ++S) {
        const int spl = (nst + S - 1) / S;
        const int Se = (nst + spl - 1) / spl;
        if (spl > spl_max) continue;
        const int units = NB * Se;
        const int grid = std::min(units, sm_count);
        const int waves = (units + grid - 1) / grid;
        const double cost = (double)waves * spl + (Se > 1 ? 1.0 * waves : 0.0);
        if (cost < best - 1e-9) {
            best = cost;
            p->nst = nst; p->NB = NB; p->S = Se; p->spl = spl; p->units = units;
            p->grid = grid;
        }
        if (Se == nst) break;
    }
    p->XS = p->spl * STAGE_K * act_bytes + pad;
    p->smem = fixed + (size_t)M * p->XS;
    p->ws_bytes = 0;
    if (p->S > 1)
        p->ws_bytes = (((size_t)p->NB * 4 + 255) / 256) * 256 + (size_t)p->S * M * N * 4;
    return true;
}

int launch_w4a16_gemv(const CUtensorMap& tm, const GemvArgs& a, const GemvPlan& p,
                      cudaStream_t st) {
    const int gq = a.G / 32;
    const int cpg = (gq % 8 == 0) ? 8 : (gq % 4 == 0) ? 4 : (gq % 2 == 0) ? 2 : 1;
    const bool asym = a.zeros != nullptr;
    if (a.M <= 8)
        return asym ? launch_w4a16_cpg<1, true>(cpg, tm, a, p, st)
                    : launch_w4a16_cpg<1, false>(cpg, tm, a, p, st);
    return asym ? launch_w4a16_cpg<2, true>(cpg, tm, a, p, st)
                : launch_w4a16_cpg<2, false>(cpg, tm, a, p, st);
}

int launch_w4a8_gemv(const CUtensorMap& tm, const GemvArgs& a, const GemvPlan& p,
                     cudaStream_t st) {
    if (a.M <= 1) return launch(k_w4a8_gemv<1>, tm, a, p, st);
    if (a.M <= 2) return launch(k_w4a8_gemv<2>, tm, a, p, st);
    if (a.M <= 4) return launch(k_w4a8_gemv<4>, tm, a, p, st);
    if (a.M <= 8) return launch(k_w4a8_gemv<8>, tm, a, p, st);
    return launch(k_w4a8_gemv<16>, tm, a, p, st);
}

}  // namespace w4
